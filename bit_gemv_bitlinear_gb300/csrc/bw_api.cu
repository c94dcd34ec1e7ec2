// bw_api.cu -- the C ABI of libbw: argument validation, launch planning and
// status codes.  Every check happens on the host before any launch; the
// GEMV path neither allocates nor synchronises.
#include <cstdio>

#include "bw_internal.cuh"

namespace bw {

namespace {
thread_local int g_last_cuda_error = 0;

bw_status cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return BW_OK;
  g_last_cuda_error = int(e);
  return BW_ERR_CUDA;
}

bool aligned(const void *p, uintptr_t a) {
  return (reinterpret_cast<uintptr_t>(p) % a) == 0;
}

bw_status check_mnk(int M, int N, int K) {
  if (M < 1 || N < 1 || K < 4) return BW_ERR_INVALID_ARG;
  if (K % 4 != 0) return BW_ERR_UNSUPPORTED_SHAPE;
  if (M > BW_MAX_M || N > BW_MAX_N || K > BW_MAX_K)
    return BW_ERR_UNSUPPORTED_SHAPE;
  return BW_OK;
}

constexpr int kMaxDevices = 64;
std::atomic<int> g_sm_count[kMaxDevices];  // 0: not queried yet

// The checks every product entry point makes (pointers, shape, scale
// segments, alignment); fills the segments.
bw_status check_product(const int8_t *x, const uint8_t *packed,
                        const float *s, const bw_bf16 *ws,
                        const int *ws_bounds, int n_ws, int M, int N, int K,
                        const void *out, bool acc_out, WsSegments *seg) {
  if (!x || !packed || !out) return BW_ERR_INVALID_ARG;
  bw_status st = check_mnk(M, N, K);
  if (st != BW_OK) return st;
  *seg = WsSegments{};
  if (!acc_out) {
    if (!s || !ws || !ws_bounds) return BW_ERR_INVALID_ARG;
    if (n_ws < 1 || n_ws > BW_MAX_WS) return BW_ERR_INVALID_ARG;
    if (ws_bounds[0] != 0 || ws_bounds[n_ws] != N) return BW_ERR_INVALID_ARG;
    for (int i = 0; i < n_ws; ++i)
      if (ws_bounds[i + 1] <= ws_bounds[i]) return BW_ERR_INVALID_ARG;
    seg->n_ws = n_ws;
    for (int i = 0; i <= n_ws; ++i) seg->bounds[i] = ws_bounds[i];
    if (!aligned(s, 4) || !aligned(ws, 2) || !aligned(out, 2))
      return BW_ERR_MISALIGNED;
  } else if (!aligned(out, 4)) {
    return BW_ERR_MISALIGNED;
  }
  if (!aligned(x, 4) || !aligned(packed, 16)) return BW_ERR_MISALIGNED;
  return BW_OK;
}

// Shared validation and launch of both GEMV entry points.
bw_status gemv_common(const int8_t *x, const uint8_t *packed, const float *s,
                      const bw_bf16 *ws, const int *ws_bounds, int n_ws,
                      int M, int N, int K, void *out, bool acc_out,
                      cudaStream_t stream) {
  WsSegments seg;
  bw_status st = check_product(x, packed, s, ws, ws_bounds, n_ws, M, N, K, out,
                               acc_out, &seg);
  if (st != BW_OK) return st;

  const int sms = device_sm_count();
  if (sms <= 0) return cuda_status(cudaErrorNoDevice);

  GemvArgs a{};
  a.w = packed;
  a.ws = reinterpret_cast<const __nv_bfloat16 *>(ws);
  a.K = K;
  a.N = N;
  a.x_ld = K;
  a.out_ld = N;
  a.chunks = chunks_per_row(K);
  a.n_groups = int(padded_rows(N) / kGroupRows);
  a.vec_x = aligned(x, 16) && (K % 16 == 0);
  a.seg = seg;
  const size_t out_elem = acc_out ? sizeof(int32_t) : sizeof(bw_bf16);

  // Batched activations: tcgen05 tensor cores, tiles of up to kTcMaxRows
  // (128) rows.
  if (M >= kMmaMinRows && tc_fits(a)) {
    for (int m0 = 0; m0 < M; m0 += kTcMaxRows) {
      const int rows = M - m0 < kTcMaxRows ? M - m0 : kTcMaxRows;
      a.x = x + size_t(m0) * K;
      a.s = acc_out ? nullptr : s + m0;
      a.out = static_cast<char *>(out) + size_t(m0) * N * out_elem;
      cudaError_t e = launch_gemv_tc(a, rows, acc_out, stream);
      if (e != cudaSuccess) return cuda_status(e);
    }
    return BW_OK;
  }

  // Otherwise (activation rows not 16-byte aligned): mma.sync tiles of 16
  // (or 8) rows.
  const int tile = (M >= kMmaMinRows && K <= kMmaMaxK) ? mma_tile_rows(K) : 0;
  if (tile) {
    for (int m0 = 0; m0 < M; m0 += tile) {
      const int rows = M - m0 < tile ? M - m0 : tile;
      a.x = x + size_t(m0) * K;
      a.s = acc_out ? nullptr : s + m0;
      a.out = static_cast<char *>(out) + size_t(m0) * N * out_elem;
      cudaError_t e = launch_gemv_mma(a, rows, acc_out, stream);
      if (e != cudaSuccess) return cuda_status(e);
    }
    return BW_OK;
  }

  // Activation rows in tiles of 4, then 2, then 1.
  int m0 = 0;
  while (m0 < M) {
    const int left = M - m0;
    const int mt = left >= 4 ? 4 : (left >= 2 ? 2 : 1);
    a.x = x + size_t(m0) * K;
    a.s = acc_out ? nullptr : s + m0;
    a.out = static_cast<char *>(out) + size_t(m0) * N * out_elem;
    cudaError_t e;
    if (pipe_fits(mt, K)) {
      e = launch_gemv_pipe(a, mt, acc_out, stream);
    } else {  // activations too long for shared memory: register-streamed
      GemvPlan plan = plan_gemv(mt, N, K, sms);
      a.passes = plan.passes;
      e = launch_gemv(plan, a, acc_out, stream);
    }
    if (e != cudaSuccess) return cuda_status(e);
    m0 += mt;
  }
  return BW_OK;
}

// The pair-table variant: the same validation, then M-tiles of 4, 2 and 1
// rows, all checked to fit before the first launch.
bw_status gemv_lut_common(const int8_t *x, const uint8_t *packed,
                          const float *s, const bw_bf16 *ws,
                          const int *ws_bounds, int n_ws, int M, int N, int K,
                          void *out, bool acc_out, cudaStream_t stream) {
  WsSegments seg;
  bw_status st = check_product(x, packed, s, ws, ws_bounds, n_ws, M, N, K, out,
                               acc_out, &seg);
  if (st != BW_OK) return st;
  if (device_sm_count() <= 0) return cuda_status(cudaErrorNoDevice);
  for (int left = M; left > 0;) {
    const int mt = left >= 4 ? 4 : (left >= 2 ? 2 : 1);
    if (!lut_fits(mt, N, K)) return BW_ERR_UNSUPPORTED_SHAPE;
    left -= mt;
  }
  GemvArgs a{};
  a.w = packed;
  a.ws = reinterpret_cast<const __nv_bfloat16 *>(ws);
  a.K = K;
  a.N = N;
  a.x_ld = K;
  a.out_ld = N;
  a.chunks = chunks_per_row(K);
  a.n_groups = int(padded_rows(N) / kGroupRows);
  a.seg = seg;
  const size_t out_elem = acc_out ? sizeof(int32_t) : sizeof(bw_bf16);
  for (int m0 = 0; m0 < M;) {
    const int left = M - m0;
    const int mt = left >= 4 ? 4 : (left >= 2 ? 2 : 1);
    a.x = x + size_t(m0) * K;
    a.s = acc_out ? nullptr : s + m0;
    a.out = static_cast<char *>(out) + size_t(m0) * N * out_elem;
    cudaError_t e = launch_gemv_lut(a, mt, acc_out, stream);
    if (e != cudaSuccess) return cuda_status(e);
    m0 += mt;
  }
  return BW_OK;
}

// The prefill product: validation, then the token conversion and the
// 256-token tensor-core tiles (two launches).
bw_status gemm_common(const int8_t *x, const uint8_t *packed, const float *s,
                      const bw_bf16 *ws, const int *ws_bounds, int n_ws,
                      int M, int N, int K, void *out, bool acc_out,
                      void *workspace, size_t workspace_bytes,
                      cudaStream_t stream) {
  WsSegments seg;
  bw_status st = check_product(x, packed, s, ws, ws_bounds, n_ws, M, N, K, out,
                               acc_out, &seg);
  if (st != BW_OK) return st;
  if (K > kMmaMaxK) return BW_ERR_UNSUPPORTED_SHAPE;
  if (!workspace || workspace_bytes < gemm_workspace_bytes(M, K))
    return BW_ERR_INVALID_ARG;
  if (!aligned(workspace, 256)) return BW_ERR_MISALIGNED;
  if (device_sm_count() <= 0) return cuda_status(cudaErrorNoDevice);
  GemvArgs a{};
  a.x = x;
  a.w = packed;
  a.s = acc_out ? nullptr : s;
  a.ws = reinterpret_cast<const __nv_bfloat16 *>(ws);
  a.out = out;
  a.K = K;
  a.N = N;
  a.x_ld = K;
  a.out_ld = N;
  a.chunks = chunks_per_row(K);
  a.n_groups = int(padded_rows(N) / kGroupRows);
  a.seg = seg;
  return cuda_status(launch_gemm(a, M, acc_out, workspace, stream));
}

}  // namespace

int device_sm_count() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
    return 0;
  int n = g_sm_count[dev].load(std::memory_order_relaxed);
  if (n == 0) {
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) !=
        cudaSuccess)
      return 0;
    g_sm_count[dev].store(n, std::memory_order_relaxed);
  }
  return n;
}

void record_cuda_error(int err) { g_last_cuda_error = err; }

bw_status gemv_internal(const int8_t *x, const uint8_t *packed, const float *s,
                        const bw_bf16 *ws, const int *ws_bounds, int n_ws,
                        int M, int N, int K, bw_bf16 *y, cudaStream_t stream) {
  return gemv_common(x, packed, s, ws, ws_bounds, n_ws, M, N, K, y, false,
                     stream);
}

}  // namespace bw

using namespace bw;

extern "C" {

const char *bw_status_string(bw_status status) {
  switch (status) {
    case BW_OK: return "BW_OK";
    case BW_ERR_INVALID_ARG: return "BW_ERR_INVALID_ARG";
    case BW_ERR_UNSUPPORTED_SHAPE: return "BW_ERR_UNSUPPORTED_SHAPE";
    case BW_ERR_MISALIGNED: return "BW_ERR_MISALIGNED";
    case BW_ERR_BAD_CODE: return "BW_ERR_BAD_CODE";
    case BW_ERR_CUDA: return "BW_ERR_CUDA";
    case BW_ERR_TIMEOUT: return "BW_ERR_TIMEOUT";
  }
  return "BW_ERR_UNKNOWN";
}

int bw_last_cuda_error(void) { return g_last_cuda_error; }

int bw_version(void) { return 100; }

bw_status bw_quant_act(const float *x, int M, int K, int8_t *q, float *s,
                       bw_stream_t stream) {
  if (!x || !q || !s || M < 1 || K < 1) return BW_ERR_INVALID_ARG;
  if (M > BW_MAX_M || K > BW_MAX_K) return BW_ERR_UNSUPPORTED_SHAPE;
  if (!aligned(x, 4) || !aligned(s, 4)) return BW_ERR_MISALIGNED;
  return cuda_status(launch_quant_act(x, M, K, q, s,
                                      reinterpret_cast<cudaStream_t>(stream)));
}

size_t bw_gemv_workspace_bytes(int M, int N, int K) {
  (void)M;
  (void)N;
  (void)K;
  return 0;  // partial sums never leave a CTA's shared memory
}

size_t bw_repack_bytes(int N, int K) {
  if (N < 1 || K < 4 || N > BW_MAX_N || K > BW_MAX_K) return 0;
  return size_t(padded_rows(N)) * size_t(chunks_per_row(K)) * kChunkBytes;
}

bw_status bw_repack(const uint8_t *canon, int N, int K, uint8_t *packed,
                    bw_stream_t stream) {
  if (!canon || !packed) return BW_ERR_INVALID_ARG;
  bw_status st = check_mnk(1, N, K);
  if (st != BW_OK) return st;
  if (!aligned(packed, 16)) return BW_ERR_MISALIGNED;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  unsigned int *bad = nullptr;
  unsigned int bad_host = 0;
  cudaError_t e = cudaMallocAsync(reinterpret_cast<void **>(&bad),
                                  sizeof(unsigned int), cs);
  if (e != cudaSuccess) return cuda_status(e);
  e = cudaMemsetAsync(bad, 0, sizeof(unsigned int), cs);
  if (e == cudaSuccess) e = launch_repack(canon, N, K, packed, bad, cs);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(&bad_host, bad, sizeof(unsigned int),
                        cudaMemcpyDeviceToHost, cs);
  cudaError_t ef = cudaFreeAsync(bad, cs);
  if (e == cudaSuccess) e = ef;
  if (e == cudaSuccess) e = cudaStreamSynchronize(cs);
  if (e != cudaSuccess) return cuda_status(e);
  return bad_host ? BW_ERR_BAD_CODE : BW_OK;
}

bw_status bw_quant_weight(const float *W, int N, int K, const int *ws_bounds,
                          int n_ws, uint8_t *canon, bw_bf16 *ws,
                          bw_stream_t stream) {
  if (!W || !canon || !ws || !ws_bounds) return BW_ERR_INVALID_ARG;
  bw_status st = check_mnk(1, N, K);
  if (st != BW_OK) return st;
  if (n_ws < 1 || n_ws > BW_MAX_WS) return BW_ERR_INVALID_ARG;
  if (ws_bounds[0] != 0 || ws_bounds[n_ws] != N) return BW_ERR_INVALID_ARG;
  for (int i = 0; i < n_ws; ++i)
    if (ws_bounds[i + 1] <= ws_bounds[i]) return BW_ERR_INVALID_ARG;
  if (!aligned(W, 16) || !aligned(ws, 2)) return BW_ERR_MISALIGNED;
  WsSegments seg{};
  seg.n_ws = n_ws;
  for (int i = 0; i <= n_ws; ++i) seg.bounds[i] = ws_bounds[i];
  return cuda_status(launch_quant_weight(
      W, N, K, seg, canon, reinterpret_cast<__nv_bfloat16 *>(ws),
      reinterpret_cast<cudaStream_t>(stream)));
}

bw_status bw_unrepack(const uint8_t *packed, int N, int K, uint8_t *canon,
                      bw_stream_t stream) {
  if (!canon || !packed) return BW_ERR_INVALID_ARG;
  bw_status st = check_mnk(1, N, K);
  if (st != BW_OK) return st;
  if (!aligned(packed, 16)) return BW_ERR_MISALIGNED;
  return cuda_status(launch_unrepack(packed, N, K, canon,
                                     reinterpret_cast<cudaStream_t>(stream)));
}

bw_status bw_gemv_w2a8(const int8_t *x, const uint8_t *packed, const float *s,
                       const bw_bf16 *ws, const int *ws_bounds, int n_ws,
                       int M, int N, int K, bw_bf16 *y, bw_stream_t stream) {
  return gemv_common(x, packed, s, ws, ws_bounds, n_ws, M, N, K, y, false,
                     reinterpret_cast<cudaStream_t>(stream));
}

bw_status bw_device_error(unsigned int *bits, bw_stream_t stream) {
  if (!bits) return BW_ERR_INVALID_ARG;
  cudaError_t e =
      read_device_error(reinterpret_cast<cudaStream_t>(stream), bits);
  if (e != cudaSuccess) return cuda_status(e);
  if (*bits & ~(16u | 128u)) return BW_ERR_TIMEOUT;  // caller errors: 16, 128
  return *bits ? BW_ERR_INVALID_ARG : BW_OK;
}

bw_status bw_selftest_wait_timeout(unsigned int *bits, bw_stream_t stream) {
  if (!bits) return BW_ERR_INVALID_ARG;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = launch_selftest_wait(cs);
  if (e == cudaSuccess) e = launch_selftest_poll(cs);
  if (e == cudaSuccess) e = read_device_error(cs, bits);
  if (e != cudaSuccess) return cuda_status(e);
  return *bits ? BW_ERR_TIMEOUT : BW_OK;
}

bw_status bw_gemv_w2a8_acc(const int8_t *x, const uint8_t *packed, int M,
                           int N, int K, int32_t *acc, bw_stream_t stream) {
  return gemv_common(x, packed, nullptr, nullptr, nullptr, 0, M, N, K, acc,
                     true, reinterpret_cast<cudaStream_t>(stream));
}

bw_status bw_gemv_w2a8_lut(const int8_t *x, const uint8_t *packed,
                           const float *s, const bw_bf16 *ws,
                           const int *ws_bounds, int n_ws, int M, int N, int K,
                           bw_bf16 *y, bw_stream_t stream) {
  return gemv_lut_common(x, packed, s, ws, ws_bounds, n_ws, M, N, K, y, false,
                         reinterpret_cast<cudaStream_t>(stream));
}

bw_status bw_gemv_w2a8_lut_acc(const int8_t *x, const uint8_t *packed, int M,
                               int N, int K, int32_t *acc,
                               bw_stream_t stream) {
  return gemv_lut_common(x, packed, nullptr, nullptr, nullptr, 0, M, N, K,
                         acc, true, reinterpret_cast<cudaStream_t>(stream));
}

size_t bw_gemm_workspace_bytes(int M, int K) {
  if (M < 1 || M > BW_MAX_M || K < 4 || K % 4 != 0 || K > kMmaMaxK) return 0;
  return gemm_workspace_bytes(M, K);
}

bw_status bw_gemm_w2a8(const int8_t *x, const uint8_t *packed, const float *s,
                       const bw_bf16 *ws, const int *ws_bounds, int n_ws,
                       int M, int N, int K, bw_bf16 *y, void *workspace,
                       size_t workspace_bytes, bw_stream_t stream) {
  return gemm_common(x, packed, s, ws, ws_bounds, n_ws, M, N, K, y, false,
                     workspace, workspace_bytes,
                     reinterpret_cast<cudaStream_t>(stream));
}

bw_status bw_gemm_w2a8_acc(const int8_t *x, const uint8_t *packed, int M,
                           int N, int K, int32_t *acc, void *workspace,
                           size_t workspace_bytes, bw_stream_t stream) {
  return gemm_common(x, packed, nullptr, nullptr, nullptr, 0, M, N, K, acc,
                     true, workspace, workspace_bytes,
                     reinterpret_cast<cudaStream_t>(stream));
}

}  // extern "C"
