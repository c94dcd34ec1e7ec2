// bw_misc.cu -- activation quantisation and weight repacking for sm_103a.
//
// Sources: "BitNet GPU 推理框架：从零构建 W2A8 的 2-bit 大模型 CUDA GEMV 内核",
// §六 item 3 (per-row absmax quantisation s = 127 / max|x|, round, clamp to
// [-128, 127]) and §5.1/§5.2 (offline packing of the ternary weights; the
// device layout produced here is specified in bw.h).
#include "bw_internal.cuh"

namespace bw {
namespace {

constexpr int kQuantThreads = 256;

// Block-wide max of a non-negative value (every thread gets the result).
__device__ __forceinline__ float block_max(float v, float *warp_max) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1)
    v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  if ((threadIdx.x & 31) == 0) warp_max[threadIdx.x >> 5] = v;
  __syncthreads();
  v = 0.0f;
  for (int w = 0; w < int(blockDim.x >> 5); ++w) v = fmaxf(v, warp_max[w]);
  return v;
}

// q = clamp(rint(x * s), -128, 127) in IEEE fp32; rintf rounds half to even.
__device__ __forceinline__ int8_t quant1(float x, float scale) {
  return static_cast<int8_t>(
      static_cast<int>(fminf(fmaxf(rintf(x * scale), -128.0f), 127.0f)));
}

// Programmatic dependent launch: let the next kernel (a GEMV that only
// prefetches weights before its own wait) start its prologue now, and wait
// for the producer of x before reading it (or writing q and s).
__device__ __forceinline__ void pdl_enter() {
  asm volatile("griddepcontrol.launch_dependents;");
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

// One CTA per activation row.  Pass 1: absmax (max is exact in any order).
// Pass 2: q = clamp(rint(x * s), -128, 127), s = 127 / max(absmax, 1e-5).
__global__ void __launch_bounds__(kQuantThreads)
quant_act_kernel(const float *__restrict__ x, int K, int8_t *__restrict__ q,
                 float *__restrict__ s) {
  __shared__ float warp_max[kQuantThreads / 32];
  pdl_enter();
  const int m = blockIdx.x;
  const float *xr = x + size_t(m) * K;
  int8_t *qr = q + size_t(m) * K;
  float amax = 0.0f;
  for (int k = threadIdx.x; k < K; k += blockDim.x)
    amax = fmaxf(amax, fabsf(xr[k]));
  amax = block_max(amax, warp_max);
  const float scale = 127.0f / fmaxf(amax, 1e-5f);
  if (threadIdx.x == 0) s[m] = scale;
  for (int k = threadIdx.x; k < K; k += blockDim.x) qr[k] = quant1(xr[k], scale);
}

// The same arithmetic for rows with K % 4 == 0 that start on a 16-byte
// boundary: V float4 per thread stay in registers between the two passes
// and q is written 4 bytes at a time.
template <int V>
__global__ void __launch_bounds__(kQuantThreads)
quant_act_vec_kernel(const float *__restrict__ x, int K,
                     int8_t *__restrict__ q, float *__restrict__ s) {
  __shared__ float warp_max[kQuantThreads / 32];
  pdl_enter();
  const int m = blockIdx.x;
  const int nv = K / 4;
  const float4 *xr = reinterpret_cast<const float4 *>(x + size_t(m) * K);
  char4 *qr = reinterpret_cast<char4 *>(q + size_t(m) * K);
  float4 v[V];
  float amax = 0.0f;
#pragma unroll
  for (int i = 0; i < V; ++i) {
    const int idx = threadIdx.x + i * kQuantThreads;
    v[i] = idx < nv ? xr[idx] : make_float4(0.f, 0.f, 0.f, 0.f);
    amax = fmaxf(amax, fmaxf(fmaxf(fabsf(v[i].x), fabsf(v[i].y)),
                             fmaxf(fabsf(v[i].z), fabsf(v[i].w))));
  }
  amax = block_max(amax, warp_max);
  const float scale = 127.0f / fmaxf(amax, 1e-5f);
  if (threadIdx.x == 0) s[m] = scale;
#pragma unroll
  for (int i = 0; i < V; ++i) {
    const int idx = threadIdx.x + i * kQuantThreads;
    if (idx < nv)
      qr[idx] = make_char4(quant1(v[i].x, scale), quant1(v[i].y, scale),
                           quant1(v[i].z, scale), quant1(v[i].w, scale));
  }
}

// One thread per 16-byte output chunk, enumerated in memory order:
// idx = ((group * C) + j) * 8 + row_in_group.
__global__ void repack_kernel(const uint8_t *__restrict__ canon, int N, int K,
                              int chunks, int64_t total,
                              uint8_t *__restrict__ packed,
                              unsigned int *__restrict__ bad) {
  const int64_t row_bytes = K / 4;
  for (int64_t idx = blockIdx.x * int64_t(blockDim.x) + threadIdx.x;
       idx < total; idx += int64_t(gridDim.x) * blockDim.x) {
    const int64_t r = idx % kGroupRows;
    const int64_t j = (idx / kGroupRows) % chunks;
    const int64_t grp = idx / (int64_t(kGroupRows) * chunks);
    const int64_t n = grp * kGroupRows + r;
    uint32_t word[4] = {0u, 0u, 0u, 0u};
    bool bad_code = false;
    for (int i = 0; i < kChunkWeights; ++i) {
      const int64_t k = j * kChunkWeights + i;
      uint32_t code = 1u;  // padding: weight 0
      if (n < N && k < K) {
        code = (canon[n * row_bytes + k / 4] >> (2 * (k % 4))) & 3u;
        bad_code |= code == 3u;
      }
      const int t = i / 16, e = i % 16;
      word[t] |= code << (8 * (e % 4) + 2 * (e / 4));
    }
    if (bad_code) atomicOr(bad, 1u);
    reinterpret_cast<uint4 *>(packed)[idx] =
        make_uint4(word[0], word[1], word[2], word[3]);
  }
}

// One thread per canonical byte.
__global__ void unrepack_kernel(const uint8_t *__restrict__ packed, int N,
                                int K, int chunks,
                                uint8_t *__restrict__ canon) {
  const int64_t row_bytes = K / 4;
  const int64_t total = int64_t(N) * row_bytes;
  for (int64_t idx = blockIdx.x * int64_t(blockDim.x) + threadIdx.x;
       idx < total; idx += int64_t(gridDim.x) * blockDim.x) {
    const int64_t n = idx / row_bytes;
    const int64_t b = idx % row_bytes;
    uint32_t byte = 0u;
    for (int t = 0; t < 4; ++t) {
      const int64_t k = 4 * b + t;
      const int64_t j = k / kChunkWeights;
      const int wt = int(k % kChunkWeights) / 16;
      const int e = int(k % 16);
      const int64_t off =
          ((n / kGroupRows) * chunks + j) * kGroupChunkBytes +
          (n % kGroupRows) * kChunkBytes + wt * 4 + (e % 4);
      const uint32_t code = (packed[off] >> (2 * (e / 4))) & 3u;
      byte |= code << (2 * t);
    }
    canon[idx] = static_cast<uint8_t>(byte);
  }
}

int grid_for(int64_t items, int threads) {
  const int64_t blocks = (items + threads - 1) / threads;
  const int64_t cap = int64_t(device_sm_count()) * 16;
  return int(blocks < cap ? (blocks > 0 ? blocks : 1) : cap);
}

}  // namespace

cudaError_t launch_quant_act(const float *x, int M, int K, int8_t *q,
                             float *s, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(M);
  cfg.blockDim = dim3(kQuantThreads);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const bool vec = K % 4 == 0 && reinterpret_cast<uintptr_t>(x) % 16 == 0 &&
                   reinterpret_cast<uintptr_t>(q) % 4 == 0;
  const int per_thread = (K / 4 + kQuantThreads - 1) / kQuantThreads;
  if (vec && per_thread <= 1)
    return cudaLaunchKernelEx(&cfg, quant_act_vec_kernel<1>, x, K, q, s);
  if (vec && per_thread <= 2)
    return cudaLaunchKernelEx(&cfg, quant_act_vec_kernel<2>, x, K, q, s);
  if (vec && per_thread <= 4)
    return cudaLaunchKernelEx(&cfg, quant_act_vec_kernel<4>, x, K, q, s);
  if (vec && per_thread <= 8)
    return cudaLaunchKernelEx(&cfg, quant_act_vec_kernel<8>, x, K, q, s);
  return cudaLaunchKernelEx(&cfg, quant_act_kernel, x, K, q, s);
}

cudaError_t launch_repack(const uint8_t *canon, int N, int K,
                          uint8_t *packed, unsigned int *bad,
                          cudaStream_t stream) {
  const int chunks = chunks_per_row(K);
  const int64_t total = padded_rows(N) * chunks;
  repack_kernel<<<grid_for(total, 256), 256, 0, stream>>>(
      canon, N, K, chunks, total, packed, bad);
  return cudaGetLastError();
}

cudaError_t launch_unrepack(const uint8_t *packed, int N, int K,
                            uint8_t *canon, cudaStream_t stream) {
  const int64_t total = int64_t(N) * (K / 4);
  unrepack_kernel<<<grid_for(total, 256), 256, 0, stream>>>(
      packed, N, K, chunks_per_row(K), canon);
  return cudaGetLastError();
}

}  // namespace bw
