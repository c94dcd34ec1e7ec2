// bw_attn.cu -- one decode step of grouped-query attention over a bf16 KV
// cache: RoPE on the new key and on the queries, the append of the new key
// and value at position p, and softmax attention over positions 0..p.
//
// Sources: "BitNet GPU 推理框架：从零构建 W2A8 的 2-bit 大模型 CUDA GEMV 内核",
// §一 (BitNet-2B: 20 query heads over 5 KV heads of 128 dims), §4.1 (the
// model's RoPE turns adjacent pairs of head dims, which is why the
// checkpoint conversion interleaves the Q/K rows), §六 item 2 (the KV cache
// is preallocated and attention takes a flash path).
//
// Design for sm_103a.  The step reads 2 Hkv (p + 1) D bf16 values of cache
// and little else, so it is bound by HBM at long contexts and by latency
// at short ones:
//  * CTA (c, g) takes split c of the positions 0..p for KV head g and all
//    G = H / Hkv query heads that read it, so every K and V row is loaded
//    once for the G heads.  The number of splits is fixed at launch from
//    the cache capacity (at most 128, at least 64 positions each); the
//    position p is read on the device, so one launch serves every step of
//    a graph-replayed decode loop, and splits past the context are empty.
//  * A half-warp takes one position: lane l holds head dims 8 (l % 16) ..
//    8 (l % 16) + 7, one 16-byte load per row; the G dot products are
//    summed over the half-warp with four shuffles each.
//  * Inside a CTA the softmax has two passes over the scores in shared
//    memory (largest score, then exp and sum); the CTA writes its largest
//    scores m, exp sums l and unnormalised outputs to the workspace.
//  * The last CTA of KV head g to finish (a fence and an atomic counter;
//    nothing spins) merges the splits: out = sum_c e^(m_c - M) acc_c /
//    sum_c e^(m_c - M) l_c, and sets the counter back to zero.
//  * The CTA whose split holds p rotates the new key, rounds it to bf16,
//    uses it for the score of p and writes key and value to row p of the
//    cache; no CTA reads row p from memory.
// Arithmetic: fp32 throughout (fp32 angles p * f_i with f_i =
// theta^(-2i/D) rounded to fp32 on the host, sincosf, expf), bf16 cache.
#include "bw_pipe.cuh"

namespace bw {
namespace {

using pipe::pdl_trigger;
using pipe::pdl_wait;

constexpr int kAttnD = 128;             // head dim
constexpr int kAttnPairs = kAttnD / 2;
constexpr int kAttnThreads = 128;
constexpr int kAttnWarps = kAttnThreads / 32;
constexpr int kAttnMinChunk = 64;       // positions per split, at least
constexpr int kAttnMaxSplits = 128;
constexpr int kAttnMaxChunk = BW_ATTN_MAX_S / kAttnMaxSplits;  // 512
constexpr unsigned int kAttnErrPosition = 16u;  // device error word bit
static_assert(kAttnThreads == kAttnD, "thread t owns head dim t in the sums");

struct AttnArgs {
  const __nv_bfloat16 *qkv;  // [(H + 2 Hkv) D]
  const int *pos;            // [1]
  __nv_bfloat16 *kc, *vc;    // [Hkv][S][D]
  float *out;                // [H][D]
  float *part;               // [Hkv][n_split][G][2 + D]
  unsigned int *count;       // [Hkv]
  int H, Hkv, S, n_split;
  float inv_sqrt_d;
  float freq[kAttnPairs];    // f_i = theta^(-2i/D), fp32
  unsigned int *err;
};

__host__ __device__ inline int attn_splits(int S) {
  const int n = (S + kAttnMinChunk - 1) / kAttnMinChunk;
  return n < 1 ? 1 : (n > kAttnMaxSplits ? kAttnMaxSplits : n);
}

// Shared memory: pair cos/sin, rotated queries, the new key, scores (later
// the merge weights), per-warp outputs, reduction scratch.
template <int G>
struct AttnSmem {
  static constexpr int kCs = 0;                              // [64] float2
  static constexpr int kQ = kCs + 2 * kAttnPairs;            // [G][D]
  static constexpr int kKn = kQ + G * kAttnD;                // [D]
  static constexpr int kSc = kKn + kAttnD;                   // [chunk][G]
  static constexpr int kWacc = kSc + kAttnMaxChunk * G;      // [warps][G][D]
  static constexpr int kRed = kWacc + kAttnWarps * G * kAttnD;  // [warps][G]
  static constexpr int kFloats = kRed + kAttnWarps * G;
  static constexpr size_t kBytes = size_t(kFloats) * 4;
};

__device__ __forceinline__ void bf16x8_to_f32(uint4 raw, float (&v)[8]) {
  const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    v[2 * i] = __uint_as_float(w[i] << 16);
    v[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

// Max (kMax) or sum over the CTA of G values per thread, in a fixed order;
// every thread receives the results.  `red` holds kAttnWarps * G floats.
template <int G, bool kMax>
__device__ __forceinline__ void cta_reduce(float (&v)[G], float *red) {
#pragma unroll
  for (int h = 0; h < G; ++h)
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float t = __shfl_xor_sync(0xffffffffu, v[h], o);
      v[h] = kMax ? fmaxf(v[h], t) : v[h] + t;
    }
  __syncthreads();
  if ((threadIdx.x & 31) == 0)
#pragma unroll
    for (int h = 0; h < G; ++h) red[(threadIdx.x >> 5) * G + h] = v[h];
  __syncthreads();
#pragma unroll
  for (int h = 0; h < G; ++h) {
    float t = red[h];
#pragma unroll
    for (int w = 1; w < kAttnWarps; ++w)
      t = kMax ? fmaxf(t, red[w * G + h]) : t + red[w * G + h];
    v[h] = t;
  }
  __syncthreads();  // red may be reused at once
}

template <int G>
__global__ void __launch_bounds__(kAttnThreads)
attn_decode_kernel(const AttnArgs a) {
  extern __shared__ __align__(16) float sm[];
  using L = AttnSmem<G>;
  float2 *cs = reinterpret_cast<float2 *>(sm + L::kCs);
  float *q_sm = sm + L::kQ;
  float *kn_sm = sm + L::kKn;
  float *sc = sm + L::kSc;
  float *wacc = sm + L::kWacc;
  float *red = sm + L::kRed;
  __shared__ int s_last;

  const int c = blockIdx.x, g = blockIdx.y;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int hl = lane & 15, half = lane >> 4;
  constexpr int D = kAttnD;

  // Every input may come from the preceding kernel (the q|k|v GEMV, an
  // update of the position, the previous step's append).
  pdl_wait();
  pdl_trigger();

  const int p = *a.pos;
  const bool valid = p >= 0 && p < a.S;
  int n_eff = 0, j0 = 0, j1 = 0;
  if (valid) {
    const int len = p + 1;
    n_eff = min(a.n_split, (len + kAttnMinChunk - 1) / kAttnMinChunk);
    if (c < n_eff) {
      j0 = int(int64_t(c) * len / n_eff);
      j1 = int(int64_t(c + 1) * len / n_eff);
    }
  }
  const int n = j1 - j0;  // positions of this CTA (<= kAttnMaxChunk)
  float *part = a.part + (size_t(g) * a.n_split + c) * G * (D + 2);
  const size_t head_row = size_t(g) * a.S;  // row 0 of KV head g

  if (n > 0) {
    // ---- RoPE: pair angles, rotated queries, the new key (CTA holding p)
    if (tid < kAttnPairs) {
      float sn, cn;
      sincosf(__fmul_rn(float(p), a.freq[tid]), &sn, &cn);
      cs[tid] = make_float2(cn, sn);
    }
    __syncthreads();
    for (int e = tid; e < G * kAttnPairs; e += kAttnThreads) {
      const int h = e / kAttnPairs, i = e - h * kAttnPairs;
      const __nv_bfloat16 *qh = a.qkv + size_t(g * G + h) * D;
      const float x0 = __bfloat162float(qh[2 * i]);
      const float x1 = __bfloat162float(qh[2 * i + 1]);
      const float2 r = cs[i];
      q_sm[h * D + 2 * i] = x0 * r.x - x1 * r.y;
      q_sm[h * D + 2 * i + 1] = x0 * r.y + x1 * r.x;
    }
    const bool has_p = j0 <= p && p < j1;
    if (has_p && tid < kAttnPairs) {
      const int i = tid;
      const __nv_bfloat16 *kh = a.qkv + size_t(a.H + g) * D;
      const __nv_bfloat16 *vh = a.qkv + size_t(a.H + a.Hkv + g) * D;
      const float x0 = __bfloat162float(kh[2 * i]);
      const float x1 = __bfloat162float(kh[2 * i + 1]);
      const float2 r = cs[i];
      const __nv_bfloat16 k0 = __float2bfloat16_rn(x0 * r.x - x1 * r.y);
      const __nv_bfloat16 k1 = __float2bfloat16_rn(x0 * r.y + x1 * r.x);
      kn_sm[2 * i] = __bfloat162float(k0);
      kn_sm[2 * i + 1] = __bfloat162float(k1);
      __nv_bfloat16 *krow = a.kc + (head_row + p) * D;
      __nv_bfloat16 *vrow = a.vc + (head_row + p) * D;
      krow[2 * i] = k0;
      krow[2 * i + 1] = k1;
      vrow[2 * i] = vh[2 * i];
      vrow[2 * i + 1] = vh[2 * i + 1];
    }
    __syncthreads();

    // ---- scores: a half-warp per position, 8 dims per lane ----
    float qr[G][8];
#pragma unroll
    for (int h = 0; h < G; ++h)
#pragma unroll
      for (int e = 0; e < 8; ++e) qr[h][e] = q_sm[h * D + 8 * hl + e];
    for (int jb = 2 * warp; jb < n; jb += 2 * kAttnWarps) {  // warp-uniform
      const int jj = jb + half;
      const bool act = jj < n;
      const int j = j0 + jj;
      float kv[8];
      if (act && j == p) {
#pragma unroll
        for (int e = 0; e < 8; ++e) kv[e] = kn_sm[8 * hl + e];
      } else if (act) {
        bf16x8_to_f32(__ldg(reinterpret_cast<const uint4 *>(
                          a.kc + (head_row + j) * D + 8 * hl)),
                      kv);
      } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) kv[e] = 0.0f;
      }
      float d[G];
#pragma unroll
      for (int h = 0; h < G; ++h) {
        float t = 0.0f;
#pragma unroll
        for (int e = 0; e < 8; ++e) t = fmaf(qr[h][e], kv[e], t);
        d[h] = t;
      }
#pragma unroll
      for (int h = 0; h < G; ++h)
#pragma unroll
        for (int o = 8; o > 0; o >>= 1)
          d[h] += __shfl_xor_sync(0xffffffffu, d[h], o);  // within the half
      if (act && hl == 0)
#pragma unroll
        for (int h = 0; h < G; ++h) sc[jj * G + h] = d[h] * a.inv_sqrt_d;
    }
    __syncthreads();

    // ---- softmax of the split: largest score, then exp and sum ----
    float m[G], l[G];
#pragma unroll
    for (int h = 0; h < G; ++h) m[h] = -INFINITY;
    for (int jj = tid; jj < n; jj += kAttnThreads)
#pragma unroll
      for (int h = 0; h < G; ++h) m[h] = fmaxf(m[h], sc[jj * G + h]);
    cta_reduce<G, true>(m, red);
#pragma unroll
    for (int h = 0; h < G; ++h) l[h] = 0.0f;
    for (int jj = tid; jj < n; jj += kAttnThreads)
#pragma unroll
      for (int h = 0; h < G; ++h) {
        const float e = expf(sc[jj * G + h] - m[h]);
        sc[jj * G + h] = e;
        l[h] += e;
      }
    cta_reduce<G, false>(l, red);  // its barriers also publish sc

    // ---- weighted values ----
    float acc[G][8];
#pragma unroll
    for (int h = 0; h < G; ++h)
#pragma unroll
      for (int e = 0; e < 8; ++e) acc[h][e] = 0.0f;
    for (int jb = 2 * warp; jb < n; jb += 2 * kAttnWarps) {
      const int jj = jb + half;
      if (jj < n) {
        const int j = j0 + jj;
        float vv[8];
        if (j == p) {
          const __nv_bfloat16 *vh = a.qkv + size_t(a.H + a.Hkv + g) * D;
#pragma unroll
          for (int e = 0; e < 8; ++e) vv[e] = __bfloat162float(vh[8 * hl + e]);
        } else {
          bf16x8_to_f32(__ldg(reinterpret_cast<const uint4 *>(
                            a.vc + (head_row + j) * D + 8 * hl)),
                        vv);
        }
#pragma unroll
        for (int h = 0; h < G; ++h) {
          const float w = sc[jj * G + h];
#pragma unroll
          for (int e = 0; e < 8; ++e) acc[h][e] = fmaf(w, vv[e], acc[h][e]);
        }
      }
    }
#pragma unroll
    for (int h = 0; h < G; ++h)
#pragma unroll
      for (int e = 0; e < 8; ++e)
        acc[h][e] += __shfl_xor_sync(0xffffffffu, acc[h][e], 16);
    if (half == 0)
#pragma unroll
      for (int h = 0; h < G; ++h)
#pragma unroll
        for (int e = 0; e < 8; ++e)
          wacc[(warp * G + h) * D + 8 * hl + e] = acc[h][e];
    __syncthreads();
#pragma unroll
    for (int h = 0; h < G; ++h) {  // thread tid: dim tid of every head
      float t = wacc[h * D + tid];
#pragma unroll
      for (int w = 1; w < kAttnWarps; ++w) t += wacc[(w * G + h) * D + tid];
      part[h * (D + 2) + 2 + tid] = t;
      if (tid == h) {
        part[h * (D + 2)] = m[h];
        part[h * (D + 2) + 1] = l[h];
      }
    }
  }

  // ---- the last CTA of KV head g merges the splits ----
  __threadfence();
  __syncthreads();
  if (tid == 0) {
    const unsigned int prev = atomicAdd(&a.count[g], 1u);
    s_last = prev == unsigned(a.n_split) - 1u;
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  if (tid == 0) a.count[g] = 0u;  // every CTA of this step has counted
  float *o = a.out + size_t(g) * G * D;
  if (!valid) {
#pragma unroll
    for (int h = 0; h < G; ++h) o[h * D + tid] = 0.0f;
    if (tid == 0) atomicOr(a.err, kAttnErrPosition);
    return;
  }
  const float *pbase = a.part + size_t(g) * a.n_split * G * (D + 2);
  float mx[G], ls[G];
#pragma unroll
  for (int h = 0; h < G; ++h) mx[h] = -INFINITY;
  for (int cc = tid; cc < n_eff; cc += kAttnThreads)
#pragma unroll
    for (int h = 0; h < G; ++h)
      mx[h] = fmaxf(mx[h], __ldcg(pbase + (size_t(cc) * G + h) * (D + 2)));
  cta_reduce<G, true>(mx, red);
  float *wgt = sc;  // [n_eff][G] merge weights (n_eff <= 128 <= chunk)
#pragma unroll
  for (int h = 0; h < G; ++h) ls[h] = 0.0f;
  for (int cc = tid; cc < n_eff; cc += kAttnThreads)
#pragma unroll
    for (int h = 0; h < G; ++h) {
      const float *pc = pbase + (size_t(cc) * G + h) * (D + 2);
      const float w = expf(__ldcg(pc) - mx[h]);
      wgt[cc * G + h] = w;
      ls[h] += w * __ldcg(pc + 1);
    }
  cta_reduce<G, false>(ls, red);  // its barriers also publish wgt
#pragma unroll
  for (int h = 0; h < G; ++h) {  // thread tid: dim tid of every head
    float t = 0.0f;
    for (int cc = 0; cc < n_eff; ++cc)
      t = fmaf(wgt[cc * G + h],
               __ldcg(pbase + (size_t(cc) * G + h) * (D + 2) + 2 + tid), t);
    o[h * D + tid] = t / ls[h];
  }
}

template <int G>
cudaError_t launch_g(const AttnArgs &a, cudaStream_t stream) {
  static bool configured[64];
  auto kernel = attn_decode_kernel<G>;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!configured[dev]) {
    e = cudaFuncSetAttribute(kernel,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             int(AttnSmem<G>::kBytes));
    if (e != cudaSuccess) return e;
    configured[dev] = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(a.n_split), unsigned(a.Hkv));
  cfg.blockDim = dim3(kAttnThreads);
  cfg.dynamicSmemBytes = AttnSmem<G>::kBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, a);
}

size_t part_bytes(int H, int Hkv, int S) {
  const size_t b = size_t(Hkv) * attn_splits(S) * size_t(H / Hkv) *
                   (kAttnD + 2) * sizeof(float);
  return (b + 255) / 256 * 256;
}

bool aligned(const void *p, uintptr_t a) {
  return reinterpret_cast<uintptr_t>(p) % a == 0;
}

bw_status check_attn_shape(int H, int Hkv, int D, int S) {
  if (H < 1 || Hkv < 1 || D < 1 || S < 1) return BW_ERR_INVALID_ARG;
  if (H % Hkv != 0) return BW_ERR_INVALID_ARG;
  const int G = H / Hkv;
  if (D != kAttnD || (G != 1 && G != 2 && G != 4 && G != 8) ||
      Hkv > BW_ATTN_MAX_KV_HEADS || S > BW_ATTN_MAX_S)
    return BW_ERR_UNSUPPORTED_SHAPE;
  return BW_OK;
}

}  // namespace
}  // namespace bw

using namespace bw;

extern "C" size_t bw_attn_workspace_bytes(int H, int Hkv, int D, int S) {
  if (check_attn_shape(H, Hkv, D, S) != BW_OK) return 0;
  return part_bytes(H, Hkv, S) + size_t(Hkv) * sizeof(unsigned int);
}

extern "C" bw_status bw_attn_decode(const bw_bf16 *qkv, const int *pos, int H,
                                    int Hkv, int D, int S, float theta,
                                    bw_bf16 *k_cache, bw_bf16 *v_cache,
                                    float *out, void *workspace,
                                    size_t workspace_bytes,
                                    bw_stream_t stream) {
  if (!qkv || !pos || !k_cache || !v_cache || !out || !workspace)
    return BW_ERR_INVALID_ARG;
  bw_status st = check_attn_shape(H, Hkv, D, S);
  if (st != BW_OK) return st;
  if (!(theta > 0.0f) || !(theta < 3.0e38f)) return BW_ERR_INVALID_ARG;
  if (workspace_bytes < bw_attn_workspace_bytes(H, Hkv, D, S))
    return BW_ERR_INVALID_ARG;
  if (!aligned(qkv, 2) || !aligned(pos, 4) || !aligned(k_cache, 16) ||
      !aligned(v_cache, 16) || !aligned(out, 4) || !aligned(workspace, 16))
    return BW_ERR_MISALIGNED;

  AttnArgs a{};
  a.qkv = reinterpret_cast<const __nv_bfloat16 *>(qkv);
  a.pos = pos;
  a.kc = reinterpret_cast<__nv_bfloat16 *>(k_cache);
  a.vc = reinterpret_cast<__nv_bfloat16 *>(v_cache);
  a.out = out;
  a.part = static_cast<float *>(workspace);
  a.count = reinterpret_cast<unsigned int *>(
      static_cast<uint8_t *>(workspace) + part_bytes(H, Hkv, S));
  a.H = H;
  a.Hkv = Hkv;
  a.S = S;
  a.n_split = attn_splits(S);
  a.inv_sqrt_d = float(1.0 / sqrt(double(D)));
  for (int i = 0; i < kAttnPairs; ++i)
    a.freq[i] = float(pow(double(theta), -2.0 * i / double(D)));
  a.err = device_error_word();
  if (!a.err) {
    record_cuda_error(int(cudaErrorInvalidSymbol));
    return BW_ERR_CUDA;
  }
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cudaSuccess;
  switch (H / Hkv) {
    case 1: e = launch_g<1>(a, cs); break;
    case 2: e = launch_g<2>(a, cs); break;
    case 4: e = launch_g<4>(a, cs); break;
    default: e = launch_g<8>(a, cs); break;
  }
  if (e != cudaSuccess) {
    record_cuda_error(int(e));
    return BW_ERR_CUDA;
  }
  return BW_OK;
}
