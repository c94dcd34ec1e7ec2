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
// at short ones.  Two kernels share the per-split work (attend_split):
//  * Caches of at most 4096 positions: one thread-block cluster of up to 16
//    CTAs per KV head (attn_cluster_kernel, described at its definition):
//    the splits merge through distributed shared memory.
//  * Longer caches: the kernel below, whose splits merge through the
//    caller's workspace (both kernels' split plans: bw_attn_plan.cuh):
//  * CTA (c, g) takes split c of the positions 0..p for KV head g and all
//    G = H / Hkv query heads that read it, so every K and V row is loaded
//    once for the G heads.  The number of splits is fixed at launch: one
//    CTA per SM over the KV heads where the cache allows (150 CTAs for 5 KV
//    heads on 152 SMs), never more than 160 positions per split.  The
//    position p is read on the device, so one launch serves every step of
//    a graph-replayed decode loop: a context of L tokens uses min(splits,
//    ceil(L / 64)) of them, the others are empty.  A context of at most 128
//    tokens takes one split, finished by that CTA alone straight from its
//    shared memory: no partial, fence, counter or merge.
//  * The rows of a split are contiguous in the cache: tiled copies (TMA, one
//    box per 32 rows and 64 dims, 128-byte swizzled) bring its keys and its
//    values into shared memory while the CTA rotates its queries; the keys
//    complete on their own mbarrier, so the scores start before the values
//    have landed.  Every wait is bounded.
//  * Scores and weighted values run on the tensor cores (mma.sync, bf16
//    operands from ldmatrix, fp32 accumulation): S = K q^T per 16-position
//    tile with the fp32 queries as a bf16 pair q_hi + q_lo, and out^T =
//    V^T P with the fp32 exp weights as a bf16 pair likewise, so both
//    products keep about 16 bits beyond one bf16 rounding.
//  * Inside a CTA the softmax has two passes over the scores in shared
//    memory (largest score, then exp and sum); the CTA writes its largest
//    scores m, exp sums l and unnormalised outputs to the workspace.
//  * The last CTA of KV head g to finish (a fence and an atomic counter;
//    nothing spins) merges the splits: out = sum_c e^(m_c - M) acc_c /
//    sum_c e^(m_c - M) l_c.  It loads every m and l at once, keeps the
//    weights in shared memory, then sums the outputs with 16-byte loads,
//    the splits shared between the two halves of the CTA; it sets the
//    counter back to zero.
//  * The CTA whose split holds p rotates the new key, rounds it to bf16 and
//    puts key and value into its staged rows and into row p of the cache.
// Arithmetic: fp32 (fp32 angles p * f_i with f_i = theta^(-2i/D) rounded
// to fp32 on the host, sincosf, expf, the softmax and the merges), bf16
// cache; the two contractions on the tensor cores take their fp32 operand
// (queries, exp weights) as a sum of two bf16 values and accumulate in fp32.
// The caches are read through tensor maps (encoded per launch: 2-D, Hkv S
// rows of D bf16).
#include "bw_attn_plan.cuh"
#include "bw_tc.cuh"

namespace bw {
namespace {

using pipe::pdl_trigger;
using pipe::pdl_wait;

constexpr int kAttnD = 128;             // head dim
constexpr int kAttnPairs = kAttnD / 2;
constexpr int kAttnThreads = 256;
constexpr int kAttnWarps = kAttnThreads / 32;
// Splits of a cache of S positions: at most ceil(S / 64) (the workspace is
// sized for that), at least ceil(S / kAttnChunk).
constexpr int kAttnMaxSplits = (BW_ATTN_MAX_S + kAttnMinChunk - 1) / kAttnMinChunk;
constexpr unsigned int kAttnErrPosition = 16u;  // device error word bit

struct AttnArgs {
  const __nv_bfloat16 *qkv;  // [(H + 2 Hkv) D]
  const int *pos;            // [1]
  __nv_bfloat16 *kc, *vc;    // [Hkv][S][D]
  float *out;                // [H][D]
  float *part;               // [Hkv][n_split] blocks of G (D + 4) floats
  unsigned int *count;       // [Hkv]
  int H, Hkv, S, n_split;
  float inv_sqrt_d;
  float freq[kAttnPairs];    // f_i = theta^(-2i/D), fp32
  unsigned int *err;
  // Optional (layer stack): statistics of the output for the next RMSNorm,
  // one entry per KV head: (sum of out^2, max |out * norm_gamma|).
  const float *norm_gamma;   // [H][D] or null
  float2 *norm_part;         // [Hkv] or null
  // Nonzero: *pos and the cache rows before it are final before the
  // preceding kernel on the stream starts (BW_ATTN_PAST_READY).
  int past_ready;
};

// BW_ATTN_PAST_READY: a position read after the dependency wait that
// differs from the one read before it means the caller's promise was
// broken (device error word bit).
constexpr unsigned int kAttnErrPastReady = 128u;

// With past_ready, after the dependency wait: early = {j0, n} of the plan
// thread 0 made from the position it read before the wait (its copies
// started when n > 0), pl the plan of the position read after it, which
// decides everything that follows.  If this CTA's rows differ, the early
// copies are of other rows: they are let land (bounded), the split's
// barriers invalidated, the broken promise reported, and the split copies
// its own rows as usual; if they do not land, the CTA gets no rows
// (pl.n = 0).  Returns whether the CTA's copies are in flight already.
// Every thread of the CTA calls it, after a barrier that publishes early.
__device__ __forceinline__ bool settle_early(const AttnArgs &a,
                                             const int *early, SplitPlan &pl,
                                             uint64_t *bar) {
  if (early[1] == 0) return false;
  if (early[0] == pl.j0 && early[1] == pl.n) return true;
  __shared__ int s_landed;
  if (threadIdx.x == 0) {
    const bool ok = pipe::mbar_wait(&bar[0], 0u) && pipe::mbar_wait(&bar[1], 0u);
    if (ok) {
      asm volatile("mbarrier.inval.shared::cta.b64 [%0];" ::"r"(
                       pipe::smem_addr(&bar[0]))
                   : "memory");
      asm volatile("mbarrier.inval.shared::cta.b64 [%0];" ::"r"(
                       pipe::smem_addr(&bar[1]))
                   : "memory");
    }
    atomicOr(a.err, ok ? kAttnErrPastReady : kAttnErrPastReady | 2u);
    s_landed = ok;
  }
  __syncthreads();
  if (!s_landed) pl.n = 0;
  return false;
}

// A split's partial: acc [G][D] (16-byte aligned rows), then m [G] and
// l [G], padded to G (D + 4) floats so that every block stays 16-byte
// aligned.
template <int G>
struct AttnPart {
  static constexpr int kStride = G * (kAttnD + 4);
  static constexpr int kM = G * kAttnD;
  static constexpr int kL = kM + G;
};

// Shared memory (bytes): staged key and value rows, pair cos/sin, rotated
// queries, scores (the merge reuses the key rows for its weights),
// per-warp outputs, reduction scratch.
template <int G, int kChunk = kAttnChunk>
struct AttnSmem {
  static constexpr uint32_t kRowBytes = kAttnD * 2;
  static constexpr uint32_t kK = 0;
  static constexpr uint32_t kV = kK + kChunk * kRowBytes;
  static constexpr uint32_t kCs = kV + kChunk * kRowBytes;      // float2[64]
  static constexpr uint32_t kQ = kCs + kAttnPairs * 8;          // [G][D]
  static constexpr uint32_t kSc = kQ + G * kAttnD * 4;          // [chunk][G]
  // the split's output [G][D]; the workspace merge's [threads] float4 sums
  static constexpr uint32_t kWacc = kSc + kChunk * G * 4;
  static constexpr uint32_t kWaccBytes =
      G * kAttnD * 4 > kAttnThreads * 16 ? G * kAttnD * 4 : kAttnThreads * 16;
  static constexpr uint32_t kRed = kWacc + kWaccBytes;
  static constexpr size_t kBytes = kRed + kAttnWarps * (G < 2 ? 2 : G) * 4 + 16;
};
// The merge keeps [splits][G] weights, [splits][G] exp sums and G totals
// in the staging rows.
static_assert((2 * kAttnMaxSplits * 8 + 8) * 4 <= 2 * kAttnChunk * kAttnD * 2,
              "merge scratch fits in the staging rows");

// Staged key and value rows: blocks of 32 rows, each two boxes (dims 0..63,
// 64..127) of 32 rows x 128 bytes in the 128-byte swizzle of the tiled copy:
// the 16-byte piece c of row r of a box is stored at piece c ^ (r mod 8).
constexpr int kAttnBlockRows = 32;
constexpr uint32_t kAttnBlockBytes = kAttnBlockRows * kAttnD * 2;  // 8 KB
__device__ __forceinline__ uint32_t staged_offset(int row, int dim) {
  const int r = row & (kAttnBlockRows - 1);
  return uint32_t(row / kAttnBlockRows) * kAttnBlockBytes +
         uint32_t(dim >> 6) * (kAttnBlockBytes / 2) + uint32_t(r) * 128u +
         ((uint32_t((dim & 63) >> 3) ^ uint32_t(r & 7)) << 4) +
         uint32_t(dim & 7) * 2u;
}

// Four 8x8 bf16 matrices from shared memory (lane l gives the row address
// of matrix l / 8), as mma fragments; .trans: transposed.
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile(
      "ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
      : "r"(addr)
      : "memory");
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile(
      "ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
      : "r"(addr)
      : "memory");
}

// C (16 x 8, fp32) += A (16 x 16, bf16, row-major) B (16 x 8, bf16).
__device__ __forceinline__ void mma_bf16(float (&c)[4], const uint32_t (&a)[4],
                                         uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
      "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t bf162_bits(__nv_bfloat162 v) {
  return *reinterpret_cast<const uint32_t *>(&v);
}

// Max (kMax) or sum over the CTA of G values per thread, in a fixed order;
// every thread receives the results.  `red` holds kAttnWarps * max(G, 2)
// floats.
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
  // No trailing barrier: the next writer of `red` is the next reduction,
  // whose first barrier comes after every thread has read these values.
}

// Sum and max of one value per thread over the CTA in one exchange (the
// next RMSNorm's statistics); `red` holds 2 kAttnWarps floats.
__device__ __forceinline__ void cta_sum_max(float &ss, float &mx, float *red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    ss += __shfl_xor_sync(0xffffffffu, ss, o);
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  }
  __syncthreads();
  if ((threadIdx.x & 31) == 0) {
    red[threadIdx.x >> 5] = ss;
    red[kAttnWarps + (threadIdx.x >> 5)] = mx;
  }
  __syncthreads();
  ss = red[0];
  mx = red[kAttnWarps];
#pragma unroll
  for (int w = 1; w < kAttnWarps; ++w) {
    ss += red[w];
    mx = fmaxf(mx, red[kAttnWarps + w]);
  }
}

// What a CTA of KV head g reads from the q|k|v vector: the query pairs it
// rotates (pair e = h D / 2 + i of the G heads, e = tid + u kAttnThreads)
// and, for tid < D / 2, pair tid of the new key and value.  Loaded right
// after the dependency wait together with the position, which they do not
// depend on, so the three loads overlap.  The vector is only 2-byte aligned:
// scalar loads.
template <int G>
struct QkvPre {
  static constexpr int kQ = (G * kAttnPairs + kAttnThreads - 1) / kAttnThreads;
  __nv_bfloat16 q[kQ][2];
  __nv_bfloat16 k[2], v[2];

  __device__ __forceinline__ void load(const AttnArgs &a, int g) {
    const int tid = threadIdx.x;
    const __nv_bfloat16 *qg = a.qkv + size_t(g) * G * kAttnD;
#pragma unroll
    for (int u = 0; u < kQ; ++u) {
      const int e = tid + u * kAttnThreads;
      const bool in = e < G * kAttnPairs;
      q[u][0] = in ? qg[2 * e] : __float2bfloat16_rn(0.0f);
      q[u][1] = in ? qg[2 * e + 1] : __float2bfloat16_rn(0.0f);
    }
    k[0] = k[1] = v[0] = v[1] = __float2bfloat16_rn(0.0f);
    if (tid < kAttnPairs) {
      const __nv_bfloat16 *kh = a.qkv + size_t(a.H + g) * kAttnD;
      const __nv_bfloat16 *vh = a.qkv + size_t(a.H + a.Hkv + g) * kAttnD;
      k[0] = kh[2 * tid];
      k[1] = kh[2 * tid + 1];
      v[0] = vh[2 * tid];
      v[1] = vh[2 * tid + 1];
    }
  }
};

// The copies of a split's n key rows and n value rows from cache row row0
// on (thread 0 only): 32-row blocks of two swizzled boxes of 64 dims each
// (tiled TMA), the keys on bar[0] and the values on bar[1], which it
// initialises.  Rows past the split (up to the end of its last block) come
// along; the split never uses them.
template <int G, int kChunk>
__device__ __forceinline__ void split_copies(const CUtensorMap *kmap,
                                             const CUtensorMap *vmap,
                                             int row0, int n, uint8_t *smem,
                                             uint64_t *bar) {
  using L = AttnSmem<G, kChunk>;
  uint8_t *kst = smem + L::kK;
  uint8_t *vst = smem + L::kV;
  const int nb = (n + kAttnBlockRows - 1) / kAttnBlockRows;
  pipe::mbar_init(&bar[0], 1);
  pipe::mbar_init(&bar[1], 1);
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  pipe::mbar_arrive_expect_tx(&bar[0], uint32_t(nb) * kAttnBlockBytes);
  pipe::mbar_arrive_expect_tx(&bar[1], uint32_t(nb) * kAttnBlockBytes);
  for (int b = 0; b < nb; ++b)
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      const int row = row0 + b * kAttnBlockRows;
      tma_load_2d(kst + b * kAttnBlockBytes + hh * (kAttnBlockBytes / 2),
                  kmap, hh * 64, row, &bar[0]);
      tma_load_2d(vst + b * kAttnBlockBytes + hh * (kAttnBlockBytes / 2),
                  vmap, hh * 64, row, &bar[1]);
    }
}

// The partial of one split, positions j0 .. j0 + n - 1 of KV head g (n >= 1,
// n <= kChunk): the tiled copies of its key and value rows (unless `issued`:
// thread 0 started them already, before the dependency wait), the rotated
// queries, the append of the new token when the split holds p, the scores,
// the split's softmax (largest score m and exp sum l per query head, the
// same in every thread) and its unnormalised output in the first wacc row
// of the layout.  pre: this thread's loads of the q|k|v vector.  bar: the
// split's two mbarriers.  Returns false if the key copy did not land (the
// CTA then has no partial).
template <int G, int kChunk>
__device__ __forceinline__ bool attend_split(const AttnArgs &a,
                                             const CUtensorMap *kmap,
                                             const CUtensorMap *vmap,
                                             const QkvPre<G> &pre, int g,
                                             int p, int j0, int n,
                                             bool issued, uint8_t *smem,
                                             uint64_t *bar, float (&m)[G],
                                             float (&l)[G]) {
  using L = AttnSmem<G, kChunk>;
  uint8_t *kst = smem + L::kK;
  uint8_t *vst = smem + L::kV;
  float2 *cs = reinterpret_cast<float2 *>(smem + L::kCs);
  float *q_sm = reinterpret_cast<float *>(smem + L::kQ);
  float *sc = reinterpret_cast<float *>(smem + L::kSc);
  float *wacc = reinterpret_cast<float *>(smem + L::kWacc);
  float *red = reinterpret_cast<float *>(smem + L::kRed);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  constexpr int D = kAttnD;
  const size_t head_row = size_t(g) * a.S;  // row 0 of KV head g
  const int n_mt = (n + 15) / 16;           // 16-position tiles
  // ---- the split's key rows and value rows ----
  if (tid == 0 && !issued)
    split_copies<G, kChunk>(kmap, vmap, int(head_row) + j0, n, smem, bar);
  // ---- RoPE of the queries meanwhile ----
  if (tid < kAttnPairs) {
    float sn, cn;
    sincosf(__fmul_rn(float(p), a.freq[tid]), &sn, &cn);
    cs[tid] = make_float2(cn, sn);
  }
  __syncthreads();  // cos/sin ready; the barriers are initialised
#pragma unroll
  for (int u = 0; u < QkvPre<G>::kQ; ++u) {
    const int e = tid + u * kAttnThreads;
    if (e < G * kAttnPairs) {
      const int h = e / kAttnPairs, i = e - h * kAttnPairs;
      const float x0 = __bfloat162float(pre.q[u][0]);
      const float x1 = __bfloat162float(pre.q[u][1]);
      const float2 r = cs[i];
      q_sm[h * D + 2 * i] = x0 * r.x - x1 * r.y;
      q_sm[h * D + 2 * i + 1] = x0 * r.y + x1 * r.x;
    }
  }
  const bool has_p = j0 <= p && p < j0 + n;
  if (!__syncthreads_and(pipe::mbar_wait(&bar[0], 0u))) {
    // Never expected: report, let the copies land (bounded) before the
    // CTA may leave, and contribute no partial.
    if (tid == 0) {
      atomicOr(a.err, 4u);
      if (!pipe::mbar_wait(&bar[0], 0u) || !pipe::mbar_wait(&bar[1], 0u))
        atomicOr(a.err, 2u);
    }
    __syncthreads();
    return false;
  }
  // ---- the new token's rotated key: staged and appended (the key copy has
  // landed, so neither write can be overwritten or read by it) ----
  if (has_p && tid < kAttnPairs) {
    const int i = tid;
    const float x0 = __bfloat162float(pre.k[0]);
    const float x1 = __bfloat162float(pre.k[1]);
    const float2 r = cs[i];
    const __nv_bfloat162 k2 = __halves2bfloat162(
        __float2bfloat16_rn(x0 * r.x - x1 * r.y),
        __float2bfloat16_rn(x0 * r.y + x1 * r.x));
    *reinterpret_cast<__nv_bfloat162 *>(kst + staged_offset(p - j0, 2 * i)) = k2;
    reinterpret_cast<__nv_bfloat162 *>(a.kc + (head_row + p) * D)[i] = k2;
  }
  __syncthreads();

  // ---- scores ----
  {
    // Tensor cores: S = K q^T per 16-position tile (the A operand, ldmatrix
    // from the swizzled rows) against the G rotated queries (the B operand,
    // heads padded to 8), bf16 with fp32 accumulation; the fp32 queries
    // enter as q_hi + q_lo (two bf16), so the products keep ~16 more bits
    // than q rounded once.
    const int fg = lane >> 2, ft = lane & 3;  // fragment row / column pair
    uint32_t qh[8][2], ql[8][2];
#pragma unroll
    for (int kk = 0; kk < 8; ++kk)
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        float x0 = 0.0f, x1 = 0.0f;
        if (fg < G) {
          const int d = 16 * kk + 2 * ft + 8 * u;
          x0 = q_sm[fg * D + d];
          x1 = q_sm[fg * D + d + 1];
        }
        const __nv_bfloat162 hi = __floats2bfloat162_rn(x0, x1);
        const __nv_bfloat162 lo = __floats2bfloat162_rn(
            x0 - __low2float(hi), x1 - __high2float(hi));
        qh[kk][u] = bf162_bits(hi);
        ql[kk][u] = bf162_bits(lo);
      }
    for (int mt = warp; mt < n_mt; mt += kAttnWarps) {
      // four independent accumulators (q_hi / q_lo, even / odd k-steps),
      // summed at the end: short dependency chains
      float c[4][4] = {};
      const int row = 16 * mt + (lane & 15);
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        uint32_t fa[4];
        ldsm_x4(pipe::smem_addr(kst + staged_offset(row, 16 * kk + 8 * (lane >> 4))),
                fa);
        mma_bf16(c[kk & 1], fa, qh[kk][0], qh[kk][1]);
        mma_bf16(c[2 + (kk & 1)], fa, ql[kk][0], ql[kk][1]);
      }
      // c0, c1: position 16 mt + fg, heads 2 ft, 2 ft + 1; c2, c3: + 8
#pragma unroll
      for (int v = 0; v < 4; ++v) {
        const int jj = 16 * mt + fg + 8 * (v >> 1), h = 2 * ft + (v & 1);
        const float t = (c[0][v] + c[1][v]) + (c[2][v] + c[3][v]);
        if (h < G && jj < n) sc[jj * G + h] = t * a.inv_sqrt_d;
      }
    }
  }
  __syncthreads();

  // ---- softmax of the split: largest score, then exp and sum ----
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

  // ---- weighted values (the value copy landed during the scores) ----
  if (!__syncthreads_and(pipe::mbar_wait(&bar[1], 0u))) {
    if (tid == 0) {
      atomicOr(a.err, 4u);
      if (!pipe::mbar_wait(&bar[1], 0u)) atomicOr(a.err, 2u);
    }
    __syncthreads();
  }
  // Rows n .. 16 ceil(n / 16) - 1 enter the products with weight 0; they
  // hold other positions (or rows not yet written), so they are zeroed: a
  // non-finite value there would not vanish.
  for (int e = tid; e < (16 * n_mt - n) * 16; e += kAttnThreads) {
    const int row = n + e / 16, q16 = e & 15;  // 16-byte pieces of the row
    *reinterpret_cast<uint4 *>(vst + staged_offset(row, 8 * q16)) =
        make_uint4(0u, 0u, 0u, 0u);
  }
  if (has_p && tid < kAttnPairs) {  // the new token's value
    const int i = tid;
    const __nv_bfloat162 v2 = __halves2bfloat162(pre.v[0], pre.v[1]);
    *reinterpret_cast<__nv_bfloat162 *>(vst + staged_offset(p - j0, 2 * i)) = v2;
    reinterpret_cast<__nv_bfloat162 *>(a.vc + (head_row + p) * D)[i] = v2;
  }
  __syncthreads();
  {
    // Tensor cores: out^T = V^T P.  Warp w owns dims 16 w .. 16 w + 15 (the
    // A operand: V^T, ldmatrix.trans from the swizzled rows) over all
    // positions, 16 per step (the B operand: the exp weights, heads padded
    // to 8, as p_hi + p_lo); the result is the split's whole output for its
    // dims, written to the first wacc row (no sum over warps).
    const int fg = lane >> 2, ft = lane & 3;
    const int d0 = 16 * warp;
    float c[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    float cl[4] = {0.0f, 0.0f, 0.0f, 0.0f};  // the p_lo products
    for (int ks = 0; ks < n_mt; ++ks) {
      uint32_t fa[4];
      ldsm_x4_t(pipe::smem_addr(vst + staged_offset(
                    16 * ks + ((lane >> 4) << 3) + (lane & 7),
                    d0 + (((lane >> 3) & 1) << 3))),
                fa);
      float w[4];
#pragma unroll
      for (int v = 0; v < 4; ++v) {  // P[16 ks + 2 ft + (v & 1) + 8 (v >> 1)][fg]
        const int jj = 16 * ks + 2 * ft + (v & 1) + 8 * (v >> 1);
        w[v] = (fg < G && jj < n) ? sc[jj * G + fg] : 0.0f;
      }
      const __nv_bfloat162 h01 = __floats2bfloat162_rn(w[0], w[1]);
      const __nv_bfloat162 h23 = __floats2bfloat162_rn(w[2], w[3]);
      const __nv_bfloat162 l01 = __floats2bfloat162_rn(
          w[0] - __low2float(h01), w[1] - __high2float(h01));
      const __nv_bfloat162 l23 = __floats2bfloat162_rn(
          w[2] - __low2float(h23), w[3] - __high2float(h23));
      mma_bf16(c, fa, bf162_bits(h01), bf162_bits(h23));
      mma_bf16(cl, fa, bf162_bits(l01), bf162_bits(l23));
    }
    // c0, c1: dim d0 + fg, heads 2 ft, 2 ft + 1; c2, c3: dim + 8
#pragma unroll
    for (int v = 0; v < 4; ++v) {
      const int h = 2 * ft + (v & 1), d = d0 + fg + 8 * (v >> 1);
      if (h < G) wacc[h * D + d] = c[v] + cl[v];
    }
  }
  __syncthreads();
  return true;
}

template <int G>
__global__ void __launch_bounds__(kAttnThreads)
attn_decode_kernel(const AttnArgs a, const __grid_constant__ CUtensorMap kmap,
                   const __grid_constant__ CUtensorMap vmap) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // the swizzled staging wants a 1024-byte aligned base
  uint8_t *smem = smem_raw + ((1024u - (pipe::smem_addr(smem_raw) & 1023u)) & 1023u);
  using L = AttnSmem<G>;
  using P = AttnPart<G>;
  __nv_bfloat16 *kst = reinterpret_cast<__nv_bfloat16 *>(smem + L::kK);
  __nv_bfloat16 *vst = reinterpret_cast<__nv_bfloat16 *>(smem + L::kV);
  float2 *cs = reinterpret_cast<float2 *>(smem + L::kCs);
  float *q_sm = reinterpret_cast<float *>(smem + L::kQ);
  float *sc = reinterpret_cast<float *>(smem + L::kSc);
  float *wacc = reinterpret_cast<float *>(smem + L::kWacc);
  float *red = reinterpret_cast<float *>(smem + L::kRed);
  __shared__ __align__(8) uint64_t bar[2];  // keys, values
  __shared__ int s_last;

  const int c = blockIdx.x, g = blockIdx.y;
  const int tid = threadIdx.x;
  constexpr int D = kAttnD;

  if (tid == 0) {  // the copies' descriptors, while the wait lasts
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&kmap))
                 : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&vmap))
                 : "memory");
  }
  // With past_ready the position and the cache rows before it are final
  // before the preceding kernel started: read the position and start the
  // split's copies while the dependency wait lasts.  Otherwise every input
  // may come from the preceding kernel (the q|k|v GEMV, an update of the
  // position, the previous step's append).
  __shared__ int s_early[2];  // thread 0's early plan: j0, n
  if (a.past_ready && tid == 0) {
    const SplitPlan e = ws_plan(__ldcg(a.pos), a.S, a.n_split, c);
    s_early[0] = e.j0;
    s_early[1] = e.n;
    if (e.n > 0)
      split_copies<G, kAttnChunk>(&kmap, &vmap, g * a.S + e.j0, e.n, smem, bar);
  }
  pdl_wait();
  pdl_trigger();

  QkvPre<G> pre;
  pre.load(a, g);
  const int p = __ldcg(a.pos);  // final now: the same plan in every CTA
  SplitPlan pl = ws_plan(p, a.S, a.n_split, c);
  bool issued = false;
  if (a.past_ready) {
    __syncthreads();  // s_early
    issued = settle_early(a, s_early, pl, bar);
  }
  const bool valid = pl.valid;
  const int n_eff = pl.n_eff, j0 = pl.j0;
  const int n = pl.n;  // positions of this CTA (<= kAttnChunk)
  float *part = a.part + (size_t(g) * a.n_split + c) * P::kStride;

  if (n > 0) {
    float m[G], l[G];
    if (attend_split<G, kAttnChunk>(a, &kmap, &vmap, pre, g, p, j0, n,
                                    issued, smem, bar, m, l)) {
      if (n_eff == 1) {
        // One split holds the whole context: its sums are final.  Write
        // the outputs (and the next RMSNorm's statistics) directly; no
        // partial, fence, counter or merge.
        float *o = a.out + size_t(g) * G * D;
        float ss = 0.0f, amx = 0.0f;
        for (int e = tid; e < G * D; e += kAttnThreads) {
          const float t = wacc[e];
          const int h = e / D;
          float lh = l[0];
#pragma unroll
          for (int hh = 1; hh < G; ++hh)
            if (hh == h) lh = l[hh];
          const float y = t / lh;
          o[e] = y;
          if (a.norm_part) {
            ss += y * y;
            amx = fmaxf(amx, fabsf(__fmul_rn(
                                 y, a.norm_gamma[size_t(g) * G * D + e])));
          }
        }
        if (a.norm_part) {
          cta_sum_max(ss, amx, red);
          if (tid == 0) a.norm_part[g] = make_float2(ss, amx);
        }
        return;
      }
      for (int e = tid; e < G * D; e += kAttnThreads)
        part[e] = wacc[e];  // [h][d]: e = h D + d
      if (tid < G) {
#pragma unroll
        for (int h = 0; h < G; ++h)
          if (tid == h) {
            part[P::kM + h] = m[h];
            part[P::kL + h] = l[h];
          }
      }
    }
  }
  // A single split finished the head above; the other CTAs have no work.
  if (valid && n_eff == 1) return;

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
    for (int e = tid; e < G * D; e += kAttnThreads) o[e] = 0.0f;
    if (tid == 0) {
      atomicOr(a.err, kAttnErrPosition);
      if (a.norm_part) a.norm_part[g] = make_float2(0.0f, 0.0f);
    }
    return;
  }
  const float *pbase = a.part + size_t(g) * a.n_split * P::kStride;
  // Thread (lane s, vec v) sums the splits s, s + kLanesPerVec, ... of
  // float4 v of the [G][D] block.  Its first 16 splits' outputs are loaded
  // before the weights are known: they do not depend on them.
  constexpr int kVec = G * D / 4;
  constexpr int kLanesPerVec = kAttnThreads / kVec;
  static_assert(kLanesPerVec * kVec == kAttnThreads, "vec lanes");
  const int v = tid % kVec, s_lane = tid / kVec;
  const int hv = v / (D / 4);
  float4 x[16];
#pragma unroll
  for (int u = 0; u < 16; ++u) {
    const int cc = s_lane + u * kLanesPerVec;
    x[u] = cc < n_eff ? __ldcg(reinterpret_cast<const float4 *>(
                                   pbase + size_t(cc) * P::kStride) + v)
                      : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
  }
  // Every split's m and l at once; weights w_c = e^(m_c - M) and the sums
  // sum_c w_c l_c, kept in the staging rows (free now).
  float *wgt = reinterpret_cast<float *>(smem + L::kK);  // [n_eff][G]
  float *lbuf = wgt + kAttnMaxSplits * G;                 // [n_eff][G]
  float *lsum = lbuf + kAttnMaxSplits * G;                // [G]
  float mx[G];
#pragma unroll
  for (int h = 0; h < G; ++h) mx[h] = -INFINITY;
  for (int e = tid; e < n_eff * G; e += kAttnThreads) {
    const int cc = e / G, h = e - cc * G;
    const float *pc = pbase + size_t(cc) * P::kStride;
    const float mv = __ldcg(pc + P::kM + h);
    wgt[e] = mv;
    lbuf[e] = __ldcg(pc + P::kL + h);
#pragma unroll
    for (int hh = 0; hh < G; ++hh)
      if (hh == h) mx[hh] = fmaxf(mx[hh], mv);
  }
  cta_reduce<G, true>(mx, red);  // its barriers also publish wgt and lbuf
  float ls[G];
#pragma unroll
  for (int h = 0; h < G; ++h) ls[h] = 0.0f;
  for (int e = tid; e < n_eff * G; e += kAttnThreads) {
    const int h = e % G;
    float w = 0.0f;
#pragma unroll
    for (int hh = 0; hh < G; ++hh)
      if (hh == h) w = expf(wgt[e] - mx[hh]);
    wgt[e] = w;  // the element this thread read
#pragma unroll
    for (int hh = 0; hh < G; ++hh)
      if (hh == h) ls[hh] = fmaf(w, lbuf[e], ls[hh]);
  }
  cta_reduce<G, false>(ls, red);  // its barriers also publish wgt
  if (tid < G) {
#pragma unroll
    for (int h = 0; h < G; ++h)
      if (tid == h) lsum[h] = ls[h];
  }
  float4 t = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
  for (int c0 = s_lane;; c0 += 16 * kLanesPerVec) {
#pragma unroll
    for (int u = 0; u < 16; ++u) {
      const int cc = c0 + u * kLanesPerVec;
      const float w = cc < n_eff ? wgt[cc * G + hv] : 0.0f;
      t.x = fmaf(w, x[u].x, t.x);
      t.y = fmaf(w, x[u].y, t.y);
      t.z = fmaf(w, x[u].z, t.z);
      t.w = fmaf(w, x[u].w, t.w);
    }
    if (c0 + 16 * kLanesPerVec >= n_eff) break;
#pragma unroll
    for (int u = 0; u < 16; ++u) {  // the next 16 splits of this lane
      const int cc = c0 + (16 + u) * kLanesPerVec;
      x[u] = cc < n_eff ? __ldcg(reinterpret_cast<const float4 *>(
                                     pbase + size_t(cc) * P::kStride) + v)
                        : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    }
  }
  float4 *mergebuf = reinterpret_cast<float4 *>(wacc);  // [lanes][kVec]
  mergebuf[s_lane * kVec + v] = t;
  __syncthreads();
  if (tid < kVec) {  // output float4 tid: the lanes' sums in order
    float4 sum = mergebuf[tid];
    for (int sl = 1; sl < kLanesPerVec; ++sl) {
      const float4 u = mergebuf[sl * kVec + tid];
      sum.x += u.x;
      sum.y += u.y;
      sum.z += u.z;
      sum.w += u.w;
    }
    const float inv = lsum[tid / (D / 4)];
    reinterpret_cast<float4 *>(o)[tid] =
        make_float4(sum.x / inv, sum.y / inv, sum.z / inv, sum.w / inv);
  }
  if (a.norm_part) {
    // The next RMSNorm's partial statistics over this head's G D outputs
    // (each thread re-reads what it stored), in a fixed order.
    float ss = 0.0f, amx = 0.0f;
    if (tid < kVec) {
      const float4 y = reinterpret_cast<const float4 *>(o)[tid];
      const float4 gm = reinterpret_cast<const float4 *>(
          a.norm_gamma + size_t(g) * G * D)[tid];
      ss = y.x * y.x + y.y * y.y + y.z * y.z + y.w * y.w;
      amx = fmaxf(fmaxf(fabsf(__fmul_rn(y.x, gm.x)), fabsf(__fmul_rn(y.y, gm.y))),
                  fmaxf(fabsf(__fmul_rn(y.z, gm.z)), fabsf(__fmul_rn(y.w, gm.w))));
    }
    cta_sum_max(ss, amx, red);
    if (tid == 0) a.norm_part[g] = make_float2(ss, amx);
  }
}

// ---------------------------------------------------------------------------
// Caches of at most kClMaxS positions: one thread-block cluster per KV head.
// CTA c owns slice c of the head's G D outputs (per outputs, a multiple of
// 4).  The CTAs take consecutive splits of positions 0..p (at least
// kClMinChunk each); as soon as its split is done a CTA pushes it through
// distributed shared memory: its m and l to every CTA, and each slice of its
// unnormalised output to the slice's owner.  After one cluster barrier every
// CTA merges its slice from its own shared memory.  With the layer stack's
// RMSNorm statistics, each CTA then stores its share into CTA 0's shared
// memory, and after a second barrier CTA 0 sums them in order.  No
// workspace, fence or counter, and no partial leaves the chip.  A barrier
// phase that every CTA arrives at before its split (and waits for before
// its first push) guarantees that all CTAs of the cluster have started
// before any shared memory of another is written.  Which positions each CTA
// takes (cl_plan) and how many CTAs a launch uses are in bw_attn_plan.cuh.

// Outputs per slice for a cluster of cl CTAs: ceil(G D / cl) rounded up to
// a multiple of 4 (so that slices move as 16-byte vectors).
template <int G>
__device__ __forceinline__ int cl_slice(int cl) {
  return ((G * kAttnD + cl - 1) / cl + 3) & ~3;
}

// The pushed partials after the split's layout: [cl][slice] outputs
// (cl * slice <= G D + 4 cl), [16][G] (m, l) pairs, [16] statistics.
template <int G, int kChunk>
struct ClSmem {
  using L = AttnSmem<G, kChunk>;
  static constexpr uint32_t kRecv = uint32_t((L::kBytes + 15) / 16 * 16);
  static constexpr uint32_t kMl = kRecv + (G * kAttnD + 4 * kClMaxCtas) * 4;
  static constexpr uint32_t kStats = kMl + kClMaxCtas * G * 8;
  static constexpr size_t kBytes = kStats + kClMaxCtas * 8;
};

__device__ __forceinline__ uint32_t cl_map(const void *p, int rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;"
               : "=r"(r)
               : "r"(pipe::smem_addr(p)), "r"(rank));
  return r;
}
__device__ __forceinline__ void cl_st2(uint32_t addr, float a, float b) {
  asm volatile("st.shared::cluster.v2.f32 [%0], {%1, %2};" ::"r"(addr),
               "f"(a), "f"(b)
               : "memory");
}
__device__ __forceinline__ void cl_st4(uint32_t addr, float4 v) {
  asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(addr),
               "f"(v.x), "f"(v.y), "f"(v.z), "f"(v.w)
               : "memory");
}
__device__ __forceinline__ void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile(
      "barrier.cluster.arrive.release.aligned;\n\t"
      "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

template <int G, int kChunk>
__global__ void __launch_bounds__(kAttnThreads)
attn_cluster_kernel(const AttnArgs a, const __grid_constant__ CUtensorMap kmap,
                    const __grid_constant__ CUtensorMap vmap) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // the swizzled staging wants a 1024-byte aligned base (the same offset in
  // every CTA, so distributed shared memory addresses still match)
  uint8_t *smem = smem_raw + ((1024u - (pipe::smem_addr(smem_raw) & 1023u)) & 1023u);
  using L = AttnSmem<G, kChunk>;
  using CS = ClSmem<G, kChunk>;
  float *wacc = reinterpret_cast<float *>(smem + L::kWacc);
  float *red = reinterpret_cast<float *>(smem + L::kRed);
  float *recv = reinterpret_cast<float *>(smem + CS::kRecv);
  float2 *ml = reinterpret_cast<float2 *>(smem + CS::kMl);
  float2 *stats = reinterpret_cast<float2 *>(smem + CS::kStats);
  __shared__ __align__(8) uint64_t bar[2];  // keys, values
  constexpr int D = kAttnD;
  const int c = blockIdx.x, g = blockIdx.y, cl = gridDim.x;  // c = rank
  const int tid = threadIdx.x;

  if (tid == 0) {  // the copies' descriptors, while the wait lasts
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&kmap))
                 : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&vmap))
                 : "memory");
  }
  // With past_ready the position and the cache rows before it are final
  // before the preceding kernel started: read the position and start the
  // split's copies while the dependency wait lasts.  Otherwise every input
  // may come from the preceding kernel.
  __shared__ int s_early[2];  // thread 0's early plan: j0, n
  if (a.past_ready && tid == 0) {
    const SplitPlan e = cl_plan(__ldcg(a.pos), a.S, cl, c, cl * kChunk);
    s_early[0] = e.j0;
    s_early[1] = e.n;
    if (e.n > 0)
      split_copies<G, kChunk>(&kmap, &vmap, g * a.S + e.j0, e.n, smem, bar);
  }
  pdl_wait();
  pdl_trigger();

  QkvPre<G> pre;
  pre.load(a, g);
  // final now: the same plan in every CTA of the cluster
  const int p = __ldcg(a.pos);
  SplitPlan pl = cl_plan(p, a.S, cl, c, cl * kChunk);
  bool issued = false;
  if (a.past_ready) {
    __syncthreads();  // s_early
    issued = settle_early(a, s_early, pl, bar);
  }
  const bool valid = pl.valid;
  float m[G], l[G];
#pragma unroll
  for (int h = 0; h < G; ++h) {
    m[h] = -INFINITY;
    l[h] = 0.0f;
  }
  if (pl.solo) {
    // ---- CTA 0 alone: the whole context, or zeros for a bad position ----
    if (c != 0) return;
    const bool have =
        pl.n > 0 && attend_split<G, kChunk>(a, &kmap, &vmap, pre, g, p, 0,
                                              pl.n, issued, smem, bar, m, l);
    float *o = a.out + size_t(g) * G * D;
    float ss = 0.0f, amx = 0.0f;
    for (int e = tid; e < G * D; e += kAttnThreads) {
      float y = 0.0f;
      if (have) {
        const float t = wacc[e];
        const int h = e / D;
        float lh = l[0];
#pragma unroll
        for (int hh = 1; hh < G; ++hh)
          if (hh == h) lh = l[hh];
        y = t / lh;
      }
      o[e] = y;
      if (a.norm_part) {
        ss += y * y;
        amx = fmaxf(amx,
                    fabsf(__fmul_rn(y, a.norm_gamma[size_t(g) * G * D + e])));
      }
    }
    if (a.norm_part) {
      cta_sum_max(ss, amx, red);
      if (tid == 0) a.norm_part[g] = make_float2(ss, amx);
    }
    if (!valid && tid == 0) atomicOr(a.err, kAttnErrPosition);
    return;
  }
  cluster_arrive_relaxed();  // this CTA has started
  const int n_eff = pl.n_eff, j0 = pl.j0, n = pl.n;
  const int per = cl_slice<G>(cl);
  // ---- this CTA's partial ----
  bool have = false;
  if (n > 0)
    have = attend_split<G, kChunk>(a, &kmap, &vmap, pre, g, p, j0, n,
                                     issued, smem, bar, m, l);
  cluster_wait();  // every CTA has started: its shared memory may be written
  if (c < n_eff) {
    // ---- pushed to the owners: output slices, then m and l to every CTA
    for (int e = 4 * tid; e < G * D; e += 4 * kAttnThreads) {
      float4 t = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
      if (have) t = *reinterpret_cast<const float4 *>(wacc + e);
      const int own = e / per;  // < cl: G D <= cl per
      cl_st4(cl_map(recv + c * per + (e - own * per), own), t);
    }
    if (tid < cl * G) {
      const int dst = tid / G, h = tid - dst * G;
      float mv = -INFINITY, lv = 0.0f;
      if (have)
#pragma unroll
        for (int hh = 0; hh < G; ++hh)
          if (hh == h) {
            mv = m[hh];
            lv = l[hh];
          }
      cl_st2(cl_map(ml + c * G + h, dst), mv, lv);
    }
  }
  cluster_sync_all();  // every partial of the head has been pushed

  // ---- merge: this CTA's slice, from its own shared memory ----
  const int e_lo = c * per, e_hi = min(G * D, e_lo + per);
  float *o = a.out + size_t(g) * G * D;
  float ss = 0.0f, amx = 0.0f;
  for (int e = e_lo + tid; e < e_hi; e += kAttnThreads) {
    const int h = e / D;
    float mx = -INFINITY;
    for (int cc = 0; cc < n_eff; ++cc) mx = fmaxf(mx, ml[cc * G + h].x);
    float lsum = 0.0f, acc = 0.0f;
    for (int cc = 0; cc < n_eff; ++cc) {
      const float2 v = ml[cc * G + h];
      const float w = expf(v.x - mx);
      lsum = fmaf(w, v.y, lsum);
      acc = fmaf(w, recv[cc * per + (e - e_lo)], acc);
    }
    const float y = acc / lsum;
    o[e] = y;
    if (a.norm_part) {
      ss += y * y;
      amx = fmaxf(amx, fabsf(__fmul_rn(y, a.norm_gamma[size_t(g) * G * D + e])));
    }
  }
  if (a.norm_part) {  // the same for every CTA of the launch
    cta_sum_max(ss, amx, red);
    if (tid == 0) cl_st2(cl_map(stats + c, 0), ss, amx);
    cluster_sync_all();  // every share is in CTA 0
    if (c == 0 && tid == 0) {
      float ts = 0.0f, tm = 0.0f;
      for (int cc = 0; cc < cl; ++cc) {
        ts += stats[cc].x;
        tm = fmaxf(tm, stats[cc].y);
      }
      a.norm_part[g] = make_float2(ts, tm);
    }
  }
}

// Whether clusters of kClMaxCtas CTAs of this kernel can be resident (once
// per device and size).
template <int G, int kChunk>
bool cluster_ok(int dev) {
  static std::atomic<int> state[64];  // 0 unknown, 1 yes, 2 no
  if (state[dev].load(std::memory_order_relaxed) == 0) {
    auto kernel = attn_cluster_kernel<G, kChunk>;
    constexpr size_t kSmem = ClSmem<G, kChunk>::kBytes + 1024;
    bool ok =
        cudaFuncSetAttribute(kernel,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             int(kSmem)) == cudaSuccess &&
        cudaFuncSetAttribute(kernel,
                             cudaFuncAttributeNonPortableClusterSizeAllowed,
                             1) == cudaSuccess;
    if (ok) {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(kClMaxCtas, 1);
      cfg.blockDim = dim3(kAttnThreads);
      cfg.dynamicSmemBytes = kSmem;
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = kClMaxCtas;
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = 1;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      int clusters = 0;
      ok = cudaOccupancyMaxActiveClusters(&clusters, kernel, &cfg) ==
               cudaSuccess &&
           clusters >= 1;
    }
    cudaGetLastError();  // a refused query is not an error of the call
    state[dev].store(ok ? 1 : 2, std::memory_order_relaxed);
  }
  return state[dev].load(std::memory_order_relaxed) == 1;
}

template <int G, int kChunk>
cudaError_t launch_cluster_g(const AttnArgs &a, const CUtensorMap &kmap,
                             const CUtensorMap &vmap, int cl,
                             cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(cl), unsigned(a.Hkv));
  cfg.blockDim = dim3(kAttnThreads);
  cfg.dynamicSmemBytes = ClSmem<G, kChunk>::kBytes + 1024;  // base alignment
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = unsigned(cl);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, attn_cluster_kernel<G, kChunk>, a, kmap,
                            vmap);
}

// The cluster kernel of staging kChunk for G, if its clusters fit.
template <int kChunk>
bool try_cluster(int G, int dev, const AttnArgs &a, const CUtensorMap &kmap,
                 const CUtensorMap &vmap, int cl, cudaStream_t stream,
                 cudaError_t *e) {
  switch (G) {
    case 1:
      if (!cluster_ok<1, kChunk>(dev)) return false;
      *e = launch_cluster_g<1, kChunk>(a, kmap, vmap, cl, stream);
      return true;
    case 2:
      if (!cluster_ok<2, kChunk>(dev)) return false;
      *e = launch_cluster_g<2, kChunk>(a, kmap, vmap, cl, stream);
      return true;
    case 4:
      if (!cluster_ok<4, kChunk>(dev)) return false;
      *e = launch_cluster_g<4, kChunk>(a, kmap, vmap, cl, stream);
      return true;
    default:
      if (!cluster_ok<8, kChunk>(dev)) return false;
      *e = launch_cluster_g<8, kChunk>(a, kmap, vmap, cl, stream);
      return true;
  }
}

template <int G>
cudaError_t launch_g(const AttnArgs &a, const CUtensorMap &kmap,
                     const CUtensorMap &vmap, cudaStream_t stream) {
  static std::atomic<bool> configured[64];
  auto kernel = attn_decode_kernel<G>;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!configured[dev].load(std::memory_order_relaxed)) {
    e = cudaFuncSetAttribute(kernel,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             int(AttnSmem<G>::kBytes + 1024));
    if (e != cudaSuccess) return e;
    configured[dev].store(true, std::memory_order_relaxed);
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(a.n_split), unsigned(a.Hkv));
  cfg.blockDim = dim3(kAttnThreads);
  cfg.dynamicSmemBytes = AttnSmem<G>::kBytes + 1024;  // base alignment
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, a, kmap, vmap);
}

// Partials for the most splits any device uses for this cache.
size_t part_bytes(int H, int Hkv, int S) {
  const size_t b = size_t(Hkv) * max_splits(S) * size_t(H / Hkv) *
                   (kAttnD + 4) * sizeof(float);
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

size_t attn_workspace_bytes(int H, int Hkv, int D, int S) {
  if (check_attn_shape(H, Hkv, D, S) != BW_OK) return 0;
  return part_bytes(H, Hkv, S) + size_t(Hkv) * sizeof(unsigned int);
}

cudaError_t launch_attn(const AttnLaunch &l, cudaStream_t stream) {
  const int sms = device_sm_count();
  if (sms <= 0) return cudaErrorNoDevice;
  AttnArgs a{};
  a.qkv = l.qkv;
  a.pos = l.pos;
  a.kc = l.kc;
  a.vc = l.vc;
  a.out = l.out;
  a.part = static_cast<float *>(l.workspace);
  a.count = reinterpret_cast<unsigned int *>(
      static_cast<uint8_t *>(l.workspace) + part_bytes(l.H, l.Hkv, l.S));
  a.H = l.H;
  a.Hkv = l.Hkv;
  a.S = l.S;
  a.n_split = attn_splits(l.S, l.Hkv, sms);
  a.inv_sqrt_d = float(1.0 / sqrt(double(kAttnD)));
  for (int i = 0; i < kAttnPairs; ++i)
    a.freq[i] = float(pow(double(l.theta), -2.0 * i / double(kAttnD)));
  a.err = device_error_word();
  if (!a.err) return cudaErrorInvalidSymbol;
  a.norm_gamma = l.norm_gamma;
  a.norm_part = l.norm_part;
  a.past_ready = l.past_ready ? 1 : 0;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  const int G = l.H / l.Hkv;
  // The caches as 2-D tensors of Hkv S rows of D bf16, boxes of 32 rows x 64
  // dims in the 128-byte swizzle (rows past the end read as zero).
  CUtensorMap kmap, vmap;
  if (!encode_2d(&kmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, l.kc, kAttnD,
                 uint64_t(l.Hkv) * uint64_t(l.S), kAttnD * 2, 64,
                 kAttnBlockRows, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_2d(&vmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, l.vc, kAttnD,
                 uint64_t(l.Hkv) * uint64_t(l.S), kAttnD * 2, 64,
                 kAttnBlockRows, CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  // The contexts this launch serves: every context of the cache, or (the
  // layer stack's short-context launches) at most l.max_len positions.
  const int max_len = (l.max_len > 0 && l.max_len < l.S) ? l.max_len : l.S;
  if (max_len <= kClMaxS) {  // one cluster per KV head, merged on chip
    cudaError_t le = cudaSuccess;
    if (max_len <= kClMaxCtas * kClChunkSmall && max_len < l.S) {
      // the smaller staging: CTAs of half the shared memory
      const int cl = cl_ctas_small(max_len);
      a.n_split = cl;
      if (try_cluster<kClChunkSmall>(G, dev, a, kmap, vmap, cl, stream, &le))
        return le;
    }
    const int cl = cl_ctas(max_len);
    a.n_split = cl;
    if (try_cluster<kClChunk>(G, dev, a, kmap, vmap, cl, stream, &le))
      return le;
    a.n_split = attn_splits(l.S, l.Hkv, sms);
  }
  switch (G) {
    case 1: return launch_g<1>(a, kmap, vmap, stream);
    case 2: return launch_g<2>(a, kmap, vmap, stream);
    case 4: return launch_g<4>(a, kmap, vmap, stream);
    default: return launch_g<8>(a, kmap, vmap, stream);
  }
}

bw_status check_attn(int H, int Hkv, int D, int S) {
  return check_attn_shape(H, Hkv, D, S);
}

}  // namespace bw

using namespace bw;

extern "C" size_t bw_attn_workspace_bytes(int H, int Hkv, int D, int S) {
  return attn_workspace_bytes(H, Hkv, D, S);
}

extern "C" bw_status bw_attn_decode_ex(const bw_bf16 *qkv, const int *pos,
                                       int H, int Hkv, int D, int S,
                                       float theta, bw_bf16 *k_cache,
                                       bw_bf16 *v_cache, float *out,
                                       void *workspace, size_t workspace_bytes,
                                       unsigned int flags,
                                       bw_stream_t stream) {
  if (!qkv || !pos || !k_cache || !v_cache || !out || !workspace)
    return BW_ERR_INVALID_ARG;
  if (flags & ~unsigned(BW_ATTN_PAST_READY)) return BW_ERR_INVALID_ARG;
  bw_status st = check_attn_shape(H, Hkv, D, S);
  if (st != BW_OK) return st;
  if (!(theta > 0.0f) || !(theta < 3.0e38f)) return BW_ERR_INVALID_ARG;
  if (workspace_bytes < attn_workspace_bytes(H, Hkv, D, S))
    return BW_ERR_INVALID_ARG;
  if (!aligned(qkv, 2) || !aligned(pos, 4) || !aligned(k_cache, 16) ||
      !aligned(v_cache, 16) || !aligned(out, 4) || !aligned(workspace, 16))
    return BW_ERR_MISALIGNED;
  AttnLaunch l{};
  l.qkv = reinterpret_cast<const __nv_bfloat16 *>(qkv);
  l.pos = pos;
  l.kc = reinterpret_cast<__nv_bfloat16 *>(k_cache);
  l.vc = reinterpret_cast<__nv_bfloat16 *>(v_cache);
  l.out = out;
  l.workspace = workspace;
  l.H = H;
  l.Hkv = Hkv;
  l.S = S;
  l.theta = theta;
  l.past_ready = (flags & BW_ATTN_PAST_READY) ? 1 : 0;
  const cudaError_t e =
      launch_attn(l, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) {
    record_cuda_error(int(e));
    return BW_ERR_CUDA;
  }
  return BW_OK;
}

extern "C" bw_status bw_attn_decode(const bw_bf16 *qkv, const int *pos, int H,
                                    int Hkv, int D, int S, float theta,
                                    bw_bf16 *k_cache, bw_bf16 *v_cache,
                                    float *out, void *workspace,
                                    size_t workspace_bytes,
                                    bw_stream_t stream) {
  return bw_attn_decode_ex(qkv, pos, H, Hkv, D, S, theta, k_cache, v_cache,
                           out, workspace, workspace_bytes, 0u, stream);
}
