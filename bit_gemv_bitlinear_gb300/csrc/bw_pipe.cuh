// bw_pipe.cuh -- the TMA-streamed W2A8 GEMV machinery shared by the public
// GEMV (bw_gemv_tma.cu) and the fused layer stack (bw_stack.cu).
//
// Source: "BitNet GPU 推理框架：从零构建 W2A8 的 2-bit 大模型 CUDA GEMV 内核",
// §5.2 (2-bit decode), §5.3 (dp4a dot product, shuffle reduction, scale
// epilogue).  The kernel template streams the packed weights; what feeds it
// (the int8 activations and their scales) and what it writes (bf16 outputs,
// int32 accumulators, or a residual update) are policies:
//
//   Prologue policy, called by every thread:
//     using Pre = ...;                        (state loaded before the wait)
//     __device__ Pre pre_wait() const;        (static inputs only)
//     template <int MT> __device__ void stage(const Pre &pre,
//         const StageCtx &c, int (&part)[MT]) const;  (after the wait)
//   stages MT int8 activation rows at c.xs + m c.xrow (zero from K up to
//   64 chunks), their scales in c.s_sm[m], and returns this thread's share
//   of sum_k x[m][k] in part[m].  It may use CTA barriers (__syncthreads)
//   and the 64 floats at c.red.  Loads issued right after the wait are
//   plain loads: a bulk copy here would queue behind the CTA's weight
//   copies in the TMA unit.
//
//   Epilogue policy:
//     __device__ float scale_value() const;   (after the wait)
//   scale_value() returns, for thread t < BW_MAX_WS, the t-th weight scale
//   (fp32) that finish() finds in ws_sm[t]; it is loaded before the
//   prologue and stored after it, so the two loads overlap.
//     __device__ float4 prefetch(const PipeArgs &a, int g_lo, int n_g) const;
//     template <int MT> __device__ void finish(const PipeArgs &a,
//         const int *tot, const int (&sx)[MT], int g_lo, int n_g,
//         const float *s_sm, const float *ws_sm, float *red,
//         float4 pre) const;
//   prefetch() runs right after the dependency wait, before the prologue;
//   whatever it returns reaches finish() of the same thread as `pre` (e.g.
//   a value of the thread's first output row, loaded early).  Issuing it
//   after the prologue measured 1 % slower on the stack.
//   finish() is called by every thread once the CTA's row totals are
//   complete: the exact int32 dot product of output n = 8 G + r (G =
//   phys_group(a, g_lo + gl)), row m, is tot[(gl MT + m) 8 + r] - sx[m].
//   It may use CTA barriers and the 64 floats at `red`.
#pragma once

#include <type_traits>

#include "bw_internal.cuh"

namespace bw {
namespace pipe {

constexpr long long kWaitLimitCycles = 2000000000LL;  // about one second

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)),
               "r"(count)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(
                   smem_addr(bar))
               : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar,
                                                      uint32_t bytes) {
  asm volatile(
      "mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(
          smem_addr(bar)),
      "r"(bytes)
      : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar,
                                              uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return done != 0;
}

// Wait for the phase of `parity` to complete, for at most `limit` cycles
// (about a second by default).
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity,
                                          long long limit = kWaitLimitCycles) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity))
    if (clock64() - t0 > limit) return false;
  return true;
}

__device__ __forceinline__ void bulk_copy_g2s(void *dst, const void *src,
                                              uint32_t bytes, uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes "
      "[%0], [%1], %2, [%3];" ::"r"(smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}

__device__ __forceinline__ void pdl_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;");
}

__device__ __forceinline__ int dp4a_us(uint32_t a, uint32_t b, int c) {
  int d;
  asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

// Activations in shared memory: row m, chunk j (64 int8 values) at byte
// m xrow + 64 j, zero beyond K.
__host__ __device__ inline uint32_t xs_row_bytes(int chunks) {
  return uint32_t(chunks) * 64u;
}

// Products of one chunk: 16 bytes of packed codes (row r, 64 weights) at
// wp against the 64 activations of each row m at xp + m xrow.
template <int MT>
__device__ __forceinline__ void dot_chunk(const uint8_t *wp, const int8_t *xp,
                                          uint32_t xrow, int (&acc)[MT][4]) {
  const uint4 wv = *reinterpret_cast<const uint4 *>(wp);
  const uint32_t wd[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
  for (int t = 0; t < 4; ++t) {
    const uint32_t c0w = wd[t] & 0x03030303u;
    const uint32_t c1w = wd[t] & 0x0c0c0c0cu;
    const uint32_t c2w = wd[t] & 0x30303030u;
    const uint32_t c3w = wd[t] & 0xc0c0c0c0u;
#pragma unroll
    for (int m = 0; m < MT; ++m) {
      // activation words 4t..4t+3 of the chunk: k = 64j + 16t + 4i + b
      const uint4 xv = *reinterpret_cast<const uint4 *>(xp + m * xrow + 16 * t);
      acc[m][0] = dp4a_us(c0w, xv.x, acc[m][0]);
      acc[m][1] = dp4a_us(c1w, xv.y, acc[m][1]);
      acc[m][2] = dp4a_us(c2w, xv.z, acc[m][2]);
      acc[m][3] = dp4a_us(c3w, xv.w, acc[m][3]);
    }
  }
}

// Dot products of `chunks` consecutive chunks of one row group held in
// shared memory at wbase, the first being chunk c0 of the row: lane (q, r)
// takes chunks 4 pq + q of row r.  acc[m][i] collects slot i (codes scaled
// by 4^i) against activation row m.  Two pointers advance by constants;
// only the last, partial quad is predicated.
template <int MT>
__device__ __forceinline__ void dot_row_group(const uint8_t *wbase,
                                              const int8_t *xs, uint32_t xrow,
                                              int c0, int chunks, int q,
                                              int r, int (&acc)[MT][4]) {
  const uint8_t *wp = wbase + q * kGroupChunkBytes + r * kChunkBytes;
  const int8_t *xp = xs + (c0 + q) * kChunkWeights;
  const int quads = chunks >> 2;
#pragma unroll 2
  for (int pq = 0; pq < quads; ++pq) {
    dot_chunk<MT>(wp, xp, xrow, acc);
    wp += 4 * kGroupChunkBytes;
    xp += 4 * kChunkWeights;
  }
  if (q < (chunks & 3)) dot_chunk<MT>(wp, xp, xrow, acc);
}

// Remove the slot factors: (((a3/4 + a2)/4 + a1)/4 + a0, exact because a_i is
// a multiple of 4^i; then sum the 4 chunk lanes of the row.
__device__ __forceinline__ int fold_row(const int (&a)[4]) {
  int v = ((((a[3] >> 2) + a[2]) >> 2) + a[1]) >> 2;
  v += a[0];
  v += __shfl_xor_sync(0xffffffffu, v, 8);
  v += __shfl_xor_sync(0xffffffffu, v, 16);
  return v;
}

// The default dot-product policy of the pipe kernel: unsigned codes masked
// in place and fed to dp4a against the int8 activations staged in shared
// memory (xs_chunk_bytes: shared-memory bytes per chunk of K and activation
// row; run: the products of a run of chunks; fold: a lane's partial sums to
// its share of the row value, summed over the row's 4 chunk lanes).
struct DotDp4a {
  static constexpr uint32_t kXsChunkBytes = 64;  // per activation row
  template <int MT>
  __device__ __forceinline__ static void run(const uint8_t *wbase,
                                             const int8_t *xs, uint32_t xrow,
                                             int c0, int chunks, int q, int r,
                                             int (&acc)[MT][4]) {
    dot_row_group<MT>(wbase, xs, xrow, c0, chunks, q, r, acc);
  }
  __device__ __forceinline__ static int fold(const int (&a)[4]) {
    return fold_row(a);
  }
};

// ---------------------------------------------------------------------------
// Balanced per-warp pipelines (pipe mode).
//
// CTA b owns the k consecutive row groups b k .. b k + k - 1 (the last CTA
// may own fewer); its 8 warps split the CTA's k C chunks into 8 contiguous,
// equal runs.  A warp walks its run in pieces of at most `slot_chunks`
// chunks that never cross a row-group boundary; each piece is one bulk copy
// into the next slot of the warp's own ring of `slots` slots.  Lane 0 of the
// warp issues the copies: the first `slots` pieces before
// griddepcontrol.wait, then piece i + slots into the slot of piece i as soon
// as the warp has read it, so each warp keeps slots - 1 pieces in flight
// whatever the other warps do.  When a piece ends a row group or the run, the
// warp folds its partial sums and adds them (int32, exact in any order) to
// the CTA's row totals in shared memory; one epilogue per CTA then scales
// and stores the k * 8 rows.  Every warp has the same amount of work and
// every CTA but the last the same number of groups, so no tail of the grid
// runs on a few warps with few bytes in flight.
struct PipeLayout {
  uint32_t ring, xs, sums, red, tot, bars, total;
};

// Chunks of the longest warp run of a CTA with k groups of `chunks` chunks.
__host__ __device__ inline int max_run_chunks(int k, int chunks, int warps) {
  return (k * chunks + warps - 1) / warps;
}

// xs: the staged activations, [MT][chunks] chunks for the CTA, or (per-warp
// staging) [warps][MT][max run] chunks, each warp its own run's;
// sums: [MT] activation scales s, [BW_MAX_WS] weight scales (as fp32),
// [warps][MT] per-warp activation sums; red: 64 floats of prologue
// reduction scratch; tot: [k][MT][8] row totals; bars: the ring barriers.
__host__ __device__ inline PipeLayout pipe_layout(
    int mt, int chunks, int slot_chunks, int slots, int warps, int k,
    uint32_t xs_chunk_bytes = DotDp4a::kXsChunkBytes, int per_warp_x = 0) {
  PipeLayout l;
  l.ring = 0;
  l.xs = uint32_t(warps * slots * slot_chunks) * kGroupChunkBytes;
  const uint32_t xs_chunks =
      per_warp_x ? uint32_t(warps) * uint32_t(max_run_chunks(k, chunks, warps))
                 : uint32_t(chunks);
  l.sums = l.xs + uint32_t(mt) * xs_chunks * xs_chunk_bytes;
  const uint32_t sums_bytes = uint32_t((mt + BW_MAX_WS + warps * mt) * 4);
  l.red = (l.sums + sums_bytes + 15) / 16 * 16;
  l.tot = l.red + 64 * 4;
  l.bars = l.tot + uint32_t(k * mt * 8 * 4);
  l.total = l.bars + uint32_t(warps * slots * 8);
  return l;
}

// What a prologue policy's stage() gets: the activation tile to fill, the
// scale slots and reduction scratch.
struct StageCtx {
  int8_t *xs;
  uint32_t xrow;
  int chunks;
  float *s_sm;
  float *red;
};

constexpr int kPipeWarps = 8;
constexpr int kPipeMaxGroupsPerCta = 256;
constexpr int kPipeMinGroupsPerCta = 2;  // fewer CTAs staging x for small N

// Orders this warp's earlier generic-proxy reads of a slot before the
// bulk copy (async proxy) that overwrites it.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Position in a warp's run: chunk u of the CTA's range = chunk c of the
// CTA's row group g.
struct RunCursor {
  int u, g, c;
  __device__ __forceinline__ int piece(int ks, int chunks, int end) const {
    return min(min(ks, chunks - c), end - u);
  }
  __device__ __forceinline__ void advance(int len, int chunks) {
    u += len;
    c += len;
    if (c == chunks) {
      c = 0;
      ++g;
    }
  }
};

// What the kernel streams and how it is split (see launch_pipe).
struct PipeArgs {
  const uint8_t *w;     // packed weights, device layout
  int N;                // output rows
  int chunks;           // C = ceil(K / 64)
  int n_groups;         // ceil(N / 8)
  int slot_chunks;      // chunks per piece (at most)
  int slots;            // ring slots per warp (caller's choice; 0: 2)
  int groups_per_cta;   // k
  int pair_half;        // 0, or H: group order 0, H, 1, H + 1, ... (2H groups)
  unsigned int *err;    // device error word (time-out bits)
  // 1: each warp stages only the activations of its own run, which touches
  // at most two row groups of every CTA (launch_pipe decides; prologues with
  // kPerWarpX only)
  int per_warp_x;
};

// Whether each of the 8 warp runs of a CTA with n_g groups of `chunks`
// chunks is at most one row long, so that it touches at most two row groups
// (the end of one and the start of the next).
__host__ __device__ inline bool runs_in_two_groups(int n_g, int chunks,
                                                   int warps) {
  const int U = n_g * chunks;
  for (int w = 0; w < warps; ++w)
    if (U * (w + 1) / warps - U * w / warps > chunks) return false;
  return true;
}

// Prologue policies that can stage per warp declare kPerWarpX = true.
template <class P, class = void>
struct has_per_warp_x : std::false_type {};
template <class P>
struct has_per_warp_x<P, std::void_t<decltype(P::kPerWarpX)>>
    : std::integral_constant<bool, P::kPerWarpX> {};

// Physical row group of the g-th group in streaming order.  With pair_half
// H the two halves of the rows are interleaved group by group, so that a
// CTA owning an even number of consecutive groups holds matching groups of
// both halves (e.g. gate and up rows of the same features).
__host__ __device__ __forceinline__ int phys_group(const PipeArgs &a, int g) {
  return a.pair_half ? (g >> 1) + (g & 1) * a.pair_half : g;
}

// Sum and maximum over the CTA's 8 warps in one exchange (fixed shuffle
// tree, then the 8 warp values in order); every thread gets both results.
// `red` holds 64 floats.
__device__ __forceinline__ void cta_sum_max(float &sum, float &mx,
                                            float *red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    sum += __shfl_xor_sync(0xffffffffu, sum, o);
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  }
  __syncthreads();
  if ((threadIdx.x & 31) == 0) {
    red[threadIdx.x >> 5] = sum;
    red[32 + (threadIdx.x >> 5)] = mx;
  }
  __syncthreads();
  sum = 0.0f;
  mx = 0.0f;
#pragma unroll
  for (int w = 0; w < kPipeWarps; ++w) {
    sum += red[w];
    mx = fmaxf(mx, red[32 + w]);
  }
}

// Deterministic reductions over the CTA's 8 warps (fixed shuffle tree, then
// the 8 warp values in order); `red` holds 32 floats; every thread returns
// the same value.
__device__ __forceinline__ float cta_sum(float v, float *red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  __syncthreads();
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  float t = 0.0f;
#pragma unroll
  for (int w = 0; w < kPipeWarps; ++w) t += red[w];
  return t;
}

__device__ __forceinline__ float cta_max(float v, float *red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1)
    v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  __syncthreads();
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  float t = 0.0f;
#pragma unroll
  for (int w = 0; w < kPipeWarps; ++w) t = fmaxf(t, red[w]);
  return t;
}

// kPW: the per-warp activation staging (a.per_warp_x set; prologues with
// kPerWarpX only), a kernel of its own so that the CTA-wide form keeps its
// registers.
template <int MT, class Pro, class Epi, class Dot = DotDp4a, bool kPW = false>
__global__ void __launch_bounds__(kPipeWarps * 32)
pipe_gemv_kernel(const PipeArgs a, const Pro pro, const Epi epi) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int KS = a.slot_chunks;
  const int R = a.slots;
  const int C = a.chunks;
  const int k = a.groups_per_cta;
  const uint32_t slot_bytes = uint32_t(KS) * kGroupChunkBytes;
  const uint32_t xrow = xs_row_bytes(C);
  constexpr bool kCanPerWarp = kPW && has_per_warp_x<Pro>::value;
  constexpr bool per_warp = kCanPerWarp;
  const PipeLayout L = pipe_layout(MT, C, KS, R, kPipeWarps, k,
                                   Dot::kXsChunkBytes, per_warp ? 1 : 0);
  uint8_t *ring = smem + L.ring + size_t(warp) * R * slot_bytes;
  int8_t *xs = reinterpret_cast<int8_t *>(smem + L.xs);
  float *s_sm = reinterpret_cast<float *>(smem + L.sums);
  float *ws_sm = s_sm + MT;
  int *sx_part = reinterpret_cast<int *>(ws_sm + BW_MAX_WS);  // [warps][MT]
  float *red = reinterpret_cast<float *>(smem + L.red);
  int *tot = reinterpret_cast<int *>(smem + L.tot);  // [k][MT][8]
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + L.bars) + warp * R;

  const int g_lo = int(blockIdx.x) * k;
  const int n_g = max(0, min(k, a.n_groups - g_lo));
  const int U = n_g * C;  // chunks of this CTA (k C <= 256 * 1024)
  const int run_lo = U * warp / kPipeWarps;
  const int run_hi = U * (warp + 1) / kPipeWarps;

  RunCursor iss;  // next piece to copy (lane 0)
  iss.u = run_lo;
  iss.g = run_lo / C;
  iss.c = run_lo - iss.g * C;
  RunCursor cur = iss;  // next piece to consume (whole warp)
  int issued = 0;
  auto issue_next = [&](int slot) {
    const int len = iss.piece(KS, C, run_hi);
    const uint32_t bytes = uint32_t(len) * kGroupChunkBytes;
    mbar_arrive_expect_tx(&full[slot], bytes);
    const size_t pg = size_t(phys_group(a, g_lo + iss.g));
    bulk_copy_g2s(ring + size_t(slot) * slot_bytes,
                  a.w + (pg * C + iss.c) * kGroupChunkBytes, bytes,
                  &full[slot]);
    iss.advance(len, C);
    ++issued;
  };
  if (lane == 0) {
    for (int s = 0; s < R; ++s) mbar_init(&full[s], 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    // The weights are static once written (bw_repack synchronises its
    // stream): the first pieces are requested before the dependency wait.
    for (int s = 0; s < R && iss.u < run_hi; ++s) issue_next(s);
  }
  for (int t = threadIdx.x; t < n_g * MT * 8; t += blockDim.x) tot[t] = 0;
  // Per-warp staging: this warp's run covers chunks [xa_lo, xa_lo + len_a)
  // of the CTA's group g_a and chunks [0, len_b) of the next one; the warp
  // stages those activations in its own region, in that order, and needs no
  // CTA barrier after the dependency wait, so the zeroed totals are
  // published before it.
  const int g_a = run_lo / C;
  const int xa_lo = run_lo - g_a * C;
  const int len_a = min(run_hi - run_lo, C - xa_lo);
  const int len_b = (run_hi - run_lo) - len_a;
  const int max_run = max_run_chunks(k, C, kPipeWarps);
  const uint32_t xrow_w = uint32_t(max_run) * Dot::kXsChunkBytes;
  int8_t *xs_w = xs + size_t(warp) * MT * xrow_w;
  if (per_warp) __syncthreads();
  const typename Pro::Pre pro_pre = pro.pre_wait();
  pdl_wait();
  // Dependents may start their pre-wait part (their own weight requests)
  // once this grid's dependency has resolved: one launch of lookahead.
  // Triggering before the wait lets a chain run many launches ahead (1.8 %
  // more on alternating decode shapes, 17 % slower on back-to-back calls of
  // one small shape); triggering after staging is 1.5-3.4 % slower.
  pdl_trigger();

  const float wsv = epi.scale_value();
  const float4 pre = epi.prefetch(a, g_lo, n_g);
  int part[MT];
  // per-warp staging: the sums of the staged activations per row, of the
  // first group's segment and of the next group's
  int xsum_a[MT], xsum_b[MT];
#pragma unroll
  for (int m = 0; m < MT; ++m) xsum_a[m] = xsum_b[m] = 0;
  if constexpr (kCanPerWarp) {
    pro.template stage_warp<MT>(pro_pre, xs_w, xrow_w, xa_lo, len_a, len_b,
                                s_sm, xsum_a, xsum_b);
    if (threadIdx.x < BW_MAX_WS) ws_sm[threadIdx.x] = wsv;
    __syncwarp();  // the warp's activations staged, its barriers set up
  } else {
    const StageCtx sc{xs, xrow, C, s_sm, red};
    pro.template stage<MT>(pro_pre, sc, part);
    if (threadIdx.x < BW_MAX_WS) ws_sm[threadIdx.x] = wsv;
#pragma unroll
    for (int m = 0; m < MT; ++m) {
#pragma unroll
      for (int o = 16; o > 0; o >>= 1)
        part[m] += __shfl_xor_sync(0xffffffffu, part[m], o);
      if (lane == 0) sx_part[warp * MT + m] = part[m];
    }
    __syncthreads();  // activations staged, totals zeroed, barriers set up
  }

  const int q = lane >> 3;  // chunk residue (relative to the piece) mod 4
  const int r = lane & 7;   // row inside the group
  int acc[MT][4];
#pragma unroll
  for (int m = 0; m < MT; ++m)
#pragma unroll
    for (int t = 0; t < 4; ++t) acc[m][t] = 0;
  bool ok = true;
  int consumed = 0, slot = 0;
  uint32_t phase = 0;
  while (cur.u < run_hi) {
    // warp-uniform outcome before any full-mask shuffle below
    if (!__all_sync(0xffffffffu, mbar_wait(&full[slot], phase))) {
      ok = false;
      break;
    }
    const int len = cur.piece(KS, C, run_hi);
    if (per_warp)
      Dot::template run<MT>(ring + size_t(slot) * slot_bytes, xs_w, xrow_w,
                            cur.g == g_a ? cur.c - xa_lo : len_a + cur.c, len,
                            q, r, acc);
    else
      Dot::template run<MT>(ring + size_t(slot) * slot_bytes, xs, xrow, cur.c,
                            len, q, r, acc);
    __syncwarp();
    if (lane == 0 && iss.u < run_hi) {  // piece consumed + R: this slot
      fence_proxy_async_smem();
      issue_next(slot);
    }
    const int g = cur.g;
    cur.advance(len, C);
    ++consumed;
    if (cur.c == 0 || cur.u == run_hi) {  // row group or run finished
#pragma unroll
      for (int m = 0; m < MT; ++m) {
        // per-warp staging: the warp folds each of its (at most two) groups
        // once, and the sum of the activations it covered there comes off
        const int v = Dot::fold(acc[m]) - (g == g_a ? xsum_a[m] : xsum_b[m]);
        if (q == 0) atomicAdd(&tot[(g * MT + m) * 8 + r], v);
#pragma unroll
        for (int t = 0; t < 4; ++t) acc[m][t] = 0;
      }
    }
    if (++slot == R) {
      slot = 0;
      phase ^= 1u;
    }
  }
  if (!ok && lane == 0) {
    atomicOr(a.err, 4u);
    // copies still in flight land before the CTA may leave
    for (int i = consumed; i < issued; ++i)
      if (!mbar_wait(&full[i % R], uint32_t(i / R) & 1u)) atomicOr(a.err, 2u);
  }
  __syncthreads();  // every partial sum is in `tot`

  int sx[MT];  // sum_k x[m][k] over the whole row (per-warp: already off)
#pragma unroll
  for (int m = 0; m < MT; ++m) {
    sx[m] = 0;
    if (!per_warp)
#pragma unroll
      for (int w = 0; w < kPipeWarps; ++w) sx[m] += sx_part[w * MT + m];
  }
  epi.template finish<MT>(a, tot, sx, g_lo, n_g, s_sm, ws_sm, red, pre);
}

// Epilogue: y[m][n] = bf16((acc / s[m]) * ws[seg(n)]) (IEEE fp32, round to
// nearest even), or the int32 accumulator itself.
template <bool ACC>
struct EpiOut {
  void *out;  // bf16 or int32 [m][out_ld]
  int out_ld;
  const __nv_bfloat16 *ws;
  WsSegments seg;

  __device__ __forceinline__ float scale_value() const {
    return (!ACC && int(threadIdx.x) < seg.n_ws)
               ? __bfloat162float(ws[threadIdx.x])
               : 0.0f;
  }
  __device__ __forceinline__ void store(int n, int m, int total,
                                        const float *s_sm,
                                        const float *ws_sm) const {
    if (ACC) {
      static_cast<int *>(out)[size_t(m) * out_ld + n] = total;
    } else {
      int sg = 0;
#pragma unroll
      for (int i = 1; i < BW_MAX_WS; ++i)
        if (i < seg.n_ws && n >= seg.bounds[i]) sg = i;
      const float scaled = static_cast<float>(total) / s_sm[m];
      const float v = scaled * ws_sm[sg];
      static_cast<__nv_bfloat16 *>(out)[size_t(m) * out_ld + n] =
          __float2bfloat16_rn(v);
    }
  }
  __device__ __forceinline__ float4 prefetch(const PipeArgs &, int,
                                             int) const {
    return make_float4(0.0f, 0.0f, 0.0f, 0.0f);
  }
  template <int MT>
  __device__ __forceinline__ void finish(const PipeArgs &a, const int *tot,
                                         const int (&sx)[MT], int g_lo,
                                         int n_g, const float *s_sm,
                                         const float *ws_sm, float *red,
                                         float4 pre) const {
    (void)red;
    (void)pre;
    for (int t = threadIdx.x; t < n_g * 8; t += blockDim.x) {
      const int gl = t >> 3, rr = t & 7;
      const int n = (g_lo + gl) * kGroupRows + rr;  // no row pairing here
      if (n < a.N) {
#pragma unroll
        for (int m = 0; m < MT; ++m)
          store(n, m, tot[(gl * MT + m) * 8 + rr] - sx[m], s_sm, ws_sm);
      }
    }
  }
};

// Sets the opt-in shared-memory size once per device and returns how many
// CTAs of `kernel` are resident on the device at once (at least one).
// configured: the caller's per-device flags for this kernel (host threads
// may race on them; setting the attribute twice is harmless).
template <class Kernel>
cudaError_t resident_ctas(Kernel kernel, std::atomic<bool> *configured,
                          int threads,
                          uint32_t smem, int64_t *resident) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!configured[dev].load(std::memory_order_relaxed)) {
    e = cudaFuncSetAttribute(kernel,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             227 * 1024);
    if (e != cudaSuccess) return e;
    configured[dev].store(true, std::memory_order_relaxed);
  }
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, threads,
                                                    smem) != cudaSuccess ||
      per_sm < 1)
    per_sm = 1;
  *resident = int64_t(per_sm) * device_sm_count();
  return cudaSuccess;
}

// Pieces of up to 4 KB.  Ring slots per warp are chosen by the caller
// (PipeArgs::slots, 2 if unset): 2 slots = 64 KB of ring per 8-warp CTA,
// about three CTAs per SM for K <= 8192; 3 slots keep more bytes in flight
// per warp at two CTAs per SM.
constexpr int kPipeSlotChunks = 32;
constexpr int kPipeDefaultSlots = 2;

// Shared memory of a launch with k groups per CTA; a launch fits while this
// is at most 227 KB for k = kPipeMaxGroupsPerCta.
inline uint32_t pipe_smem_bytes(int mt, int chunks, int slot_chunks,
                                int slots, int k,
                                uint32_t xs_chunk_bytes = DotDp4a::kXsChunkBytes,
                                int per_warp_x = 0) {
  return pipe_layout(mt, chunks, slot_chunks, slots, kPipeWarps, k,
                     xs_chunk_bytes, per_warp_x)
      .total;
}

// Launches the pipe kernel with programmatic dependent launch: k groups per
// CTA with k as small as the resident CTAs allow (at least
// kPipeMinGroupsPerCta, at most kPipeMaxGroupsPerCta; beyond that the grid
// runs in waves; even with pair_half), and pieces no longer than a warp's
// run.  Fills in the split fields of `a`; *grid_out (if set) receives the
// number of CTAs.
// Per-warp staging is taken where every run of every CTA touches at most two
// row groups, the per-warp activation regions stay small (at most 16 KB a CTA)
// and the CTAs resident per SM do not drop.
constexpr uint32_t kPipeMaxPerWarpXs = 16u * 1024u;

template <int MT, class Pro, class Epi, class Dot = DotDp4a>
cudaError_t launch_pipe(PipeArgs a, const Pro &pro, const Epi &epi,
                        cudaStream_t stream, int *grid_out = nullptr) {
  static std::atomic<bool> configured[64];
  static std::atomic<bool> configured_pw[64];
  auto kernel = pipe_gemv_kernel<MT, Pro, Epi, Dot, false>;
  a.slot_chunks = kPipeSlotChunks;
  if (a.slots < 1) a.slots = kPipeDefaultSlots;
  // k from the residency at k = 1, then once more at that k (the row
  // totals grow with k).
  int64_t k = 1, resident = 0;
  for (int pass = 0; pass < 2; ++pass) {
    cudaError_t e = resident_ctas(
        kernel, configured, kPipeWarps * 32,
        pipe_smem_bytes(MT, a.chunks, a.slot_chunks, a.slots, int(k),
                        Dot::kXsChunkBytes),
        &resident);
    if (e != cudaSuccess) return e;
    k = (a.n_groups + resident - 1) / resident;
    if (k > kPipeMaxGroupsPerCta) k = kPipeMaxGroupsPerCta;
    if (k < kPipeMinGroupsPerCta) k = kPipeMinGroupsPerCta;
    if (a.pair_half) k += k & 1;  // whole pairs per CTA
  }
  const int64_t grid = (a.n_groups + k - 1) / k;
  const int64_t run = (k * a.chunks + kPipeWarps - 1) / kPipeWarps;
  if (run < a.slot_chunks) a.slot_chunks = int(run < 1 ? 1 : run);
  a.groups_per_cta = int(k);
  if (grid_out) *grid_out = int(grid);
  a.per_warp_x = 0;
  if constexpr (has_per_warp_x<Pro>::value) {
    const int last_groups = int(a.n_groups - (grid - 1) * k);
    const uint32_t pw_xs = uint32_t(kPipeWarps) * uint32_t(MT) *
                           uint32_t(max_run_chunks(int(k), a.chunks, kPipeWarps)) *
                           Dot::kXsChunkBytes;
    if (pro.per_warp_capable() && pw_xs <= kPipeMaxPerWarpXs &&
        runs_in_two_groups(int(k), a.chunks, kPipeWarps) &&
        runs_in_two_groups(last_groups, a.chunks, kPipeWarps)) {
      auto kernel_pw = pipe_gemv_kernel<MT, Pro, Epi, Dot, true>;
      int64_t resident_pw = 0;
      const cudaError_t e = resident_ctas(
          kernel_pw, configured_pw, kPipeWarps * 32,
          pipe_smem_bytes(MT, a.chunks, a.slot_chunks, a.slots, int(k),
                          Dot::kXsChunkBytes, 1),
          &resident_pw);
      if (e != cudaSuccess) return e;
      int64_t resident_now = 0;
      const cudaError_t e2 = resident_ctas(
          kernel, configured, kPipeWarps * 32,
          pipe_smem_bytes(MT, a.chunks, a.slot_chunks, a.slots, int(k),
                          Dot::kXsChunkBytes),
          &resident_now);
      if (e2 != cudaSuccess) return e2;
      if (resident_pw >= resident_now) a.per_warp_x = 1;
    }
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(grid > 0 ? grid : 1));
  cfg.blockDim = dim3(kPipeWarps * 32);
  cfg.dynamicSmemBytes =
      pipe_smem_bytes(MT, a.chunks, a.slot_chunks, a.slots, int(k),
                      Dot::kXsChunkBytes, a.per_warp_x);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (a.per_warp_x)
    return cudaLaunchKernelEx(&cfg, pipe_gemv_kernel<MT, Pro, Epi, Dot, true>,
                              a, pro, epi);
  return cudaLaunchKernelEx(&cfg, kernel, a, pro, epi);
}

}  // namespace pipe
}  // namespace bw
