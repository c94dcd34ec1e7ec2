// bw_gemv_tc.cu -- the W2A8 product for batched activations on the
// fifth-generation tensor cores (tcgen05.mma, accumulators in tensor
// memory).
//
// Same result as the CUDA-core GEMV: acc[m][n] = sum_k w[n][k] x[m][k]
// exactly, then y = bf16((acc / s[m]) * ws[seg(n)]).  Source: "BitNet GPU
// 推理框架：从零构建 W2A8 的 2-bit 大模型 CUDA GEMV 内核", §5.3 (product and scale
// epilogue), §4.2 (weight-scale segments); batching known tokens so that the
// weights are read once for all of them is the bytes-per-token report's
// "batched known tokens" item.
//
// One CTA owns 128 weight rows (16 row groups of the device layout) and all
// K, for a tile of T <= 128 tokens; per 256-k stage:
//  * one producer thread copies each stage's weights (a 2-D tensor-map box:
//    16 row groups x 512 bytes, issued before the dependency wait since the
//    weights are static) and tokens (T rows x 320 bytes, the 64 bytes past
//    the stage unused) into shared-memory rings, one tiled TMA copy each
//    (ring depths: TcCfg);
//  * 4 decode warps turn the 2-bit codes into fp16 and store them straight
//    into tensor memory: thread = weight row = TMEM lane, the MMA's A operand;
//  * 4 convert warps turn the int8 tokens into fp16 in the 128-byte-swizzled
//    K-major layout of the MMA's B operand, and sum each token's x;
//    (decode and convert warps come in two such sets, for the even and the
//    odd stages);
//  * one elected thread issues 16 tcgen05.mma (M = 128, N = T, K = 16) per
//    stage into a 128 x T fp32 accumulator in tensor memory.
// The decode and convert warps then read the accumulators back (tcgen05.ld)
// for the epilogue.
//
// Ring slots.  A shared-memory slot that a bulk copy refills is released only
// after every reading lane has issued fence.proxy.async: the readers load the
// stage with ordinary loads and use the values later, and the refill (async
// proxy) is not otherwise ordered after loads still in flight.
//
// Weight values.  fp16 bit patterns below 0x0800 are linear in the value
// (pattern * 2^-24: the subnormals and the first normal binade), so a code
// c = w + 1 left at bit 2 sl of a half (slot sl of the word interleave) and
// masked, pattern c 4^sl, is the fp16 c 4^sl 2^-24 exactly: one mask per two
// weights (plus one shift by 8 per word for the odd bytes), no table.  The
// token of that column is scaled by 4^-sl (exact in fp16), so every product
// is c x 2^-24, every partial sum an integer multiple of 2^-24 below 2^-2
// (|sum| <= 2 * 128 * K <= 2^22 for K <= 16384) and fp32 accumulation exact
// in any order; acc = 2^24 D - sum_k x (w = c - 1).
//
// Pair order.  Column j (0..7) of a 16-k step holds, in its low and high
// halves, the elements e and e + 2 of the packed word with e = 4 (j & 3) +
// (j >> 2) (byte j >> 2 and byte (j >> 2) + 2 of the word interleave, slot
// j & 3): the step's k order is the even elements, then the odd ones.  The
// token tile uses the same order and the column's scale 4^-(j & 3), so the
// sum is unchanged.
#include "bw_tc.cuh"

namespace bw {
namespace {

using namespace pipe;

// Decode and convert warps come in two sets of 4, one for the even stages
// and one for the odd ones: two stages in flight per role.
constexpr int kTcSetWarps = 4;
constexpr int kTcDecodeWarps = 2 * kTcSetWarps;                    // 0..7
constexpr int kTcConvertWarps = 2 * kTcSetWarps;                   // 8..15
constexpr int kTcProducerWarp = kTcDecodeWarps + kTcConvertWarps;  // 16
constexpr int kTcMmaWarp = kTcProducerWarp + 1;                    // 17
constexpr int kTcThreads = (kTcMmaWarp + 1) * 32;                  // 576
constexpr int kTcGroups = 16;          // row groups per CTA: 128 rows
constexpr int kTcStageChunks = 4;      // 256 k per stage
constexpr uint32_t kTcWStageBytes = kTcGroups * kTcStageChunks * kGroupChunkBytes;
constexpr uint32_t kTcTmemCols = 512;
// One CTA per SM: the tensor-memory allocation takes all 512 columns.
constexpr uint32_t kTcMinSmem = 120u * 1024u;

// Ring depths for a token tile of at most kMaxTokens tokens.  Up to 64
// tokens: 6 weight, 4 token and 3 operand stages.  Up to 128 tokens (N = 128
// MMAs): 2 of each, which is what fits in shared memory (two B stages are
// 128 KB) and in tensor memory (2 A stages + a 128-column accumulator).
template <int TM, int WS, int XS, int ABS, int XROW>
struct TcCfg {
  static constexpr int kMaxTokens = TM;
  // int8 token row of a stage in shared memory: 256 bytes, plus 64 where it
  // fits so that the convert warps' 16-byte reads of two adjacent tokens fall
  // in distinct bank groups.
  static constexpr uint32_t kXRow = XROW;
  static constexpr int kWStages = WS;     // weight stages in flight
  static constexpr int kXStages = XS;     // token stages in flight
  static constexpr int kABStages = ABS;   // fp16 operand stages (TMEM A, smem B)
  static constexpr uint32_t kDCol = ABS * 128;  // accumulator columns
  // Barrier indices.
  static constexpr int kBarFullW = 0;                        // [WS]
  static constexpr int kBarEmptyW = kBarFullW + WS;          // [WS]
  static constexpr int kBarFullX = kBarEmptyW + WS;          // [XS]
  static constexpr int kBarEmptyX = kBarFullX + XS;          // [XS]
  // A stage stored in TMEM and B stage in smem (decode + convert warps).
  static constexpr int kBarFullAB = kBarEmptyX + XS;         // [ABS]
  static constexpr int kBarDone = kBarFullAB + ABS;          // [ABS]
  static constexpr int kBarAcc = kBarDone + ABS;             // accumulators final
  static constexpr int kBarSums = kBarAcc + 1;  // token sums added, scales stored
  static_assert(kBarSums < 32, "barrier block");
  static_assert(kDCol + TM <= kTcTmemCols, "tensor memory");
};
using TcCfg64 = TcCfg<64, 6, 4, 3, 320>;
using TcCfg128 = TcCfg<128, 2, 2, 2, 320>;

// Shared-memory carve-up (offsets from a 1024-byte aligned base): weight
// ring, B ring (1024-aligned: the swizzle pattern is taken from the address),
// token ring, activation scales and their reciprocals, weight scales, token
// sums, TMEM address, barriers.
struct TcLayout {
  uint32_t w, b, x, s, r, ws, sx, tmem, bars, total;
};

template <class Cfg>
__host__ __device__ inline TcLayout tc_layout(int T) {
  TcLayout l;
  l.w = 0;
  l.b = l.w + Cfg::kWStages * kTcWStageBytes;
  l.x = l.b + Cfg::kABStages * uint32_t(T) * 512u;
  l.s = l.x + Cfg::kXStages * uint32_t(T) * Cfg::kXRow;  // fp32 s[m]
  l.r = l.s + Cfg::kMaxTokens * 4;                       // fp32 RN(1 / s[m])
  l.ws = l.r + Cfg::kMaxTokens * 4;
  l.sx = l.ws + BW_MAX_WS * 4;  // fp32 -sum_k x[m] (both stage sets)
  l.tmem = l.sx + Cfg::kMaxTokens * 4;
  l.bars = l.tmem + 16;
  l.total = l.bars + 32 * 8;
  return l;
}

// One launch: tokens [0, rows) (rows <= T <= Cfg::kMaxTokens, T a multiple
// of 16) of the activations at g.x (16-byte aligned rows, K % 16 == 0), all
// N outputs; CTA b owns row groups [16 b, 16 b + 16).
template <bool ACC, class Cfg>
__global__ void __launch_bounds__(kTcThreads, 1)
tc_gemv_kernel(const __grid_constant__ CUtensorMap wmap,
               const __grid_constant__ CUtensorMap xmap, const GemvArgs g,
               int rows, int T, unsigned int *err) {
  constexpr int kTcMaxTokens = Cfg::kMaxTokens;
  constexpr int kTcWStages = Cfg::kWStages;
  constexpr int kTcXStages = Cfg::kXStages;
  constexpr int kTcABStages = Cfg::kABStages;
  constexpr uint32_t kTcDCol = Cfg::kDCol;
  constexpr uint32_t kTcXRow = Cfg::kXRow;
  constexpr int kBarFullW = Cfg::kBarFullW, kBarEmptyW = Cfg::kBarEmptyW;
  constexpr int kBarFullX = Cfg::kBarFullX, kBarEmptyX = Cfg::kBarEmptyX;
  constexpr int kBarFullAB = Cfg::kBarFullAB, kBarDone = Cfg::kBarDone;
  constexpr int kBarAcc = Cfg::kBarAcc, kBarSums = Cfg::kBarSums;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t *smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  const TcLayout L = tc_layout<Cfg>(T);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int C = g.chunks;
  const int n_st = (C + kTcStageChunks - 1) / kTcStageChunks;
  const int g0 = int(blockIdx.x) * kTcGroups;
  const int n_grp = min(kTcGroups, g.n_groups - g0);
  uint64_t *bar = reinterpret_cast<uint64_t *>(smem + L.bars);
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L.tmem);
  float *s_sm = reinterpret_cast<float *>(smem + L.s);
  float *r_sm = reinterpret_cast<float *>(smem + L.r);
  float *ws_sm = reinterpret_cast<float *>(smem + L.ws);
  float *nsx_sm = reinterpret_cast<float *>(smem + L.sx);

  if (threadIdx.x == 0) {
    for (int i = 0; i < kTcWStages; ++i) {
      mbar_init(&bar[kBarFullW + i], 1);
      mbar_init(&bar[kBarEmptyW + i], kTcSetWarps);
    }
    for (int i = 0; i < kTcXStages; ++i) {
      mbar_init(&bar[kBarFullX + i], 1);
      mbar_init(&bar[kBarEmptyX + i], kTcSetWarps);
    }
    for (int i = 0; i < kTcABStages; ++i) {
      mbar_init(&bar[kBarFullAB + i], 2 * kTcSetWarps);
      mbar_init(&bar[kBarDone + i], 1);
    }
    mbar_init(&bar[kBarAcc], 1);
    mbar_init(&bar[kBarSums], kTcConvertWarps);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  // The two convert sets add their token sums here (before the barrier
  // below, so that every addition comes after the zero).
  if (threadIdx.x < kTcMaxTokens) nsx_sm[threadIdx.x] = 0.0f;
  if (warp == kTcMmaWarp) tmem_alloc(tmem_slot, kTcTmemCols);
  tc_fence_before();
  __syncthreads();  // barriers set up, tensor memory allocated
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  // Epilogue, run by the 8 decode and the 8 convert warps once the last MMA
  // is complete: warp (lane quarter q, part p of 4) reads accumulator
  // columns [p T/4, (p + 1) T/4) of weight rows 32 q .. 32 q + 31 and stores
  // acc = 2^24 D - sum_k x as int32 or as bf16((acc / s[m]) * ws[seg(n)]).
  // acc is exact in fp32 (an integer below 2^23); the quotient is the
  // correctly rounded one, from the token's reciprocal (div_by_recip) where
  // s is in its range, else by division.
  auto epilogue = [&](int q, int p) {
    const bool acc_ready = warp_wait(&bar[kBarAcc], 0u);
    const bool sums_ready = warp_wait(&bar[kBarSums], 0u);
    tc_fence_after();
    if (!(acc_ready && sums_ready)) {
      if (lane == 0) atomicOr(err, 4u);
      return;
    }
    const uint32_t t_lane = tmem + (uint32_t(32 * q) << 16);
    const int n = g0 * kGroupRows + 32 * q + lane;
    int sg = 0;
#pragma unroll
    for (int i = 1; i < BW_MAX_WS; ++i)
      if (i < g.seg.n_ws && n >= g.seg.bounds[i]) sg = i;
    const float wsv = ws_sm[sg];
    const int quarter = T / 4;  // a multiple of 4
    for (int j0 = p * quarter; j0 < (p + 1) * quarter; j0 += 4) {
      float d[4];
      tmem_ld4(t_lane + kTcDCol + uint32_t(j0), d);  // whole warp
      if (n >= g.N) continue;
      // the 4 results first (a token past `rows` has s = r = 1 and no token
      // sum, and is not stored), then the stores
      const float4 nx = lds4(nsx_sm + j0);
      const float a[4] = {fmaf(d[0], 16777216.0f, nx.x),
                          fmaf(d[1], 16777216.0f, nx.y),
                          fmaf(d[2], 16777216.0f, nx.z),
                          fmaf(d[3], 16777216.0f, nx.w)};
      int tv[4];
      float yv[4];
      if (ACC) {
#pragma unroll
        for (int e = 0; e < 4; ++e) tv[e] = __float2int_rn(a[e]);
      } else {
        const float4 s4 = lds4(s_sm + j0), r4 = lds4(r_sm + j0);
        const float sv[4] = {s4.x, s4.y, s4.z, s4.w};
        const float rv[4] = {r4.x, r4.y, r4.z, r4.w};
        // one branch per 4 tokens, the same in every lane
        if (rv[0] != 0.0f && rv[1] != 0.0f && rv[2] != 0.0f && rv[3] != 0.0f) {
#pragma unroll
          for (int e = 0; e < 4; ++e)
            yv[e] = div_by_recip(a[e], sv[e], rv[e]) * wsv;
        } else {
#pragma unroll
          for (int e = 0; e < 4; ++e)
            yv[e] = (rv[e] != 0.0f ? div_by_recip(a[e], sv[e], rv[e])
                                   : a[e] / sv[e]) *
                    wsv;
        }
      }
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int m = j0 + e;
        if (m >= rows) break;
        if (ACC)
          static_cast<int *>(g.out)[size_t(m) * g.out_ld + n] = tv[e];
        else
          static_cast<__nv_bfloat16 *>(g.out)[size_t(m) * g.out_ld + n] =
              __float2bfloat16_rn(yv[e]);
      }
    }
  };

  if (warp == kTcProducerWarp) {
    // ---- tiled copies: weight stages (static: before the wait), tokens ----
    if (lane == 0) {
      asm volatile("prefetch.tensormap [%0];" ::"l"(
                       reinterpret_cast<uint64_t>(&wmap))
                   : "memory");
      asm volatile("prefetch.tensormap [%0];" ::"l"(
                       reinterpret_cast<uint64_t>(&xmap))
                   : "memory");
    }
    auto issue_w = [&](int s) {
      const int slot = s % kTcWStages;
      mbar_arrive_expect_tx(&bar[kBarFullW + slot], kTcWStageBytes);
      tma_load_2d(smem + L.w + slot * kTcWStageBytes, &wmap,
                  s * kTcStageChunks * (kGroupChunkBytes / 8), g0,
                  &bar[kBarFullW + slot]);
    };
    auto issue_x = [&](int s) {
      const int slot = s % kTcXStages;
      mbar_arrive_expect_tx(&bar[kBarFullX + slot], uint32_t(T) * kTcXRow);
      tma_load_2d(smem + L.x + slot * uint32_t(T) * kTcXRow, &xmap,
                  s * kTcStageChunks * 16, 0, &bar[kBarFullX + slot]);
    };
    int sw = 0, sx = 0;
    if (lane == 0)
      for (; sw < kTcWStages && sw < n_st; ++sw) issue_w(sw);
    pdl_wait();
    pdl_trigger();
    if (lane == 0) {
      long long idle_since = clock64();
      while (sw < n_st || sx < n_st) {
        bool moved = false;
        if (sx < n_st &&
            (sx < kTcXStages ||
             mbar_try_wait(&bar[kBarEmptyX + sx % kTcXStages],
                           uint32_t(sx / kTcXStages - 1) & 1u))) {
          issue_x(sx++);
          moved = true;
        }
        if (sw < n_st &&
            mbar_try_wait(&bar[kBarEmptyW + sw % kTcWStages],
                          uint32_t(sw / kTcWStages - 1) & 1u)) {
          issue_w(sw++);
          moved = true;
        }
        if (moved) {
          idle_since = clock64();
        } else if (clock64() - idle_since > kWaitLimitCycles) {
          atomicOr(err, 4u);
          break;
        }
      }
      // Copies still in flight land before the CTA exits (their slots' last
      // phases; normally complete already).
      for (int s = max(0, sw - kTcWStages); s < sw; ++s)
        if (!mbar_wait(&bar[kBarFullW + s % kTcWStages],
                       uint32_t(s / kTcWStages) & 1u))
          atomicOr(err, 2u);
      for (int s = max(0, sx - kTcXStages); s < sx; ++s)
        if (!mbar_wait(&bar[kBarFullX + s % kTcXStages],
                       uint32_t(s / kTcXStages) & 1u))
          atomicOr(err, 2u);
    }
    __syncwarp();
  } else if (warp == kTcMmaWarp) {
    // ---- MMA issue: the warp runs the loop (uniform values), one elected
    // lane issues and commits ----
    pdl_wait();
    pdl_trigger();
    const uint32_t idesc = tc_idesc(T);
    const uint32_t b_ring = smem_addr(smem + L.b);
    const uint32_t slice16 = uint32_t(T) * 128u / 16u;  // slice, 16-byte units
    bool ok = true;
    for (int s = 0; s < n_st; ++s) {
      const int ab = s % kTcABStages;
      const uint32_t par = uint32_t(s / kTcABStages) & 1u;
      if (!warp_wait(&bar[kBarFullAB + ab], par)) {
        ok = false;
        break;
      }
      tc_fence_after();
      // One base descriptor per stage; the 16 k-steps add constants to its
      // address field (slice ks / 4 of T rows x 128 bytes, 32 bytes per step
      // within it).
      const int nks = 4 * min(kTcStageChunks, C - s * kTcStageChunks);
      const uint64_t bd0 = sw128_desc(b_ring + uint32_t(ab) * uint32_t(T) * 512u);
      const uint32_t a0 = tmem + uint32_t(ab) * 128u;
      if (elect_one()) {
#pragma unroll
        for (int ks = 0; ks < kTcStageChunks * 4; ++ks) {
          if (ks < nks)
            tc_mma(tmem + kTcDCol, a0 + uint32_t(ks) * 8u,
                   bd0 + uint64_t(uint32_t(ks >> 2) * slice16 + uint32_t(ks & 3) * 2u),
                   idesc, ks > 0 ? 1u : uint32_t(s > 0));
        }
        tc_commit(&bar[kBarDone + ab]);
      }
      __syncwarp();
    }
    if (!ok && lane == 0) atomicOr(err, 4u);
    if (elect_one()) tc_commit(&bar[kBarAcc]);  // also on a time-out
    __syncwarp();
  } else if (warp >= kTcDecodeWarps) {
    // ---- convert warps: int8 tokens -> swizzled fp16 B, token sums ----
    const int cw = (warp - kTcDecodeWarps) & 3;
    const int set = (warp - kTcDecodeWarps) >> 2;
    {
      // L2 prefetch of the token rows (a hint that returns no data, so it
      // may precede the dependency wait: the copies after it still see the
      // final values), one 128-byte line per thread across the grid.
      const size_t lo = reinterpret_cast<size_t>(g.x);
      const size_t base = lo & ~size_t(127);
      const size_t hi = lo + size_t(rows - 1) * g.x_ld + g.K;
      const int lines = int((hi - base + 127) / 128);
      const int nt = kTcConvertWarps * 32;
      for (int i = int(blockIdx.x) * nt + (threadIdx.x - kTcDecodeWarps * 32);
           i < lines; i += int(gridDim.x) * nt) {
        const size_t a = i == 0 ? lo : base + size_t(i) * 128;
        asm volatile("prefetch.global.L2 [%0];" ::"l"(a));
      }
    }
    pdl_wait();
    pdl_trigger();
    {
      const int t = threadIdx.x - kTcDecodeWarps * 32;  // 0..255
      if (!ACC && t < kTcMaxTokens) {
        const float sv = t < rows ? g.s[t] : 1.0f;
        s_sm[t] = sv;
        r_sm[t] = (sv >= 0x1p-60f && sv <= 0x1p60f) ? 1.0f / sv : 0.0f;
      }
      if (t < BW_MAX_WS)
        ws_sm[t] = t < g.seg.n_ws ? __bfloat162float(g.ws[t]) : 0.0f;
    }
    // Unit (m, gg): token m, 16 k at 16 gg of the stage.  A phase of 8
    // lanes covers gg & 3 = 0..3 for two adjacent tokens: conflict-free
    // reads (rows 320 bytes apart) and swizzled stores.
    const int gg = (lane & 3) + 4 * (lane >> 3);
    const int mpar = (lane >> 2) & 1;
    const int units = T / 8;  // per thread and stage
    int sum[kTcMaxTokens / 8];
#pragma unroll
    for (int i = 0; i < kTcMaxTokens / 8; ++i) sum[i] = 0;
    bool ok = true;
    for (int s = set; s < n_st && ok; s += 2) {
      const int xs = s % kTcXStages, ab = s % kTcABStages;
      if (!warp_wait(&bar[kBarFullX + xs], uint32_t(s / kTcXStages) & 1u)) {
        ok = false;
        break;
      }
      const int k = s * kTcStageChunks * 64 + 16 * gg;
      const uint8_t *xsrc = smem + L.x + xs * uint32_t(T) * kTcXRow + 16 * gg;
      uint4 v[kTcMaxTokens / 8];
#pragma unroll
      for (int i = 0; i < kTcMaxTokens / 8; ++i) {
        const int m = 2 * (cw + 4 * i) + mpar;
        v[i] = (i < units && m < rows && k < g.K)
                   ? *reinterpret_cast<const uint4 *>(xsrc + m * kTcXRow)
                   : make_uint4(0u, 0u, 0u, 0u);
      }
      fence_async_smem();  // as for the weight ring: reads done before a refill
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar[kBarEmptyX + xs]);
      if (s >= kTcABStages &&
          !warp_wait(&bar[kBarDone + ab], uint32_t(s / kTcABStages - 1) & 1u)) {
        ok = false;
        break;
      }
      uint8_t *bst = smem + L.b + ab * uint32_t(T) * 512u +
                     uint32_t(gg >> 2) * uint32_t(T) * 128u;
#pragma unroll
      for (int i = 0; i < kTcMaxTokens / 8; ++i) {
        if (i < units) {
          const int m = 2 * (cw + 4 * i) + mpar;
          const uint32_t wv[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
          uint32_t ev[4], od[4];
#pragma unroll
          for (int r = 0; r < 4; ++r) {
            sum[i] = __dp4a(int(wv[r]), 0x01010101, sum[i]);
            const uint32_t u = wv[r] ^ 0x80808080u;  // x + 128
            // (fp16(1024 + u) - 1152) 4^-r = x 4^-r exactly
            ev[r] = hfma2(prmt(u, 0x64646464u, 0x4240u), col_scale(r), col_bias(r));
            od[r] = hfma2(prmt(u, 0x64646464u, 0x4341u), col_scale(r), col_bias(r));
          }
          const uint32_t phys = uint32_t(2 * (gg & 3)) ^ uint32_t(m & 7);
          uint8_t *row = bst + m * 128;
          *reinterpret_cast<uint4 *>(row + phys * 16) =
              make_uint4(ev[0], ev[1], ev[2], ev[3]);
          *reinterpret_cast<uint4 *>(row + (phys ^ 1u) * 16) =
              make_uint4(od[0], od[1], od[2], od[3]);
        }
      }
      fence_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar[kBarFullAB + ab]);
    }
    if (!ok && lane == 0) atomicOr(err, 4u);
    // Token sums: the 16 lanes of one token parity (lane bits 0, 1, 3, 4).
#pragma unroll
    for (int i = 0; i < kTcMaxTokens / 8; ++i) {
      int v = sum[i];
      v += __shfl_xor_sync(0xffffffffu, v, 1);
      v += __shfl_xor_sync(0xffffffffu, v, 2);
      v += __shfl_xor_sync(0xffffffffu, v, 8);
      v += __shfl_xor_sync(0xffffffffu, v, 16);
      const int m = 2 * (cw + 4 * i) + mpar;
      if (i < units && (lane & ~4) == 0)
        atomicAdd(&nsx_sm[m], -static_cast<float>(v));  // exact: |v| < 2^22
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&bar[kBarSums]);
    epilogue(cw, 2 + set);
  } else {
    // ---- decode warps: 2-bit codes -> fp16 A in tensor memory ----
    pdl_trigger();
    const int q = warp & 3, h = warp >> 2;  // h: stage set, then column half
    const int r = 32 * q + lane;  // weight row of the tile = TMEM lane
    const uint32_t t_lane = tmem + (uint32_t(32 * q) << 16);
    bool ok = true;
    for (int s = h; s < n_st && ok; s += 2) {
      const int ws = s % kTcWStages, ab = s % kTcABStages;
      if (!warp_wait(&bar[kBarFullW + ws], uint32_t(s / kTcWStages) & 1u)) {
        ok = false;
        break;
      }
      const int nc = min(kTcStageChunks, C - s * kTcStageChunks);
      const uint8_t *src = smem + L.w + ws * kTcWStageBytes +
                           (r >> 3) * (kTcStageChunks * kGroupChunkBytes) +
                           (r & 7) * kChunkBytes;
      uint4 wq[kTcStageChunks];
#pragma unroll
      for (int c = 0; c < kTcStageChunks; ++c)
        wq[c] = c < nc ? *reinterpret_cast<const uint4 *>(src + c * kGroupChunkBytes)
                       : make_uint4(0u, 0u, 0u, 0u);
      // The slot is refilled by a bulk copy (async proxy) once released: the
      // loads above (generic proxy, values not used yet) must be complete and
      // ordered before that write, so every lane fences before the release.
      fence_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar[kBarEmptyW + ws]);
      if (s >= kTcABStages &&
          !warp_wait(&bar[kBarDone + ab], uint32_t(s / kTcABStages - 1) & 1u)) {
        ok = false;
        break;
      }
      tc_fence_after();
#pragma unroll
      for (int c = 0; c < kTcStageChunks; ++c) {
        if (c < nc) {
          uint32_t col[32];
          decode_word(wq[c].x, col);
          decode_word(wq[c].y, col + 8);
          decode_word(wq[c].z, col + 16);
          decode_word(wq[c].w, col + 24);
          tmem_st32(t_lane + uint32_t(ab) * 128u + uint32_t(c) * 32u, col);
        }
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar[kBarFullAB + ab]);
    }
    if (!ok && lane == 0) atomicOr(err, 4u);
    pdl_wait();
    epilogue(q, h);
  }
  tc_fence_before();
  __syncthreads();  // every tensor-memory access is done
  if (warp == kTcMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTcTmemCols);
  }
}



template <bool ACC, class Cfg>
cudaError_t launch_tc(const GemvArgs &g, int rows, int T, cudaStream_t stream) {
  static std::atomic<bool> configured[64];
  auto kernel = tc_gemv_kernel<ACC, Cfg>;
  unsigned int *err = device_error_word();
  if (!err) return cudaErrorInvalidSymbol;
  // 1 KB of slack to align the base; at least kTcMinSmem: one CTA per SM.
  uint32_t smem = tc_layout<Cfg>(T).total + 1024u;
  if (smem < kTcMinSmem) smem = kTcMinSmem;
  int64_t resident = 0;
  cudaError_t e = resident_ctas(kernel, configured, kTcThreads, smem, &resident);
  if (e != cudaSuccess) return e;
  // Weights: per row group, C chunks of 128 bytes as 16 C uint64; a box is
  // one stage of 16 groups.  Tokens: `rows` rows of K / 4 uint32; a box is
  // kXRow / 4 uint32 of T rows (rows past `rows`, k past K: zero).
  CUtensorMap wmap, xmap;
  if (!encode_2d(&wmap, CU_TENSOR_MAP_DATA_TYPE_UINT64, g.w,
                 uint64_t(g.chunks) * (kGroupChunkBytes / 8),
                 uint64_t(g.n_groups), uint64_t(g.chunks) * kGroupChunkBytes,
                 kTcStageChunks * (kGroupChunkBytes / 8), kTcGroups) ||
      !encode_2d(&xmap, CU_TENSOR_MAP_DATA_TYPE_UINT32, g.x, uint64_t(g.K / 4),
                 uint64_t(rows), uint64_t(g.x_ld), Cfg::kXRow / 4, uint32_t(T)))
    return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned((g.n_groups + kTcGroups - 1) / kTcGroups));
  cfg.blockDim = dim3(kTcThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, wmap, xmap, g, rows, T, err);
}

}  // namespace

static_assert(TcCfg128::kMaxTokens == kTcMaxRows, "largest token tile");

bool tc_fits(const GemvArgs &a) {
  return a.vec_x && a.K <= kMmaMaxK &&
         tc_layout<TcCfg64>(TcCfg64::kMaxTokens).total + 1024u <= 227u * 1024u &&
         tc_layout<TcCfg128>(TcCfg128::kMaxTokens).total + 1024u <= 227u * 1024u;
}

// Up to 64 tokens: the deep-ring configuration; 65..128: N = 128 MMAs with
// shallower rings.
cudaError_t launch_gemv_tc(const GemvArgs &a, int rows, bool acc_out,
                           cudaStream_t stream) {
  if (!tc_fits(a) || rows < 1 || rows > kTcMaxRows) return cudaErrorInvalidValue;
  const int T = (rows + 15) / 16 * 16;
  if (T <= TcCfg64::kMaxTokens)
    return acc_out ? launch_tc<true, TcCfg64>(a, rows, T, stream)
                   : launch_tc<false, TcCfg64>(a, rows, T, stream);
  return acc_out ? launch_tc<true, TcCfg128>(a, rows, T, stream)
                 : launch_tc<false, TcCfg128>(a, rows, T, stream);
}

}  // namespace bw
