// bw_gemm.cu -- the W2A8 product for prefill-sized batches of tokens (a few
// hundred to a few thousand) on the fifth-generation tensor cores, with
// 256-token tiles so that every decoded weight serves 256 tokens (and
// 64- or 128-token tiles for smaller batches).
//
// Source: "BitNet GPU 推理框架：从零构建 W2A8 的 2-bit 大模型 CUDA GEMV 内核",
// §一 (the model runs prefill and decode as separate paths; this is the
// prefill product in W2A8 instead of the page's BF16 matmul), §5.3 (the
// exact int32 product and the scale epilogue), §4.2 (weight-scale
// segments).  Same result as bw_gemv_w2a8: acc[m][n] = sum_k w[n][k] x[m][k]
// exactly, y = bf16((acc / s[m]) * ws[seg(n)]).
//
// Two launches per call:
//  * tok_fp16_kernel writes the tokens once as the MMA's fp16 operand into
//    the caller's workspace: per 16-k unit, the 16 values in the k order of
//    the weight decode, each scaled by 4^-slot (below), and the token sums
//    sum_k x.
//  * gemm_kernel: CTA (b, t) owns weight rows [128 b, 128 b + 128) and
//    tokens [T t, T t + T), over all K in stages of 128 k; T = 256 tokens
//    (64 or 128 for calls of at most 64 or 128 tokens):
//     - one producer thread streams each stage's weights (one 2-D box of 16
//       row groups x 256 bytes, issued before the dependency wait since the
//       weights are static) and tokens (two boxes of 64 k x T tokens,
//       128-byte swizzled by the copy itself: the layout the MMA reads) into
//       shared-memory rings with tiled TMA;
//     - 8 decode warps, two sets of 4 for the even and the odd stages
//       (thread = weight row = tensor-memory lane), turn the 2-bit codes into
//       fp16 and store them in tensor memory: the MMA's A operand;
//     - one elected thread issues 8 tcgen05.mma (M = 128, N = T, K = 16)
//       per stage into a 128 x T fp32 accumulator in tensor memory;
//       columns 0..T-1 hold it, then 4 A stages of 64 columns;
//     - the decode warps then read the accumulator back (tcgen05.ld) and
//       store acc = 2^24 D - sum_k x as int32, or the bf16 output; the
//       division by s is a product with 1 / s corrected to the IEEE
//       quotient (div_by_recip), so the outputs equal bw_gemv_w2a8's.
// Values (as in bw_gemv_tc.cu): a code c = w + 1 left in place at bit
// 2 sl of an fp16 half is the value c 4^sl 2^-24 (fp16 patterns below 0x0800
// are linear), the token of that k is x 4^-sl, so every product is
// c x 2^-24 and the fp32 accumulation is exact (|partial sums| < 2^22 units
// of 2^-24 for K <= 16384).  k order within a 16-k unit: column j of the
// weight word holds elements e, e + 2 with e = 4 (j & 3) + (j >> 2), slot
// j & 3; the token operand follows the same order.
#include "bw_tc.cuh"

namespace bw {
namespace {

constexpr int kGmRowGroups = 16;                 // 128 weight rows per CTA
constexpr int kGmStageChunks = 2;                // 128 k per stage
constexpr uint32_t kGmWStageBytes =
    kGmRowGroups * kGmStageChunks * kGroupChunkBytes;  // 4 KB
constexpr int kGmAStages = 4;
constexpr uint32_t kGmACols = kGmStageChunks * 32;  // fp16 pairs of a stage
constexpr uint32_t kGmTmemCols = 512;
// A and W slots are each used by one stage parity (one decode set).
static_assert(kGmAStages % 2 == 0, "stage sets");

constexpr int kGmSetWarps = 4;
constexpr int kGmDecodeWarps = 2 * kGmSetWarps;   // warps 0..7
constexpr int kGmProducerWarp = kGmDecodeWarps;   // 8
constexpr int kGmMmaWarp = kGmProducerWarp + 1;   // 9
constexpr int kGmThreads = (kGmMmaWarp + 1) * 32; // 320
constexpr int kGmMaxTokens = 256;                 // per-token arrays

// Per token tile: T tokens per CTA (the MMA's N: 64, 128 or 256), the ring
// depths, barrier indices and shared memory.  The smaller token stages of
// the small tiles leave room for deeper rings (more weight bytes in flight
// against HBM latency).
template <int T>
struct GmCfg {
  static constexpr uint32_t kSliceBytes = T * 128;  // 64 k x T tokens
  static constexpr uint32_t kBStageBytes = kGmStageChunks * kSliceBytes;
  static constexpr int kBStages = T == 256 ? 3 : (T == 128 ? 5 : 6);
  static constexpr int kWStages = T == 256 ? 6 : (T == 128 ? 8 : 16);
  static_assert(kWStages % 2 == 0, "stage sets");
  static constexpr uint32_t kAccCols = T;  // fp32, from column 0
  static_assert(T == 64 || T == 128 || T == 256, "token tile");
  static_assert(kAccCols + kGmAStages * kGmACols <= kGmTmemCols,
                "tensor memory");
  // Barrier indices.
  static constexpr int kBarFullW = 0;
  static constexpr int kBarEmptyW = kBarFullW + kWStages;
  static constexpr int kBarFullB = kBarEmptyW + kWStages;
  static constexpr int kBarEmptyB = kBarFullB + kBStages;
  static constexpr int kBarFullA = kBarEmptyB + kBStages;
  static constexpr int kBarDoneA = kBarFullA + kGmAStages;
  static constexpr int kBarAcc = kBarDoneA + kGmAStages;
  static constexpr int kBars = kBarAcc + 1;
  // Shared memory (offsets from a 1024-byte aligned base; the token
  // stages first, 1024-aligned as the swizzle requires).
  static constexpr uint32_t kSmB = 0;
  static constexpr uint32_t kSmW = kSmB + kBStages * kBStageBytes;
  static constexpr uint32_t kSmS = kSmW + kWStages * kGmWStageBytes;  // fp32 [256]
  static constexpr uint32_t kSmR = kSmS + kGmMaxTokens * 4;             // fp32 [256]
  static constexpr uint32_t kSmSx = kSmR + kGmMaxTokens * 4;            // fp32 [256]
  static constexpr uint32_t kSmWs = kSmSx + kGmMaxTokens * 4;           // fp32 [8]
  static constexpr uint32_t kSmTmem = kSmWs + BW_MAX_WS * 4;
  static constexpr uint32_t kSmBars = (kSmTmem + 16 + 7) / 8 * 8;
  static constexpr uint32_t kSmTotal = kSmBars + kBars * 8;
  static constexpr uint32_t kSmem = kSmTotal + 1024;  // slack for the base
  static_assert(kSmem <= 227u * 1024u, "shared memory");
};

// 32 consecutive accumulator columns of this warp's 32 lanes, loaded and
// waited for in one asm statement.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, "
      "%30, %31}, [%32];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]),
        "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]),
        "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
        "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]),
        "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
}

// Barrier among the 8 decode warps only (named barrier 1).
__device__ __forceinline__ void decode_warps_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(kGmDecodeWarps * 32) : "memory");
}

// Block m: token row m.  Per 16-k unit u (16 int8 at k = 16 u, zero past K),
// 16 fp16 at xb[m][16 u ..]: positions 2 r and 2 r + 1 hold x[4 r] and
// x[4 r + 2], positions 8 + 2 r and 9 + 2 r hold x[4 r + 1] and x[4 r + 3],
// each times 4^-r (exact: |x| <= 128).  sx[m] = sum_k x[m][k].
__global__ void __launch_bounds__(256)
tok_fp16_kernel(const int8_t *x, int x_ld, int K, int Kp, __half *xb,
                int *sx) {
  __shared__ int red[8];
  pdl_wait();  // the tokens may come from the preceding kernel
  pdl_trigger();
  const int m = blockIdx.x;
  const int8_t *xr = x + size_t(m) * x_ld;
  uint4 *dst = reinterpret_cast<uint4 *>(xb + size_t(m) * Kp);
  int sum = 0;
  for (int u = threadIdx.x; u < Kp / 16; u += blockDim.x) {
    uint32_t out[8];
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const int k = 16 * u + 4 * r;
      const uint32_t wv =
          k < K ? *reinterpret_cast<const uint32_t *>(xr + k) : 0u;  // K % 4 == 0
      sum = __dp4a(int(wv), 0x01010101, sum);
      const float sc = r == 0 ? 1.0f : (r == 1 ? 0.25f : (r == 2 ? 0.0625f : 0.015625f));
      const float v0 = float(int8_t(wv & 0xFFu)) * sc;
      const float v1 = float(int8_t((wv >> 8) & 0xFFu)) * sc;
      const float v2 = float(int8_t((wv >> 16) & 0xFFu)) * sc;
      const float v3 = float(int8_t(wv >> 24)) * sc;
      const __half2 ev = __halves2half2(__float2half_rn(v0), __float2half_rn(v2));
      const __half2 od = __halves2half2(__float2half_rn(v1), __float2half_rn(v3));
      out[r] = *reinterpret_cast<const uint32_t *>(&ev);
      out[4 + r] = *reinterpret_cast<const uint32_t *>(&od);
    }
    dst[2 * u] = make_uint4(out[0], out[1], out[2], out[3]);
    dst[2 * u + 1] = make_uint4(out[4], out[5], out[6], out[7]);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = sum;
  __syncthreads();
  if (threadIdx.x == 0) {
    int t = 0;
    for (int w = 0; w < int(blockDim.x >> 5); ++w) t += red[w];
    sx[m] = t;
  }
}

// One launch: CTA (b, t) computes outputs [256 t, 256 t + 256) x
// [128 b, 128 b + 128) of the M x N product (rows past M or N are not
// stored).  wmap: the device weight layout; bmap: the fp16 tokens
// (tok_fp16_kernel), Kp = 64 C columns; sx: the token sums.
template <bool ACC, int T>
__global__ void __launch_bounds__(kGmThreads, 1)
gemm_kernel(const __grid_constant__ CUtensorMap wmap,
            const __grid_constant__ CUtensorMap bmap, const GemvArgs g,
            const int *sx, int M, unsigned int *err) {
  using Cfg = GmCfg<T>;
  constexpr int kGmTokens = T;
  constexpr uint32_t kGmSliceBytes = Cfg::kSliceBytes;
  constexpr uint32_t kGmBStageBytes = Cfg::kBStageBytes;
  constexpr int kGmBStages = Cfg::kBStages;
  constexpr int kGmWStages = Cfg::kWStages;
  constexpr uint32_t kGmAccCols = Cfg::kAccCols;
  constexpr int kBarFullW = Cfg::kBarFullW, kBarEmptyW = Cfg::kBarEmptyW;
  constexpr int kBarFullB = Cfg::kBarFullB, kBarEmptyB = Cfg::kBarEmptyB;
  constexpr int kBarFullA = Cfg::kBarFullA, kBarDoneA = Cfg::kBarDoneA;
  constexpr int kBarAcc = Cfg::kBarAcc;
  constexpr uint32_t kSmB = Cfg::kSmB, kSmW = Cfg::kSmW, kSmS = Cfg::kSmS;
  constexpr uint32_t kSmR = Cfg::kSmR, kSmSx = Cfg::kSmSx, kSmWs = Cfg::kSmWs;
  constexpr uint32_t kSmTmem = Cfg::kSmTmem, kSmBars = Cfg::kSmBars;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t *smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int C = g.chunks;
  const int n_st = (C + kGmStageChunks - 1) / kGmStageChunks;
  const int g0 = int(blockIdx.x) * kGmRowGroups;
  const int m0 = int(blockIdx.y) * kGmTokens;
  uint64_t *bar = reinterpret_cast<uint64_t *>(smem + kSmBars);
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + kSmTmem);
  float *s_sm = reinterpret_cast<float *>(smem + kSmS);
  float *r_sm = reinterpret_cast<float *>(smem + kSmR);
  float *nsx_sm = reinterpret_cast<float *>(smem + kSmSx);
  float *ws_sm = reinterpret_cast<float *>(smem + kSmWs);

  if (threadIdx.x == 0) {
    for (int i = 0; i < kGmWStages; ++i) {
      mbar_init(&bar[kBarFullW + i], 1);
      mbar_init(&bar[kBarEmptyW + i], kGmSetWarps);
    }
    for (int i = 0; i < kGmBStages; ++i) {
      mbar_init(&bar[kBarFullB + i], 1);
      mbar_init(&bar[kBarEmptyB + i], 1);
    }
    for (int i = 0; i < kGmAStages; ++i) {
      mbar_init(&bar[kBarFullA + i], kGmSetWarps);
      mbar_init(&bar[kBarDoneA + i], 1);
    }
    mbar_init(&bar[kBarAcc], 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == kGmMmaWarp) tmem_alloc(tmem_slot, kGmTmemCols);
  tc_fence_before();
  __syncthreads();  // barriers set up, tensor memory allocated
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == kGmProducerWarp) {
    // ---- tiled copies: weight stages (static: before the wait), tokens ----
    auto issue_w = [&](int s) {
      const int slot = s % kGmWStages;
      mbar_arrive_expect_tx(&bar[kBarFullW + slot], kGmWStageBytes);
      tma_load_2d(smem + kSmW + slot * kGmWStageBytes, &wmap,
                  s * kGmStageChunks * (kGroupChunkBytes / 8), g0,
                  &bar[kBarFullW + slot]);
    };
    // A stage's token boxes: one per 64-k slice that holds a chunk (the
    // last stage of an odd chunk count has one; no box lies wholly past K).
    auto issue_b = [&](int s) {
      const int slot = s % kGmBStages;
      const int nc = min(kGmStageChunks, C - s * kGmStageChunks);
      mbar_arrive_expect_tx(&bar[kBarFullB + slot], uint32_t(nc) * kGmSliceBytes);
      for (int c = 0; c < nc; ++c)
        tma_load_2d(smem + kSmB + slot * kGmBStageBytes + c * kGmSliceBytes,
                    &bmap, (s * kGmStageChunks + c) * 64, m0,
                    &bar[kBarFullB + slot]);
    };
    int sw = 0, sb = 0;
    if (lane == 0) {
      asm volatile("prefetch.tensormap [%0];" ::"l"(
                       reinterpret_cast<uint64_t>(&wmap))
                   : "memory");
      asm volatile("prefetch.tensormap [%0];" ::"l"(
                       reinterpret_cast<uint64_t>(&bmap))
                   : "memory");
      for (; sw < kGmWStages && sw < n_st; ++sw) issue_w(sw);
    }
    pdl_wait();
    pdl_trigger();
    if (lane == 0) {
      long long idle_since = clock64();
      while (sw < n_st || sb < n_st) {
        bool moved = false;
        if (sb < n_st &&
            (sb < kGmBStages ||
             mbar_try_wait(&bar[kBarEmptyB + sb % kGmBStages],
                           uint32_t(sb / kGmBStages - 1) & 1u))) {
          issue_b(sb++);
          moved = true;
        }
        if (sw < n_st &&
            mbar_try_wait(&bar[kBarEmptyW + sw % kGmWStages],
                          uint32_t(sw / kGmWStages - 1) & 1u)) {
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
      // Copies still in flight land before the CTA exits.
      for (int s = max(0, sw - kGmWStages); s < sw; ++s)
        if (!mbar_wait(&bar[kBarFullW + s % kGmWStages],
                       uint32_t(s / kGmWStages) & 1u))
          atomicOr(err, 2u);
      for (int s = max(0, sb - kGmBStages); s < sb; ++s)
        if (!mbar_wait(&bar[kBarFullB + s % kGmBStages],
                       uint32_t(s / kGmBStages) & 1u))
          atomicOr(err, 2u);
    }
    __syncwarp();
  } else if (warp == kGmMmaWarp) {
    // ---- MMA issue: the warp runs the loop, one elected lane issues ----
    pdl_wait();
    pdl_trigger();
    const uint32_t idesc = tc_idesc(kGmTokens);
    const uint32_t b_ring = smem_addr(smem + kSmB);
    constexpr uint32_t kSlice16 = kGmSliceBytes / 16;  // 16-byte units
    bool ok = true;
    for (int s = 0; s < n_st; ++s) {
      const int ab = s % kGmAStages, bs = s % kGmBStages;
      if (!warp_wait(&bar[kBarFullA + ab], uint32_t(s / kGmAStages) & 1u) ||
          !warp_wait(&bar[kBarFullB + bs], uint32_t(s / kGmBStages) & 1u)) {
        ok = false;
        break;
      }
      tc_fence_after();
      // k-step ks: slice ks / 4 of the stage (256 token rows of 128 bytes),
      // 32 bytes per step within it; A columns 8 ks of the stage.
      const int nks = 4 * min(kGmStageChunks, C - s * kGmStageChunks);
      const uint64_t bd0 = sw128_desc(b_ring + uint32_t(bs) * kGmBStageBytes);
      const uint32_t a0 = tmem + kGmAccCols + uint32_t(ab) * kGmACols;
      if (elect_one()) {
#pragma unroll
        for (int ks = 0; ks < 4 * kGmStageChunks; ++ks) {
          if (ks < nks)
            tc_mma(tmem, a0 + uint32_t(ks) * 8u,
                   bd0 + uint64_t(uint32_t(ks >> 2) * kSlice16 +
                                  uint32_t(ks & 3) * 2u),
                   idesc, (ks > 0 || s > 0) ? 1u : 0u);
        }
        tc_commit(&bar[kBarDoneA + ab]);   // the A stage may be rewritten
        tc_commit(&bar[kBarEmptyB + bs]);  // the token stage may be refilled
      }
      __syncwarp();
    }
    if (!ok && lane == 0) atomicOr(err, 4u);
    if (elect_one()) tc_commit(&bar[kBarAcc]);  // also on a time-out
    __syncwarp();
  } else {
    // ---- decode warps: 2-bit codes -> fp16 A in tensor memory ----
    pdl_trigger();
    const int q = warp & 3, h = warp >> 2;  // lane quarter; stage set
    const int r = 32 * q + lane;            // weight row of the tile
    const uint32_t t_lane = tmem + (uint32_t(32 * q) << 16);
    bool ok = true;
    for (int s = h; s < n_st && ok; s += 2) {
      const int ws = s % kGmWStages, ab = s % kGmAStages;
      if (!warp_wait(&bar[kBarFullW + ws], uint32_t(s / kGmWStages) & 1u)) {
        ok = false;
        break;
      }
      const int nc = min(kGmStageChunks, C - s * kGmStageChunks);
      const uint8_t *src = smem + kSmW + ws * kGmWStageBytes +
                           (r >> 3) * (kGmStageChunks * kGroupChunkBytes) +
                           (r & 7) * kChunkBytes;
      uint4 wq[kGmStageChunks];
#pragma unroll
      for (int c = 0; c < kGmStageChunks; ++c)
        wq[c] = c < nc ? *reinterpret_cast<const uint4 *>(src + c * kGroupChunkBytes)
                       : make_uint4(0u, 0u, 0u, 0u);
      // The slot is refilled by a bulk copy once released: the loads above
      // are ordered before that write by the fence of every lane.
      fence_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar[kBarEmptyW + ws]);
      if (s >= kGmAStages &&
          !warp_wait(&bar[kBarDoneA + ab], uint32_t(s / kGmAStages - 1) & 1u)) {
        ok = false;
        break;
      }
      tc_fence_after();
#pragma unroll
      for (int c = 0; c < kGmStageChunks; ++c) {
        if (c < nc) {
          uint32_t col[32];
          decode_word(wq[c].x, col);
          decode_word(wq[c].y, col + 8);
          decode_word(wq[c].z, col + 16);
          decode_word(wq[c].w, col + 24);
          tmem_st32(t_lane + kGmAccCols + uint32_t(ab) * kGmACols +
                        uint32_t(c) * 32u,
                    col);
        }
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar[kBarFullA + ab]);
    }
    if (!ok && lane == 0) atomicOr(err, 4u);

    // ---- epilogue: warp (q, h) takes accumulator columns [T/2 h,
    // T/2 (h + 1)) (tokens) of weight rows 32 q .. 32 q + 31 ----
    pdl_wait();
    {
      // Per token: -sum_k x (as fp32, exact: |sum| < 2^22; +0 for a zero
      // sum), s and r = 1 / s (0 where s is outside [2^-60, 2^60]).
      const int t = threadIdx.x;  // 0..255
      nsx_sm[t] = 0.0f;  // tokens past M: computed in pairs, never stored
      s_sm[t] = 1.0f;
      r_sm[t] = 1.0f;
      if (m0 + t < M) {
        nsx_sm[t] = static_cast<float>(-sx[m0 + t]);
        if (!ACC) {
          const float sv = g.s[m0 + t];
          s_sm[t] = sv;
          r_sm[t] = (sv >= 0x1p-60f && sv <= 0x1p60f) ? 1.0f / sv : 0.0f;
        }
      }
      if (t < BW_MAX_WS)
        ws_sm[t] = t < g.seg.n_ws ? __bfloat162float(g.ws[t]) : 0.0f;
    }
    decode_warps_sync();
    const bool acc_ready = warp_wait(&bar[kBarAcc], 0u);
    tc_fence_after();
    if (!acc_ready) {
      if (lane == 0) atomicOr(err, 4u);
    } else {
      const int n = g0 * kGroupRows + r;
      int sg = 0;
#pragma unroll
      for (int i = 1; i < BW_MAX_WS; ++i)
        if (i < g.seg.n_ws && n >= g.seg.bounds[i]) sg = i;
      const float wsv = ws_sm[sg];
      for (int j0 = (T / 2) * h; j0 < (T / 2) * (h + 1); j0 += 32) {
        if (m0 + j0 >= M) break;  // warp-uniform
        uint32_t d[32];
        tmem_ld32(t_lane + uint32_t(j0), d);  // whole warp
        if (n < g.N) {  // the collective load above is the whole warp's
          // acc = 2^24 D - sum_k x, exact in fp32 (an integer below 2^24),
          // in two halves of 16 tokens: their per-token values are loaded
          // first, then the outputs go out in pairs of tokens (one
          // conversion to bf16 per pair).
#pragma unroll
          for (int hb = 0; hb < 32; hb += 16) {
            float nsx[16], sv[16], rv[16];
#pragma unroll
            for (int i = 0; i < 16; i += 4) {
              const float4 a = lds4(nsx_sm + j0 + hb + i);
              nsx[i] = a.x; nsx[i + 1] = a.y; nsx[i + 2] = a.z; nsx[i + 3] = a.w;
              if (!ACC) {
                const float4 b = lds4(s_sm + j0 + hb + i);
                const float4 c = lds4(r_sm + j0 + hb + i);
                sv[i] = b.x; sv[i + 1] = b.y; sv[i + 2] = b.z; sv[i + 3] = b.w;
                rv[i] = c.x; rv[i + 1] = c.y; rv[i + 2] = c.z; rv[i + 3] = c.w;
              }
            }
            // Every token of the half on the corrected-product path, or
            // (never for quantised activations of ordinary range) all of
            // them divided: one branch per half, the same in every lane.
            bool fast = true;
#pragma unroll
            for (int i = 0; i < 16; ++i) fast = fast && rv[i] != 0.0f;
            // All 16 results first, as independent straight-line chains
            // (tokens past M have s = r = 1 and no token sum, and are never
            // stored), then the stores, in pairs of tokens.
            float yv[16];
            if (ACC) {
#pragma unroll
              for (int e = 0; e < 16; ++e)
                yv[e] = fmaf(__uint_as_float(d[hb + e]), 16777216.0f, nsx[e]);
            } else if (fast) {
#pragma unroll
              for (int e = 0; e < 16; ++e)
                yv[e] = div_by_recip(fmaf(__uint_as_float(d[hb + e]),
                                          16777216.0f, nsx[e]),
                                     sv[e], rv[e]) *
                        wsv;
            } else {
#pragma unroll
              for (int e = 0; e < 16; ++e) {
                const float a =
                    fmaf(__uint_as_float(d[hb + e]), 16777216.0f, nsx[e]);
                yv[e] = (rv[e] != 0.0f ? div_by_recip(a, sv[e], rv[e])
                                       : a / sv[e]) *
                        wsv;
              }
            }
            const int mh = m0 + j0 + hb;  // the half's first token
            const size_t ld = size_t(g.out_ld);
            if (mh + 16 <= M) {  // warp-uniform: the whole half is stored
              if (ACC) {
                int *o = static_cast<int *>(g.out) + size_t(mh) * ld + n;
#pragma unroll
                for (int e = 0; e < 16; ++e) o[e * ld] = __float2int_rn(yv[e]);
              } else {
                __nv_bfloat16 *o =
                    static_cast<__nv_bfloat16 *>(g.out) + size_t(mh) * ld + n;
#pragma unroll
                for (int e = 0; e < 16; e += 2) {
                  const __nv_bfloat162 y2 =
                      __floats2bfloat162_rn(yv[e], yv[e + 1]);
                  o[e * ld] = y2.x;
                  o[(e + 1) * ld] = y2.y;
                }
              }
            } else {
#pragma unroll
              for (int e = 0; e < 16; e += 2) {
                const int m = mh + e;
                if (m >= M) break;
                if (ACC) {
                  int *o = static_cast<int *>(g.out) + size_t(m) * ld + n;
                  o[0] = __float2int_rn(yv[e]);
                  if (m + 1 < M) o[ld] = __float2int_rn(yv[e + 1]);
                } else {
                  const __nv_bfloat162 y2 =
                      __floats2bfloat162_rn(yv[e], yv[e + 1]);
                  __nv_bfloat16 *o = static_cast<__nv_bfloat16 *>(g.out) +
                                     size_t(m) * ld + n;
                  o[0] = y2.x;
                  if (m + 1 < M) o[ld] = y2.y;
                }
              }
            }
          }
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();  // every tensor-memory access is done
  if (warp == kGmMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kGmTmemCols);
  }
}

size_t align256(size_t b) { return (b + 255) / 256 * 256; }

template <bool ACC, int T>
cudaError_t launch_gemm_t(const GemvArgs &g, int M, void *workspace,
                          cudaStream_t stream) {
  static std::atomic<bool> configured[64];
  using Cfg = GmCfg<T>;
  unsigned int *err = device_error_word();
  if (!err) return cudaErrorInvalidSymbol;
  const int Kp = g.chunks * 64;
  __half *xb = static_cast<__half *>(workspace);
  int *sx = reinterpret_cast<int *>(static_cast<uint8_t *>(workspace) +
                                    align256(size_t(M) * Kp * 2));
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;

  cudaLaunchConfig_t pre = {};
  pre.gridDim = dim3(unsigned(M));
  pre.blockDim = dim3(256);
  pre.stream = stream;
  pre.attrs = attr;
  pre.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&pre, tok_fp16_kernel, g.x, g.x_ld, g.K,
                                     Kp, xb, sx);
  if (e != cudaSuccess) return e;

  auto kernel = gemm_kernel<ACC, T>;
  int64_t resident = 0;
  e = resident_ctas(kernel, configured, kGmThreads, Cfg::kSmem, &resident);
  if (e != cudaSuccess) return e;
  // Weights: per row group, C chunks of 128 bytes as 16 C uint64; a box is
  // one stage of 16 groups.  Tokens: M rows of Kp fp16; a box is 64 k (128
  // bytes, swizzled) of T rows (rows past M read as zero).
  CUtensorMap wmap, bmap;
  if (!encode_2d(&wmap, CU_TENSOR_MAP_DATA_TYPE_UINT64, g.w,
                 uint64_t(g.chunks) * (kGroupChunkBytes / 8),
                 uint64_t(g.n_groups), uint64_t(g.chunks) * kGroupChunkBytes,
                 kGmStageChunks * (kGroupChunkBytes / 8), kGmRowGroups) ||
      !encode_2d(&bmap, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, xb, uint64_t(Kp),
                 uint64_t(M), uint64_t(Kp) * 2, 64, T,
                 CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned((g.n_groups + kGmRowGroups - 1) / kGmRowGroups),
                     unsigned((M + T - 1) / T));
  cfg.blockDim = dim3(kGmThreads);
  cfg.dynamicSmemBytes = Cfg::kSmem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, wmap, bmap, g, sx, M, err);
}

}  // namespace

size_t gemm_workspace_bytes(int M, int K) {
  return align256(size_t(M) * size_t(chunks_per_row(K)) * 64 * 2) +
         align256(size_t(M) * sizeof(int));
}

// Token tiles of 64 up to 64 tokens, of 128 up to 128, else of 256.
cudaError_t launch_gemm(const GemvArgs &a, int M, bool acc_out,
                        void *workspace, cudaStream_t stream) {
  if (M <= 64)
    return acc_out ? launch_gemm_t<true, 64>(a, M, workspace, stream)
                   : launch_gemm_t<false, 64>(a, M, workspace, stream);
  if (M <= 128)
    return acc_out ? launch_gemm_t<true, 128>(a, M, workspace, stream)
                   : launch_gemm_t<false, 128>(a, M, workspace, stream);
  return acc_out ? launch_gemm_t<true, 256>(a, M, workspace, stream)
                 : launch_gemm_t<false, 256>(a, M, workspace, stream);
}

}  // namespace bw
