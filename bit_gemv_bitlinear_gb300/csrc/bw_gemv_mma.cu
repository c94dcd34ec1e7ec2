// bw_gemv_mma.cu -- the W2A8 product for batched activations (M >= 8) on
// tensor cores (mma.sync), streamed like the M = 1 pipe kernel.  Used where
// the activation rows are not 16-byte aligned or K % 16 != 0, which the
// tcgen05 kernel's tiled copies need (bw_gemv_tc.cu).
//
// Same result as the CUDA-core GEMV: acc[m][n] = sum_k w[n][k] x[m][k]
// exactly, then y = bf16((acc / s[m]) * ws[seg(n)]).  Source: "BitNet GPU
// 推理框架：从零构建 W2A8 的 2-bit 大模型 CUDA GEMV 内核", §5.3 (product and scale
// epilogue), §4.2 (weight-scale segments); the batching of several known
// tokens so that the weights are read once for all of them is the point of
// the bytes-per-token report's "batched known tokens" item.
//
// Exactness: ternary weights and int8 activations are exact in fp16, every
// product is exact, and every fp32 partial sum is an integer of magnitude
// at most 128 K < 2^21 (K <= 16384), so fp16 MMA with fp32 accumulation
// gives the exact integer in any order; the partial sums of a row group are
// converted to int32 and added with shared-memory atomics.
//
// Design (the streaming is that of bw_pipe.cuh):
//  * mma.sync m16n8k16 (fp16 in, fp32 accumulate) with A = 16 tokens x 16 k
//    and B = 16 k x 8 weight rows, i.e. one row group of the device layout:
//    the pieces a warp streams are the pieces of the M = 1 kernel.
//  * A CTA owns k consecutive row groups; its 8 warps split the CTA's chunks
//    into equal runs, each streamed in pieces through the warp's own ring
//    of bulk copies (the first pieces requested before the dependency wait).
//  * Activations: a tile of MT = 16 (or 8) tokens is converted once per CTA
//    to fp16 (x + 128 as the low byte of fp16(1024 + u), minus 1152) into a
//    shared tile whose rows are 16 bytes longer than 64 k per chunk, so the
//    ldmatrix.x4 that builds each A fragment is conflict-free.
//  * B fragment straight from the packed word in shared memory: thread
//    (g, t) needs codes (row g, k = 2t, 2t+1, 2t+8, 2t+9) of a 16-k word;
//    with the word interleave of the layout these sit in byte pair 2(t&1)
//    at slots t/2 and t/2 + 2, so one shift and, per two weights, one
//    mask-or and one byte permute that reads the fp16 high bytes of -1, 0,
//    +1 from a constant give two weights per 32-bit register (the weights
//    are signed here: no sum_k x correction).
#include <cuda_fp16.h>

#include "bw_pipe.cuh"

namespace bw {
namespace {

using namespace pipe;

constexpr int kMmaWarps = 16;        // warps per CTA (one CTA per SM)
constexpr int kMmaSlots = 2;         // ring slots per warp
constexpr int kMmaPieceChunks = 32;  // 4 KB pieces (2 KB where that fits)

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t s) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(s));
  return d;
}

__device__ __forceinline__ uint32_t hsub2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// fp16 of a ternary weight has a zero low byte and the high byte 0xBC
// (-1), 0x00 (0) or 0x3C (+1): byte c of this table for code c = w + 1,
// byte 3 is the zero low byte.
constexpr uint32_t kTernaryF16Hi = 0x003C00BCu;

// Two codes at bits 4-5 and 12-13 of sel (other bits ignored) -> fp16x2 of
// (code - 1): a byte permute whose selector nibbles are 3, c0, 3, c1.
__device__ __forceinline__ uint32_t decode_pair_hi(uint32_t sel) {
  return prmt(kTernaryF16Hi, 0u, (sel & 0x3030u) | 0x0303u);
}

// Four int8 (one 32-bit word) -> two fp16x2 (exact).
__device__ __forceinline__ uint2 int8x4_to_f16(uint32_t v) {
  const uint32_t u = v ^ 0x80808080u;  // x + 128 as unsigned bytes
  const uint32_t lo = prmt(u, 0x64646464u, 0x4140u);
  const uint32_t hi = prmt(u, 0x64646464u, 0x4342u);
  return make_uint2(hsub2(lo, 0x64806480u), hsub2(hi, 0x64806480u));  // -1152
}

__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4],
                                         uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
      "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void ldmatrix_x4(uint32_t (&r)[4], uint32_t addr) {
  asm volatile(
      "ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
      : "r"(addr));
}

// Row stride of the fp16 activation tile in bytes: 64 k per chunk plus 16,
// so that the 8 rows of an ldmatrix matrix fall in 8 distinct bank groups.
__host__ __device__ inline uint32_t mma_xrow_bytes(int chunks) {
  return uint32_t(chunks) * 128u + 16u;
}

// Shared-memory carve-up: ring [warps][slots][piece], x tile [MT][xrow]
// (rows past MT are never read: A rows 8..15 of an 8-token tile come from
// the zero block), zero block (16 bytes), s [16], ws [BW_MAX_WS], row
// totals [k][16][8] int32, barriers [warps][slots].
struct MmaLayout {
  uint32_t ring, xs, zero, s, ws, tot, bars, total;
};

__host__ __device__ inline MmaLayout mma_layout(int mt, int chunks, int k,
                                                int piece_chunks) {
  MmaLayout l;
  l.ring = 0;
  l.xs = uint32_t(kMmaWarps * kMmaSlots * piece_chunks) * kGroupChunkBytes;
  l.zero = l.xs + uint32_t(mt) * mma_xrow_bytes(chunks);
  l.s = l.zero + 16;
  l.ws = l.s + 16 * 4;
  l.tot = l.ws + BW_MAX_WS * 4;
  l.bars = l.tot + uint32_t(k) * 16 * 8 * 4;
  l.total = l.bars + uint32_t(kMmaWarps * kMmaSlots * 8);
  return l;
}

// One launch: tokens [0, rows) (rows <= MT) of the activations at g.x, all
// N outputs.  The split fields of `a` are set by the host (launch_tile).
template <int MT, bool ACC>
__global__ void __launch_bounds__(kMmaWarps * 32)
pipe_mma_kernel(const PipeArgs a, const GemvArgs g, int rows) {
  static_assert(MT == 8 || MT == 16, "token tile of 8 or 16");
  extern __shared__ __align__(128) uint8_t smem[];
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int KS = a.slot_chunks;
  const int R = a.slots;
  const int C = a.chunks;
  const int k = a.groups_per_cta;
  const uint32_t slot_bytes = uint32_t(KS) * kGroupChunkBytes;
  const uint32_t xrow = mma_xrow_bytes(C);
  const MmaLayout L = mma_layout(MT, C, k, KS);
  uint8_t *ring = smem + L.ring + size_t(warp) * R * slot_bytes;
  uint8_t *xs = smem + L.xs;
  float *s_sm = reinterpret_cast<float *>(smem + L.s);
  float *ws_sm = reinterpret_cast<float *>(smem + L.ws);
  int *tot = reinterpret_cast<int *>(smem + L.tot);  // [k][16][8]
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + L.bars) + warp * R;

  const int g_lo = int(blockIdx.x) * k;
  const int n_g = max(0, min(k, a.n_groups - g_lo));
  const int U = n_g * C;
  const int run_lo = U * warp / kMmaWarps;
  const int run_hi = U * (warp + 1) / kMmaWarps;

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
    bulk_copy_g2s(ring + size_t(slot) * slot_bytes,
                  a.w + (size_t(g_lo + iss.g) * C + iss.c) * kGroupChunkBytes,
                  bytes, &full[slot]);
    iss.advance(len, C);
    ++issued;
  };
  if (lane == 0) {
    for (int s = 0; s < R; ++s) mbar_init(&full[s], 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    // The weights are static once written: requested before the wait.
    for (int s = 0; s < R && iss.u < run_hi; ++s) issue_next(s);
  }
  for (int t = threadIdx.x; t < n_g * 16 * 8; t += blockDim.x) tot[t] = 0;
  if (threadIdx.x < 4)
    reinterpret_cast<uint32_t *>(smem + L.zero)[threadIdx.x] = 0u;
  pdl_wait();
  pdl_trigger();  // as in the pipe kernel: one launch of lookahead

  // Scales, then the token tile as fp16 (zero past K and past `rows`); all
  // loads of a batch are issued before its stores (issue is in order).
  const float sv = (!ACC && int(threadIdx.x) < rows) ? g.s[threadIdx.x] : 0.0f;
  const float wv = (!ACC && int(threadIdx.x) < g.seg.n_ws)
                       ? __bfloat162float(g.ws[threadIdx.x])
                       : 0.0f;
  if (g.vec_x) {
    // 16-byte rows: one 16-byte vector of each of the MT rows per thread
    // and step, all MT loads in flight before the first store.
    const int vecs = C * 4;  // 16-byte vectors per row
    for (int w = threadIdx.x; w < vecs; w += blockDim.x) {
      uint4 v[MT];
#pragma unroll
      for (int m = 0; m < MT; ++m)
        v[m] = (m < rows && 16 * w < g.K)
                   ? __ldg(reinterpret_cast<const uint4 *>(
                               g.x + size_t(m) * g.x_ld) + w)
                   : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
      for (int m = 0; m < MT; ++m) {
        // zero activations stay zero: fp16(1024 + 128) - 1152 = 0
        const uint2 h0 = int8x4_to_f16(v[m].x), h1 = int8x4_to_f16(v[m].y);
        const uint2 h2 = int8x4_to_f16(v[m].z), h3 = int8x4_to_f16(v[m].w);
        uint4 *dst = reinterpret_cast<uint4 *>(xs + m * xrow + w * 32);
        dst[0] = make_uint4(h0.x, h0.y, h1.x, h1.y);
        dst[1] = make_uint4(h2.x, h2.y, h3.x, h3.y);
      }
    }
  } else {
    constexpr int kBatch = 8;
    const int words = C * 16;  // 4 int8 per word
    const int total = MT * words;
    for (int i0 = threadIdx.x; i0 < total; i0 += kBatch * blockDim.x) {
      uint32_t v[kBatch];
#pragma unroll
      for (int b = 0; b < kBatch; ++b) {
        const int i = i0 + b * blockDim.x;
        const int m = i / words, w = i - m * words;
        v[b] = (i < total && m < rows && 4 * w < g.K)
                   ? __ldg(reinterpret_cast<const unsigned int *>(
                               g.x + size_t(m) * g.x_ld) + w)
                   : 0x00000000u;
      }
#pragma unroll
      for (int b = 0; b < kBatch; ++b) {
        const int i = i0 + b * blockDim.x;
        if (i < total) {
          const int m = i / words, w = i - m * words;
          *reinterpret_cast<uint2 *>(xs + m * xrow + w * 8) =
              int8x4_to_f16(v[b]);
        }
      }
    }
  }
  if (!ACC && int(threadIdx.x) < rows) s_sm[threadIdx.x] = sv;
  if (threadIdx.x < BW_MAX_WS) ws_sm[threadIdx.x] = wv;
  __syncthreads();  // tile staged, totals zeroed, barriers set up

  const int gq = lane >> 2, tq = lane & 3;  // fragment row / column pair
  const int shift = 16 * (tq & 1) + 2 * (tq >> 1);
  // ldmatrix.x4 row address of this lane: matrix lane/8 is (tokens 0-7 |
  // 8-15) x (k 0-7 | 8-15); tokens past MT read the zero block (no advance).
  const int a_tok = ((lane >> 3) & 1) * 8 + (lane & 7);
  const bool a_live = a_tok < MT;
  const uint32_t a_base =
      a_live ? smem_addr(xs + a_tok * xrow + ((lane >> 4) * 8) * 2)
             : smem_addr(smem + L.zero);
  const uint32_t a_step = a_live ? 2u : 0u;  // bytes per k
  // One accumulator set per 16-k step of a chunk: four independent MMA
  // chains instead of one (each MMA waits for the previous one on the same
  // accumulators).  Each set holds an exact integer below 2^21.
  float d[4][4];
#pragma unroll
  for (int w4 = 0; w4 < 4; ++w4)
#pragma unroll
    for (int e = 0; e < 4; ++e) d[w4][e] = 0.0f;
  bool ok = true;
  int consumed = 0, slot = 0;
  uint32_t phase = 0;
  while (cur.u < run_hi) {
    if (!__all_sync(0xffffffffu, mbar_wait(&full[slot], phase))) {
      ok = false;
      break;
    }
    const int len = cur.piece(KS, C, run_hi);
    const uint8_t *wp = ring + size_t(slot) * slot_bytes + gq * kChunkBytes;
    uint32_t aa = a_base + a_step * uint32_t(cur.c * kChunkWeights);
#pragma unroll 2
    for (int j = 0; j < len; ++j) {
      const uint4 wv = *reinterpret_cast<const uint4 *>(wp + j * kGroupChunkBytes);
      const uint32_t wd[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
      for (int w4 = 0; w4 < 4; ++w4) {
        const uint32_t h = wd[w4] >> shift;
        const uint32_t b0 = decode_pair_hi(h << 4);  // k 2t, 2t+1
        const uint32_t b1 = decode_pair_hi(h);       // k 2t+8, 2t+9
        uint32_t af[4];
        ldmatrix_x4(af, aa + a_step * uint32_t(16 * w4));
        mma16816(d[w4], af, b0, b1);
      }
      aa += a_step * uint32_t(kChunkWeights);
    }
    __syncwarp();
    if (lane == 0 && iss.u < run_hi) {  // piece consumed + R: this slot
      fence_proxy_async_smem();
      issue_next(slot);
    }
    const int gl = cur.g;
    cur.advance(len, C);
    ++consumed;
    if (cur.c == 0 || cur.u == run_hi) {  // row group or run finished
      // D: [0..1] = token gq, rows 2tq, 2tq+1; [2..3] = token gq + 8.
      int v[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        v[e] = __float2int_rn(d[0][e]) + __float2int_rn(d[1][e]) +
               __float2int_rn(d[2][e]) + __float2int_rn(d[3][e]);
#pragma unroll
        for (int w4 = 0; w4 < 4; ++w4) d[w4][e] = 0.0f;
      }
      int *tg = tot + gl * 16 * 8;
      if (gq < MT) {
        atomicAdd(&tg[gq * 8 + 2 * tq], v[0]);
        atomicAdd(&tg[gq * 8 + 2 * tq + 1], v[1]);
      }
      if (gq + 8 < MT) {
        atomicAdd(&tg[(gq + 8) * 8 + 2 * tq], v[2]);
        atomicAdd(&tg[(gq + 8) * 8 + 2 * tq + 1], v[3]);
      }
    }
    if (++slot == R) {
      slot = 0;
      phase ^= 1u;
    }
  }
  if (!ok && lane == 0) {
    atomicOr(a.err, 4u);
    for (int i = consumed; i < issued; ++i)
      if (!mbar_wait(&full[i % R], uint32_t(i / R) & 1u)) atomicOr(a.err, 2u);
  }
  __syncthreads();  // every partial sum is in `tot`

  // Outputs: 8 consecutive rows of one token per 8 threads.
  for (int t = threadIdx.x; t < n_g * MT * 8; t += blockDim.x) {
    const int rr = t & 7, m = (t >> 3) % MT, gl = (t >> 3) / MT;
    const int n = (g_lo + gl) * kGroupRows + rr;
    if (m >= rows || n >= g.N) continue;
    const int total = tot[(gl * 16 + m) * 8 + rr];
    if (ACC) {
      static_cast<int *>(g.out)[size_t(m) * g.out_ld + n] = total;
    } else {
      int sg = 0;
#pragma unroll
      for (int i = 1; i < BW_MAX_WS; ++i)
        if (i < g.seg.n_ws && n >= g.seg.bounds[i]) sg = i;
      const float scaled = static_cast<float>(total) / s_sm[m];
      static_cast<__nv_bfloat16 *>(g.out)[size_t(m) * g.out_ld + n] =
          __float2bfloat16_rn(scaled * ws_sm[sg]);
    }
  }
}

constexpr int kMmaMaxGroupsPerCta = 32;  // row totals: 16 KB at most
constexpr uint32_t kSmemLimit = 227u * 1024u;

// Token tile and piece size for K: 16 tokens if the fp16 tile fits beside
// a ring of 4 KB (else 2 KB) pieces, else 8 tokens likewise; false if
// neither fits.
bool mma_config(int K, int *mt, int *piece) {
  if (K > kMmaMaxK) return false;
  const int chunks = chunks_per_row(K);
  for (int t : {16, 8})
    for (int p : {kMmaPieceChunks, kMmaPieceChunks / 2})
      if (mma_layout(t, chunks, kMmaMaxGroupsPerCta, p).total <= kSmemLimit) {
        *mt = t;
        *piece = p;
        return true;
      }
  return false;
}

template <int MT, bool ACC>
cudaError_t launch_tile(const GemvArgs &g, int rows, int piece,
                        cudaStream_t stream) {
  static std::atomic<bool> configured[64];
  auto kernel = pipe_mma_kernel<MT, ACC>;
  PipeArgs a{};
  a.w = g.w;
  a.N = g.N;
  a.chunks = g.chunks;
  a.n_groups = g.n_groups;
  a.slots = kMmaSlots;
  a.slot_chunks = piece;
  a.err = device_error_word();
  if (!a.err) return cudaErrorInvalidSymbol;
  // k groups per CTA from the residency, as for the M = 1 kernel.
  int64_t k = 1, resident = 0;
  for (int pass = 0; pass < 2; ++pass) {
    cudaError_t e = resident_ctas(
        kernel, configured, kMmaWarps * 32,
        mma_layout(MT, a.chunks, int(k), a.slot_chunks).total, &resident);
    if (e != cudaSuccess) return e;
    k = (a.n_groups + resident - 1) / resident;
    if (k > kMmaMaxGroupsPerCta) k = kMmaMaxGroupsPerCta;
    if (k < 1) k = 1;
  }
  const int64_t grid = (a.n_groups + k - 1) / k;
  const int64_t run = (k * a.chunks + kMmaWarps - 1) / kMmaWarps;
  if (run < a.slot_chunks) a.slot_chunks = int(run < 1 ? 1 : run);
  a.groups_per_cta = int(k);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(grid > 0 ? grid : 1));
  cfg.blockDim = dim3(kMmaWarps * 32);
  cfg.dynamicSmemBytes =
      mma_layout(MT, a.chunks, int(k), a.slot_chunks).total;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, a, g, rows);
}

}  // namespace

int mma_tile_rows(int K) {
  int mt = 0, piece = 0;
  return mma_config(K, &mt, &piece) ? mt : 0;
}

cudaError_t launch_gemv_mma(const GemvArgs &a, int rows, bool acc_out,
                            cudaStream_t stream) {
  int mt = 0, piece = 0;
  if (!mma_config(a.K, &mt, &piece) || rows < 1 || rows > mt)
    return cudaErrorInvalidValue;
  if (mt == 16)
    return acc_out ? launch_tile<16, true>(a, rows, piece, stream)
                   : launch_tile<16, false>(a, rows, piece, stream);
  return acc_out ? launch_tile<8, true>(a, rows, piece, stream)
                 : launch_tile<8, false>(a, rows, piece, stream);
}

}  // namespace bw
