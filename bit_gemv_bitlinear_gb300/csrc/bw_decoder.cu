// bw_decoder.cu -- the decoder layer stack as ONE persistent kernel per
// bw_layer_stack call (stacks without a KV cache).
//
// Source: "BitNet GPU 推理框架：从零构建 W2A8 的 2-bit 大模型 CUDA GEMV 内核":
// §一 (BitNet-2B shape), §4.1 (the fused q|k|v and gate|up projections and
// the four RMSNorms), §六 item 3 (per-token absmax int8 quantisation before
// every W2A8 GEMV), §5.3 (dp4a dot product, scale epilogue), §7.1 (the
// decode GEMVs are memory-bound) and §六 item 1 (decode replayed from a CUDA
// graph to cut launch cost, which this kernel takes further: one launch for
// every step of the call).
//
// What a step computes is the layer of bw_stack.cu (bw.h states it).  What
// differs is how the GEMVs are chained.  With one launch per GEMV, every
// GEMV waits for the previous launch to drain, and its weights start to
// stream only when its CTAs are resident.  Here every SM runs one CTA of 16
// warps for the whole call, and the work is a list of phases: (step, layer,
// GEMV), four GEMVs per layer.
//
//  * Weights never wait for activations.  The packed weights do not depend
//    on the step's values, so each warp streams its share of EVERY phase, in
//    phase order, through its own ring of 3 slots of up to 4 KB (1-D bulk
//    copies completing on mbarriers, as in bw_pipe.cuh): as soon as a slot
//    is consumed, the next piece -- of this GEMV or of the next ones -- is
//    requested.  While a CTA waits for a phase's input, the weights of the
//    next phases are already landing.
//  * Phases hand over data through exchange buffers of 8-byte entries: the
//    fp32 value in the low half and the phase's epoch in the high half,
//    written by ONE 64-bit store, so a reader sees either an old entry or
//    the whole new one.  A consumer polls the entries it needs until every
//    epoch matches; there is no separate grid barrier, and the data arrive
//    with the poll that sees them.  Every CTA reads the whole input vector,
//    so it computes the RMSNorm statistics itself (sum of squares and the
//    largest |v * gain|, fixed-order reductions: every CTA gets the same
//    scale and codes) and quantises into shared memory.
//  * An exchange buffer is rewritten only four phases after it was written,
//    and a CTA can only reach that phase after every CTA has consumed it, so
//    one buffer per GEMV output is enough.  Epochs grow by one per phase
//    across calls (a device counter, advanced by the last CTA to leave), so
//    stale entries never match, also when the launch is replayed.
//  * Every wait is bounded (about a second of clock64).  A CTA that gives
//    up sets a bit in the device error word and an abort word that every
//    poller checks, so the whole grid leaves within one poll; every lane
//    that issued copies waits (bounded) for them before its CTA leaves.
//  * The launch is cooperative, so all CTAs are resident together, which
//    the polls require.
#include <new>

#include "bw_pipe.cuh"

namespace bw {
namespace dec {

using namespace pipe;

constexpr int kWarps = 16;
constexpr int kThreads = kWarps * 32;
constexpr int kSlots = 3;
constexpr int kSlotChunks = 32;  // pieces of up to 4 KB
constexpr uint32_t kSlotBytes = uint32_t(kSlotChunks) * kGroupChunkBytes;
constexpr int kKinds = 4;        // wqkv, wo, w13, w2
// Every exchange entry is written kReplicas times, each copy in its own
// region, and CTA b reads copy b mod kReplicas: every CTA reads the whole
// input vector of a phase, and with one copy the same lines would take a
// request from every CTA on every poll round.
constexpr int kReplicas = 8;

// Geometry of one GEMV of the layer (the same in every layer).
struct KindGeo {
  int N, K;        // output rows, reduction length
  int chunks;      // ceil(K / 64)
  int n_groups;    // ceil(N / 8)
  int pair_half;   // w13: ffn / 8 (gate and up groups paired), else 0
};

// Per-layer device pointers, in a device table.
struct LayerPtrs {
  const uint8_t *w[kKinds];
  const __nv_bfloat16 *ws;  // 7 scales: q, k, v, o, gate, up, down
  const float *gam;         // attention_norm | attn_sub_norm | ffn_norm | ffn_sub_norm
};

struct DecArgs {
  const LayerPtrs *layers;
  int n_layers, steps, phases;
  int dim, ffn, n_heads, n_kv, hd, group, v_off;
  float eps;
  KindGeo geo[kKinds];
  const float *h_in;          // [steps][dim]
  float *h_out;               // [steps][dim]
  // exchange buffers, the output of each GEMV kind: the attention output
  // [dim] (wqkv), h after the wo residual [dim], the gated product [ffn]
  // (w13), h after the w2 residual [dim]
  unsigned long long *xch[kKinds];   // copy 0; copy r at + r * xstride
  size_t xstride;                    // entries between copies
  unsigned int *ctl;          // [0] epoch of the next call's first phase,
                              // [1] CTAs that left, [2] abort
  unsigned int *err;          // device error word
  bw_stack_trace tr;          // tr.layer < 0: no trace
  int max_chunks;             // of the two reduction lengths
  int tot_ints;               // row-total capacity per CTA
};

// The per-layer pointer table is copied to shared memory at entry, so no
// phase waits on a global load for an address (at most kMaxLayers layers).
constexpr int kMaxLayers = 128;
// A warp's run of one GEMV kind, cut into pieces (at most kMaxPieces).
constexpr int kMaxPieces = 8;

struct DecLayout {
  uint32_t ring, xs, tot, red, misc, table, pieces, bars, total;
};

__host__ __device__ inline DecLayout dec_layout(int max_chunks, int tot_ints,
                                                int n_layers) {
  DecLayout l;
  l.ring = 0;
  l.xs = uint32_t(kWarps * kSlots) * kSlotBytes;
  l.tot = l.xs + uint32_t(max_chunks) * 64u;
  l.red = l.tot + (uint32_t(tot_ints) * 4u + 15u) / 16u * 16u;
  l.misc = l.red + 64u * 4u;
  l.table = l.misc + 32u * 4u;
  l.pieces = l.table + uint32_t(n_layers) * uint32_t(sizeof(LayerPtrs));
  // piece lists [kWarps][kKinds][kMaxPieces], their counts [kWarps][kKinds],
  // the CTA's first group and group count per kind
  l.bars = l.pieces + uint32_t(kWarps * kKinds * (kMaxPieces + 1) +
                               2 * kKinds) * 4u;
  l.bars = (l.bars + 7u) / 8u * 8u;
  l.total = l.bars + uint32_t(kWarps * kSlots) * 8u;
  return l;
}

// Row groups of kind g owned by CTA b of G (in streaming order; with pairs,
// whole (gate, up) pairs).
__host__ __device__ inline void cta_groups(const KindGeo &g, int b, int G,
                                           int &g_lo, int &n_g) {
  if (g.pair_half) {
    const int lo = int(int64_t(g.pair_half) * b / G);
    const int hi = int(int64_t(g.pair_half) * (b + 1) / G);
    g_lo = 2 * lo;
    n_g = 2 * (hi - lo);
  } else {
    const int lo = int(int64_t(g.n_groups) * b / G);
    const int hi = int(int64_t(g.n_groups) * (b + 1) / G);
    g_lo = lo;
    n_g = hi - lo;
  }
}

__device__ __forceinline__ int phys(int g, int pair_half) {
  return pair_half ? (g >> 1) + (g & 1) * pair_half : g;
}

__device__ __forceinline__ unsigned long long entry(float v, unsigned ep) {
  return (static_cast<unsigned long long>(ep) << 32) | __float_as_uint(v);
}

__device__ __forceinline__ void st_entry(unsigned long long *p,
                                         unsigned long long v) {
  asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v)
               : "memory");
}

// Writes one exchange entry to every copy.
__device__ __forceinline__ void publish(unsigned long long *p, size_t stride,
                                        unsigned long long v) {
#pragma unroll
  for (int r = 0; r < kReplicas; ++r) st_entry(p + r * stride, v);
}

__device__ __forceinline__ void ld_entries(const unsigned long long *p,
                                           unsigned long long &a,
                                           unsigned long long &b) {
  asm volatile("ld.relaxed.gpu.global.v2.u64 {%0, %1}, [%2];"
               : "=l"(a), "=l"(b)
               : "l"(p)
               : "memory");
}

__device__ __forceinline__ unsigned ld_flag(const unsigned int *p) {
  unsigned v;
  asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p)
               : "memory");
  return v;
}

__device__ __forceinline__ float bf16r(__nv_bfloat16 v) {
  return __bfloat162float(v);
}

// bf16((acc / s) * ws), IEEE fp32, one rounding.
__device__ __forceinline__ __nv_bfloat16 scaled(int total, float s, float ws) {
  return __float2bfloat16_rn((static_cast<float>(total) / s) * ws);
}

// rint(x * scale) in the low byte (see bw_stack.cu: |x * scale| <= 127 by
// construction of the scale, so the fp32 add of 1.5 * 2^23 rounds to the
// integer, ties to even).
__device__ __forceinline__ int quant1(float x, float scale) {
  return __float_as_int(__fadd_rn(__fmul_rn(x, scale), 12582912.0f));
}

__device__ __forceinline__ uint32_t pack4(int a, int b, int c, int d) {
  uint32_t ab, cd, r;
  asm("prmt.b32 %0, %1, %2, 0x0040;" : "=r"(ab) : "r"(a), "r"(b));
  asm("prmt.b32 %0, %1, %2, 0x0040;" : "=r"(cd) : "r"(c), "r"(d));
  asm("prmt.b32 %0, %1, %2, 0x5410;" : "=r"(r) : "r"(ab), "r"(cd));
  return r;
}

// Where a trace of the current phase goes (null pointers: nothing).
struct PhaseTrace {
  float *v;      // the fp32 input vector [K]
  int8_t *q;     // its codes [K]
  float *s;      // its scale
};

// Polls the exchange entries of this thread's groups of four values (group
// gi = threadIdx.x + i * kThreads, gi < groups) until every entry carries
// epoch ep, and returns their values in v.  Gives up (false) after `limit`
// cycles or once the abort word is set.
template <int V4>
__device__ __forceinline__ bool poll_entries(const unsigned long long *xin,
                                             int groups, unsigned ep,
                                             const unsigned int *abort,
                                             long long limit,
                                             float4 (&v)[V4]) {
  long long t0 = 0;
  int spin = 0;
  for (;;) {
    bool ok = true;
#pragma unroll
    for (int i = 0; i < V4; ++i) {
      const int gi = threadIdx.x + i * kThreads;
      if (gi < groups) {
        unsigned long long e0, e1, e2, e3;
        ld_entries(xin + 4 * gi, e0, e1);
        ld_entries(xin + 4 * gi + 2, e2, e3);
        ok = ok && unsigned(e0 >> 32) == ep && unsigned(e1 >> 32) == ep &&
             unsigned(e2 >> 32) == ep && unsigned(e3 >> 32) == ep;
        v[i] = make_float4(__uint_as_float(unsigned(e0)),
                           __uint_as_float(unsigned(e1)),
                           __uint_as_float(unsigned(e2)),
                           __uint_as_float(unsigned(e3)));
      } else {
        v[i] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
      }
    }
    if (ok) return true;
    if (spin == 0) t0 = clock64();
    if ((++spin & 31) == 0 &&
        (clock64() - t0 > limit || ld_flag(abort) != 0u))
      return false;
  }
}

// The prologue of a phase: the input vector v [K] (from the caller's h_in
// with plain loads, or polled from an exchange buffer until every entry
// carries epoch ep), its RMSNorm statistics, and the int8 codes
//   q = rint(((v * gamma) * r) * s),  r = 1 / sqrt(sum v^2 / K + eps),
//   s = 127 / max(max|v * gamma| * r, 1e-5)
// in xs (zero from K to 64 C), the scale in s_sm[0] and each warp's sum of
// the codes in sx_part.  Four consecutive values per thread and step.
// Returns false (CTA-uniform) if a poll gave up.
template <int V4>
__device__ __forceinline__ bool prologue(
    int K, int C, const float *gamma, const float *plain,
    const unsigned long long *xin, unsigned ep, float eps,
    const unsigned int *abort, int8_t *xs, float *red, float *s_sm,
    int *sx_part, const PhaseTrace &tr) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int groups = K >> 2;
  float4 gm[V4], v[V4];
#pragma unroll
  for (int i = 0; i < V4; ++i) {
    const int gi = tid + i * kThreads;
    gm[i] = gi < groups ? __ldg(reinterpret_cast<const float4 *>(gamma) + gi)
                        : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
  }
  bool failed = false;
  if (plain) {  // the caller's rows are only 4-byte aligned
#pragma unroll
    for (int i = 0; i < V4; ++i) {
      const int gi = tid + i * kThreads;
      v[i] = gi < groups
                 ? make_float4(__ldg(plain + 4 * gi), __ldg(plain + 4 * gi + 1),
                               __ldg(plain + 4 * gi + 2),
                               __ldg(plain + 4 * gi + 3))
                 : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    }
  } else {
    failed = !poll_entries<V4>(xin, groups, ep, abort, kWaitLimitCycles, v);
  }
  // statistics: sum of squares and the largest |v * gamma|, reduced over
  // the warp by a fixed shuffle tree, then over the 16 warps in order
  float ss = 0.0f, mx = 0.0f;
#pragma unroll
  for (int i = 0; i < V4; ++i) {
    ss += v[i].x * v[i].x;
    ss += v[i].y * v[i].y;
    ss += v[i].z * v[i].z;
    ss += v[i].w * v[i].w;
    mx = fmaxf(mx, fabsf(__fmul_rn(v[i].x, gm[i].x)));
    mx = fmaxf(mx, fabsf(__fmul_rn(v[i].y, gm[i].y)));
    mx = fmaxf(mx, fabsf(__fmul_rn(v[i].z, gm[i].z)));
    mx = fmaxf(mx, fabsf(__fmul_rn(v[i].w, gm[i].w)));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    ss += __shfl_xor_sync(0xffffffffu, ss, o);
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  }
  if (lane == 0) {
    red[warp] = ss;
    red[32 + warp] = mx;
  }
  if (__syncthreads_or(failed)) return false;
  ss = 0.0f;
  mx = 0.0f;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) {
    ss += red[w];
    mx = fmaxf(mx, red[32 + w]);
  }
  const float r = 1.0f / sqrtf(ss / static_cast<float>(K) + eps);
  // rounding is monotone: mx * r is exactly the largest |(v * gamma) * r|
  const float scale = 127.0f / fmaxf(__fmul_rn(mx, r), 1e-5f);
  uint32_t *xw = reinterpret_cast<uint32_t *>(xs);
  int p = 0;
#pragma unroll
  for (int i = 0; i < V4; ++i) {
    const int gi = tid + i * kThreads;
    if (gi < groups) {
      const uint32_t word =
          pack4(quant1(__fmul_rn(__fmul_rn(v[i].x, gm[i].x), r), scale),
                quant1(__fmul_rn(__fmul_rn(v[i].y, gm[i].y), r), scale),
                quant1(__fmul_rn(__fmul_rn(v[i].z, gm[i].z), r), scale),
                quant1(__fmul_rn(__fmul_rn(v[i].w, gm[i].w), r), scale));
      xw[gi] = word;
      p = dp4a_us(0x01010101u, word, p);
      if (tr.q) {  // trace buffers carry no alignment promise
#pragma unroll
        for (int b = 0; b < 4; ++b) tr.q[4 * gi + b] = int8_t(word >> (8 * b));
      }
      if (tr.v) {
        tr.v[4 * gi] = v[i].x;
        tr.v[4 * gi + 1] = v[i].y;
        tr.v[4 * gi + 2] = v[i].z;
        tr.v[4 * gi + 3] = v[i].w;
      }
    }
  }
  for (int w = groups + tid; w < C * 16; w += kThreads) xw[w] = 0u;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) p += __shfl_xor_sync(0xffffffffu, p, o);
  if (lane == 0) sx_part[warp] = p;
  if (tid == 0) {
    s_sm[0] = scale;
    if (tr.s) *tr.s = scale;
  }
  return true;
}

// A piece of a warp's run: local row group g, first chunk c, len chunks, and
// whether it ends a row group or the run (the warp then folds its sums).
__host__ __device__ inline uint32_t pack_piece(int g, int c, int len,
                                               bool fold) {
  return uint32_t(g) | (uint32_t(c) << 8) | (uint32_t(len) << 16) |
         (fold ? (1u << 24) : 0u);
}

// Cuts chunks [lo, hi) of a CTA's range (C chunks per row) into pieces of
// at most kSlotChunks that never cross a row group; writes up to cap of them
// and returns how many there are.
__host__ __device__ inline int run_pieces(int lo, int hi, int C,
                                          uint32_t *out, int cap) {
  int n = 0;
  for (int u = lo; u < hi;) {
    const int g = u / C, c = u - g * C;
    int len = C - c < kSlotChunks ? C - c : kSlotChunks;
    if (hi - u < len) len = hi - u;
    if (out && n < cap) out[n] = pack_piece(g, c, len, c + len == C || u + len == hi);
    ++n;
    u += len;
  }
  return n;
}

__global__ void __launch_bounds__(kThreads, 1) decoder_kernel(const DecArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  const DecLayout Lo = dec_layout(a.max_chunks, a.tot_ints, a.n_layers);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  uint8_t *ring = smem + Lo.ring + size_t(warp) * kSlots * kSlotBytes;
  int8_t *xs = reinterpret_cast<int8_t *>(smem + Lo.xs);
  int *tot = reinterpret_cast<int *>(smem + Lo.tot);
  float *red = reinterpret_cast<float *>(smem + Lo.red);
  float *s_sm = reinterpret_cast<float *>(smem + Lo.misc);
  int *sx_part = reinterpret_cast<int *>(smem + Lo.misc) + 8;
  unsigned *base_sm = reinterpret_cast<unsigned *>(smem + Lo.misc) + 24;
  LayerPtrs *table = reinterpret_cast<LayerPtrs *>(smem + Lo.table);
  uint32_t *plist = reinterpret_cast<uint32_t *>(smem + Lo.pieces);
  int *pcnt = reinterpret_cast<int *>(plist + kWarps * kKinds * kMaxPieces);
  int *kglo = pcnt + kWarps * kKinds;  // [kKinds]
  int *kng = kglo + kKinds;            // [kKinds]
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + Lo.bars) + warp * kSlots;
  const int G = gridDim.x;

  // ---- set-up: the pointer table, this CTA's row groups per GEMV kind,
  // and each warp's pieces per kind (the same in every layer) ----
  {
    const int words = a.n_layers * int(sizeof(LayerPtrs) / 8);
    const unsigned long long *src =
        reinterpret_cast<const unsigned long long *>(a.layers);
    unsigned long long *dst = reinterpret_cast<unsigned long long *>(table);
    for (int i = tid; i < words; i += kThreads) dst[i] = src[i];
    if (tid < kKinds) {
      int g_lo, n_g;
      cta_groups(a.geo[tid], blockIdx.x, G, g_lo, n_g);
      kglo[tid] = g_lo;
      kng[tid] = n_g;
    }
    if (tid == 0) base_sm[0] = ld_flag(a.ctl);
    __syncthreads();
    if (lane < kKinds) {
      const int k = lane, C = a.geo[k].chunks;
      const int U = kng[k] * C;
      pcnt[warp * kKinds + k] = run_pieces(
          int(int64_t(U) * warp / kWarps), int(int64_t(U) * (warp + 1) / kWarps),
          C, plist + (warp * kKinds + k) * kMaxPieces, kMaxPieces);
    }
    __syncthreads();
  }
  const unsigned base = base_sm[0];
  const int *mycnt = pcnt + warp * kKinds;
  const uint32_t *mylist = plist + warp * kKinds * kMaxPieces;

  // ---- the warp's stream of weight pieces (lane 0 issues) ----
  // Next piece to request: phase ip (layer il), piece ii of its list.
  int ip = 0, il = 0, ii = 0;
  int issued = 0, consumed = 0;
  auto next_phase = [&]() {
    ++ip;
    if ((ip & 3) == 0 && ++il == a.n_layers) il = 0;
  };
  auto skip_empty = [&]() {
    int skipped = 0;
    while (ip < a.phases && mycnt[ip & 3] == 0) {
      if (++skipped > kKinds) {  // this warp streams nothing at all
        ip = a.phases;
        break;
      }
      next_phase();
    }
  };
  auto issue_one = [&]() {
    const int k = ip & 3;
    const uint32_t e = mylist[k * kMaxPieces + ii];
    const int g = int(e & 0xffu), c = int((e >> 8) & 0xffu);
    const uint32_t bytes = ((e >> 16) & 0xffu) * kGroupChunkBytes;
    const int slot = issued % kSlots;
    const size_t pg = size_t(phys(kglo[k] + g, a.geo[k].pair_half));
    mbar_arrive_expect_tx(&full[slot], bytes);
    bulk_copy_g2s(ring + size_t(slot) * kSlotBytes,
                  table[il].w[k] + (pg * a.geo[k].chunks + c) * kGroupChunkBytes,
                  bytes, &full[slot]);
    ++issued;
    if (++ii == mycnt[k]) {
      ii = 0;
      next_phase();
      skip_empty();
    }
  };
  // Requests pieces until the ring is full (lane 0; the warp's reads of the
  // slots being refilled are complete and ordered before by the caller).
  auto top_up = [&]() {
    if (ip < a.phases && issued - consumed < kSlots) {
      fence_proxy_async_smem();
      while (ip < a.phases && issued - consumed < kSlots) issue_one();
    }
  };
  if (lane == 0) {
    for (int s = 0; s < kSlots; ++s) mbar_init(&full[s], 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    skip_empty();
    top_up();
  }
  __syncwarp();

  const int q = lane >> 3, r = lane & 7;
  float h_reg = 0.0f;  // the residual-stream row this thread owns (wo, w2)
  bool ok = true;
  const bool tracing = a.tr.layer >= 0;
  const int last_t = a.steps - 1;
  int l = 0, t = 0;    // layer and step of phase p

  for (int p = 0; p < a.phases && ok; ++p) {
    const int k = p & 3;
    if (p > 0 && k == 0 && ++l == a.n_layers) {
      l = 0;
      ++t;
    }
    const KindGeo &g = a.geo[k];
    const LayerPtrs &L = table[l];
    const unsigned ep = base + unsigned(p);
    const bool rec = tracing && t == last_t && l == a.tr.layer;
    const int glo = kglo[k], ng = kng[k];
    // static operands of the epilogue, loaded before the input arrives
    float ws0 = 0.0f, ws1 = 0.0f, ws2 = 0.0f;
    if (k == 0) {
      ws0 = bf16r(L.ws[0]);
      ws1 = bf16r(L.ws[1]);
      ws2 = bf16r(L.ws[2]);
    } else if (k == 1) {
      ws0 = bf16r(L.ws[3]);
    } else if (k == 2) {
      ws0 = bf16r(L.ws[4]);
      ws1 = bf16r(L.ws[5]);
    } else {
      ws0 = bf16r(L.ws[6]);
    }
    const int my_n = (glo + (tid >> 3)) * kGroupRows + (tid & 7);
    if (k == 1 && l == 0 && tid < ng * 8 && my_n < g.N)
      h_reg = __ldg(a.h_in + size_t(t) * a.dim + my_n);

    // ---- prologue: the input vector, its norm, the int8 codes ----
    PhaseTrace ptr{nullptr, nullptr, nullptr};
    if (rec && blockIdx.x == 0) {
      const bw_stack_trace &T = a.tr;
      if (k == 0) ptr = {T.h_in, T.q_attn, T.s_attn};
      if (k == 1) ptr = {T.attn, T.q_o, T.s_o};
      if (k == 2) ptr = {nullptr, T.q_ffn, T.s_ffn};
      if (k == 3) ptr = {nullptr, T.q_down, T.s_down};
    }
    const float *plain =
        (k == 0 && l == 0) ? a.h_in + size_t(t) * a.dim : nullptr;
    const unsigned long long *xin =
        a.xch[(k + 3) & 3] + size_t(blockIdx.x % kReplicas) * a.xstride;
    const float *gamma = L.gam + k * a.dim;  // the four gains in order
    bool pro_ok;
    if (g.K <= 4 * kThreads)
      pro_ok = prologue<1>(g.K, g.chunks, gamma, plain, xin, ep - 1u, a.eps,
                           a.ctl + 2, xs, red, s_sm, sx_part, ptr);
    else if (g.K <= 8 * kThreads)
      pro_ok = prologue<2>(g.K, g.chunks, gamma, plain, xin, ep - 1u, a.eps,
                           a.ctl + 2, xs, red, s_sm, sx_part, ptr);
    else
      pro_ok = prologue<4>(g.K, g.chunks, gamma, plain, xin, ep - 1u, a.eps,
                           a.ctl + 2, xs, red, s_sm, sx_part, ptr);
    if (!pro_ok) {
      if (tid == 0) {
        atomicOr(a.err, 32u);
        atomicExch(a.ctl + 2, 1u);
      }
      ok = false;
      break;
    }
    for (int i = tid; i < ng * 8; i += kThreads) tot[i] = 0;
    __syncthreads();  // codes, scale, code sums and zeroed totals visible

    // ---- this warp's share of the dot products ----
    int acc[1][4] = {{0, 0, 0, 0}};
    bool wait_ok = true;
    const int npieces = mycnt[k];
    for (int i = 0; i < npieces; ++i) {
      // a piece is normally requested phases ahead; if the ring could not
      // hold it yet, request it now (its slot is free)
      if (lane == 0 && issued <= consumed) {
        fence_proxy_async_smem();
        issue_one();
      }
      const int slot = consumed % kSlots;
      const uint32_t parity = uint32_t(consumed / kSlots) & 1u;
      if (!__all_sync(0xffffffffu, mbar_wait(&full[slot], parity))) {
        wait_ok = false;
        break;
      }
      const uint32_t e = mylist[k * kMaxPieces + i];
      dot_row_group<1>(ring + size_t(slot) * kSlotBytes, xs, 0u,
                       int((e >> 8) & 0xffu), int((e >> 16) & 0xffu), q, r,
                       acc);
      ++consumed;
      if (e >> 24) {  // the piece ends a row group or the run
        const int v = fold_row(acc[0]);
        if (q == 0) atomicAdd(&tot[int(e & 0xffu) * 8 + r], v);
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[0][j] = 0;
      }
    }
    __syncwarp();
    if (__syncthreads_or(!wait_ok)) {  // every row total is complete
      if (tid == 0) {
        atomicOr(a.err, 4u);
        atomicExch(a.ctl + 2, 1u);
      }
      ok = false;
      break;
    }

    // ---- epilogue: scale, publish the next phase's input ----
    int sx = 0;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) sx += sx_part[w];
    const float s = s_sm[0];
    unsigned long long *xout = a.xch[k];
    if (k == 2) {  // (gate, up) pairs -> relu(gate)^2 * up
      if (tid < (ng >> 1) * 8) {
        const int jl = tid >> 3;
        const int f = ((glo >> 1) + jl) * kGroupRows + r;
        const __nv_bfloat16 yg = scaled(tot[(2 * jl) * 8 + r] - sx, s, ws0);
        const __nv_bfloat16 yu =
            scaled(tot[(2 * jl + 1) * 8 + r] - sx, s, ws1);
        const float gv = bf16r(yg);
        const float rl = gv > 0.0f ? gv : 0.0f;
        const float gated = __fmul_rn(__fmul_rn(rl, rl), bf16r(yu));
        publish(xout + f, a.xstride, entry(gated, ep));
        if (rec && a.tr.gu) {
          reinterpret_cast<__nv_bfloat16 *>(a.tr.gu)[f] = yg;
          reinterpret_cast<__nv_bfloat16 *>(a.tr.gu)[a.ffn + f] = yu;
        }
      }
    } else if (tid < ng * 8 && my_n < g.N) {
      const int n = my_n;
      const int total = tot[tid] - sx;
      if (k == 0) {  // q | k | v; the value heads are the attention output
        const float wsv =
            n < a.n_heads * a.hd ? ws0 : (n < a.v_off ? ws1 : ws2);
        const __nv_bfloat16 y = scaled(total, s, wsv);
        if (rec && a.tr.qkv) reinterpret_cast<__nv_bfloat16 *>(a.tr.qkv)[n] = y;
        if (n >= a.v_off) {
          const int j = n - a.v_off;
          const int kv = j / a.hd, d = j - kv * a.hd;
          const unsigned long long en = entry(bf16r(y), ep);
          unsigned long long *dst = xout + size_t(kv) * a.group * a.hd + d;
          for (int u = 0; u < a.group; ++u)
            publish(dst + u * a.hd, a.xstride, en);
        }
      } else {  // wo or w2: the residual add
        const __nv_bfloat16 y = scaled(total, s, ws0);
        const float hn = h_reg + bf16r(y);
        h_reg = hn;
        if (k == 1) {
          publish(xout + n, a.xstride, entry(hn, ep));
          if (rec && a.tr.o) reinterpret_cast<__nv_bfloat16 *>(a.tr.o)[n] = y;
          if (rec && a.tr.h_mid) a.tr.h_mid[n] = hn;
        } else {
          if (l == a.n_layers - 1)
            a.h_out[size_t(t) * a.dim + n] = hn;
          else
            publish(xout + n, a.xstride, entry(hn, ep));
          if (rec && a.tr.down)
            reinterpret_cast<__nv_bfloat16 *>(a.tr.down)[n] = y;
        }
      }
    }
    // refill the ring while the next phase's input is produced
    if (lane == 0) top_up();
  }

  // Copies still in flight land before the CTA may leave.
  if (lane == 0)
    for (int i = consumed; i < issued; ++i)
      if (!mbar_wait(&full[i % kSlots], uint32_t(i / kSlots) & 1u))
        atomicOr(a.err, 2u);
  __syncthreads();
  // The last CTA to leave moves the epoch counter past this call's phases.
  if (tid == 0) {
    __threadfence();
    const unsigned prev = atomicAdd(a.ctl + 1, 1u);
    if (prev == unsigned(G) - 1u) {
      const unsigned next = base + unsigned(a.phases);
      a.ctl[1] = 0u;
      a.ctl[2] = 0u;
      a.ctl[0] = next < 0x7fff0000u ? next : 1u;
      __threadfence();
    }
  }
}



// Failure-detection self-test of the exchange poll: entries that nothing
// ever writes (a zeroed array) are polled for epoch 1 with a short limit;
// the poll must give up, set bit 64 of the device error word and return.
__device__ unsigned long long g_selftest_entries[64];
__device__ unsigned int g_selftest_abort;

__global__ void selftest_poll_kernel(unsigned int *err, long long limit) {
  float4 v[1];
  if (!poll_entries<1>(g_selftest_entries, 16, 1u, &g_selftest_abort, limit,
                       v) &&
      threadIdx.x == 0)
    atomicOr(err, 64u);
}

}  // namespace dec

// ---------------------------------------------------------------------------
// Host side.

namespace {

using namespace dec;

struct DecShape {
  KindGeo geo[kKinds];
  int max_chunks, tot_ints;
  uint32_t smem;
};

DecShape decoder_shape(int dim, int ffn, int n_heads, int n_kv, int n_layers,
                       int sms) {
  DecShape d{};
  const int hd = dim / n_heads;
  const int qkv_n = (n_heads + 2 * n_kv) * hd;
  auto geo = [](int N, int K, int pair_half) {
    KindGeo g;
    g.N = N;
    g.K = K;
    g.chunks = chunks_per_row(K);
    g.n_groups = int(padded_rows(N) / kGroupRows);
    g.pair_half = pair_half;
    return g;
  };
  d.geo[0] = geo(qkv_n, dim, 0);
  d.geo[1] = geo(dim, dim, 0);
  d.geo[2] = geo(2 * ffn, dim, ffn / kGroupRows);
  d.geo[3] = geo(dim, ffn, 0);
  d.max_chunks = chunks_per_row(dim > ffn ? dim : ffn);
  int most = 0;
  for (int k = 0; k < kKinds; ++k) {
    const KindGeo &g = d.geo[k];
    const int groups = g.pair_half ? 2 * ((g.pair_half + sms - 1) / sms)
                                   : (g.n_groups + sms - 1) / sms;
    most = groups > most ? groups : most;
  }
  d.tot_ints = most * kGroupRows;
  d.smem = dec_layout(d.max_chunks, d.tot_ints, n_layers).total;
  return d;
}

}  // namespace

// Entries between the copies of the exchange buffers (a multiple of 32, so
// every copy starts on its own 256-byte boundary).
size_t xch_stride(int dim, int ffn) {
  return (size_t(3 * dim + ffn) + 31) / 32 * 32;
}

size_t decoder_xch_bytes(int dim, int ffn) {
  return xch_stride(dim, ffn) * kReplicas * sizeof(unsigned long long);
}

size_t decoder_table_bytes(int n_layers) {
  return sizeof(LayerPtrs) * size_t(n_layers);
}

bool decoder_fits(int dim, int ffn, int n_heads, int n_kv, int n_layers) {
  const int sms = device_sm_count();
  if (sms <= 0 || n_layers > kMaxLayers) return false;
  const DecShape d = decoder_shape(dim, ffn, n_heads, n_kv, n_layers, sms);
  // one residual row per thread in the wo and w2 epilogues
  if (d.smem > 227u * 1024u || d.tot_ints > kThreads) return false;
  // every warp's run of every kind in at most kMaxPieces pieces, with its
  // row groups and chunks in the 8-bit fields of a piece
  for (int k = 0; k < kKinds; ++k) {
    const KindGeo &g = d.geo[k];
    if (g.chunks > 255) return false;
    for (int b = 0; b < sms; ++b) {
      int g_lo, n_g;
      cta_groups(g, b, sms, g_lo, n_g);
      if (n_g > 255) return false;
      const int U = n_g * g.chunks;
      for (int w = 0; w < kWarps; ++w)
        if (run_pieces(int(int64_t(U) * w / kWarps),
                       int(int64_t(U) * (w + 1) / kWarps), g.chunks, nullptr,
                       0) > kMaxPieces)
          return false;
    }
  }
  return true;
}

cudaError_t decoder_upload_table(void *table, int n_layers,
                                 const uint8_t *const *wqkv,
                                 const uint8_t *const *wo,
                                 const uint8_t *const *w13,
                                 const uint8_t *const *w2,
                                 const bw_bf16 *const *ws,
                                 const float *const *gammas) {
  LayerPtrs *host = new (std::nothrow) LayerPtrs[n_layers];
  if (!host) return cudaErrorMemoryAllocation;
  for (int l = 0; l < n_layers; ++l) {
    host[l].w[0] = wqkv[l];
    host[l].w[1] = wo[l];
    host[l].w[2] = w13[l];
    host[l].w[3] = w2[l];
    host[l].ws = reinterpret_cast<const __nv_bfloat16 *>(ws[l]);
    host[l].gam = gammas[l];
  }
  const cudaError_t e = cudaMemcpy(table, host, decoder_table_bytes(n_layers),
                                   cudaMemcpyHostToDevice);
  delete[] host;
  return e;
}

cudaError_t launch_selftest_poll(cudaStream_t stream) {
  int dev = 0, khz = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess)
    e = cudaDeviceGetAttribute(&khz, cudaDevAttrClockRate, dev);
  if (e != cudaSuccess) return e;
  unsigned int *err = device_error_word();
  if (!err) return cudaErrorInvalidSymbol;
  const long long limit = (long long)(khz > 0 ? khz : 2000000) * 10;  // ~10 ms
  selftest_poll_kernel<<<1, 32, 0, stream>>>(err, limit);
  return cudaGetLastError();
}

cudaError_t launch_decoder(const DecoderLaunch &l, cudaStream_t stream) {
  static std::atomic<bool> configured[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  const int sms = device_sm_count();
  if (sms <= 0) return cudaErrorNoDevice;
  const DecShape d =
      decoder_shape(l.dim, l.ffn, l.n_heads, l.n_kv, l.n_layers, sms);
  if (!configured[dev].load(std::memory_order_relaxed)) {
    e = cudaFuncSetAttribute(decoder_kernel,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             227 * 1024);
    if (e != cudaSuccess) return e;
    configured[dev].store(true, std::memory_order_relaxed);
  }
  int per_sm = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, decoder_kernel,
                                                    kThreads, d.smem);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) return cudaErrorInvalidConfiguration;

  DecArgs a{};
  a.layers = static_cast<const LayerPtrs *>(l.table);
  a.n_layers = l.n_layers;
  a.steps = l.steps;
  a.phases = l.steps * l.n_layers * kKinds;
  a.dim = l.dim;
  a.ffn = l.ffn;
  a.n_heads = l.n_heads;
  a.n_kv = l.n_kv;
  a.hd = l.dim / l.n_heads;
  a.group = l.n_heads / l.n_kv;
  a.v_off = (l.n_heads + l.n_kv) * a.hd;
  a.eps = l.eps;
  for (int k = 0; k < kKinds; ++k) a.geo[k] = d.geo[k];
  a.h_in = l.h_in;
  a.h_out = l.h_out;
  unsigned long long *x = static_cast<unsigned long long *>(l.xch);
  a.xch[0] = x;                          // attention output [dim]
  a.xch[1] = x + l.dim;                  // h after wo [dim]
  a.xch[2] = x + 2 * l.dim;              // gated product [ffn]
  a.xch[3] = x + 2 * l.dim + l.ffn;      // h after w2 [dim]
  a.xstride = xch_stride(l.dim, l.ffn);
  a.ctl = l.ctl;
  a.err = device_error_word();
  if (!a.err) return cudaErrorInvalidSymbol;
  if (l.trace) {
    a.tr = *l.trace;
  } else {
    a.tr = bw_stack_trace{};
    a.tr.layer = -1;
  }
  a.max_chunks = d.max_chunks;
  a.tot_ints = d.tot_ints;

  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(sms));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = d.smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, decoder_kernel, a);
}

}  // namespace bw
