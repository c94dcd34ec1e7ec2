// bw_stack.cu -- the decoder layer stack: chained W2A8 GEMVs with the fp32
// glue between them (RMSNorm, absmax requantisation, residual adds, the
// squared-ReLU gate and one-token grouped attention).
//
// Source: "BitNet GPU 推理框架：从零构建 W2A8 的 2-bit 大模型 CUDA GEMV 内核":
// §一 (BitNet-2B shape: 30 layers, dim 2560, 20 query / 5 KV heads, ffn
// 6912), §4.1 (the fused q|k|v and gate|up projections; attention_norm,
// attn_sub_norm, ffn_norm, ffn_sub_norm), §六 item 3 (per-token absmax
// quantisation before every W2A8 GEMV), §六 item 1 (decode replayed from a
// CUDA graph).
//
// One layer, M = 1 (h is the fp32 residual stream):
//   (q, s) <- quant(rmsnorm(h) * g_attn)              -> qkv = W2A8(wqkv)
//   (q, s) <- quant(rmsnorm(attn(qkv)) * g_attn_sub)  -> o   = W2A8(wo)
//   h <- h + o
//   (q, s) <- quant(rmsnorm(h) * g_ffn)               -> gu  = W2A8(w13)
//   (q, s) <- quant(rmsnorm(relu(gate)^2 up) * g_sub) -> down = W2A8(w2)
//   h <- h + down
// attn() is attention over a one-token context: the softmax of one score is
// 1, so query head h returns the value vector of KV head h / (heads / kv).
// A stack made with bw_stack_create_kv attends over a KV cache instead: one
// more launch per layer (bw_attn.cu) rotates and appends the token's key
// and value at the current position and attends over positions 0..p; the
// last launch of a step advances the position.
//
// Each GEMV is ONE launch of the pipe GEMV kernel (bw_pipe.cuh); the glue
// is split between launches so that every value is computed once:
//  * the epilogue of each launch writes, besides its bf16 output, the fp32
//    values the NEXT RMSNorm reads (the attention output, h after the
//    residual add, or the gated product; the wo and w2 epilogues add their
//    outputs into h, each element once) and, per CTA, the partial sum of
//    their squares and the partial max of |value * gain|;
//  * the prologue of the next launch reduces those partials (in the same
//    fixed order in every CTA) to the RMS factor and the absmax scale, and
//    quantises the values into its shared-memory activations.
// w13 streams its row groups in (gate j, up j) pairs so that the CTA that
// computes gate[f] also holds up[f].  The first GEMV of a step normalises h
// itself (no earlier launch).  Four launches per layer, all with
// programmatic dependent launch; one decode step is captured once as a
// CUDA graph.
#include <cstdlib>
#include <new>
#include <vector>

#include "bw_pipe.cuh"

namespace bw {
namespace {

using namespace pipe;

constexpr int kPrologueThreads = kPipeWarps * 32;
constexpr int kMaxGlueK = 32 * kPrologueThreads;  // 8192: V <= 32 per thread
constexpr int kMaxGroup = 8;          // query heads per KV head unrolled
constexpr int kPartialsPerThread = 2;  // partials loaded at once: 512 per CTA

// rint(x * scale) in the low byte of the result: the fp32 product (round to
// nearest even), then an fp32 add of 1.5 * 2^23, whose result has a unit in
// the last place of 1, so the add rounds the product to an integer (ties to
// even) and leaves it, in two's complement, in the low mantissa bits while
// |x * scale| < 2^22.  Every caller quantises with scale = 127 / max(A,
// 1e-5) where A is the exact largest |x| of the values it quantises, so
// |x * scale| <= 127 (1 + 2^-24) and the code is in [-127, 127]: the clamp
// to [-128, 127] never acts.  Two full-rate fp32 instructions, where a
// float-to-int convert runs at a fraction of that rate and every CTA
// quantises the whole vector.
__device__ __forceinline__ int quant1(float x, float scale) {
  return __float_as_int(__fadd_rn(__fmul_rn(x, scale), 12582912.0f));
}

__device__ __forceinline__ uint32_t byte_perm(uint32_t a, uint32_t b,
                                              uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}

// The low bytes of four int32 codes, packed in order into one word.
__device__ __forceinline__ uint32_t pack4(int a, int b, int c, int d) {
  const uint32_t ab = byte_perm(uint32_t(a), uint32_t(b), 0x0040u);
  const uint32_t cd = byte_perm(uint32_t(c), uint32_t(d), 0x0040u);
  return byte_perm(ab, cd, 0x5410u);
}

// Prologue of the first GEMV of a step (h comes from the caller, so no
// earlier launch has its statistics): v = h[k] for k < K, then
//   n = (v * (1 / sqrt(mean(v^2) + eps))) * gamma,
//   s = 127 / max(absmax n, 1e-5),  q = clamp(rint(n * s), -128, 127),
// all in fp32 with fixed-order CTA reductions.  CTA 0 copies q to trace_q
// and s to trace_s, each when set.
template <int V>
struct NormQuantH {
  const float *h;
  const float *gamma;
  int K;
  float eps;
  int8_t *trace_q;
  float *trace_s;

  struct Pre {  // the gains are static: loaded before the wait
    float gm[V];
  };
  __device__ __forceinline__ Pre pre_wait() const {
    Pre p;
#pragma unroll
    for (int i = 0; i < V; ++i) {
      const int k = threadIdx.x + i * kPrologueThreads;
      p.gm[i] = k < K ? gamma[k] : 0.0f;
    }
    return p;
  }

  template <int MT>
  __device__ __forceinline__ void stage(const Pre &pre, const StageCtx &c,
                                        int (&part)[MT]) const {
    static_assert(MT == 1, "the stack runs one token per step");
    int8_t *xs = c.xs;
    float *s_sm = c.s_sm, *red = c.red;
    const int chunks = c.chunks;
    const int tid = threadIdx.x;
    float v[V];
#pragma unroll
    for (int i = 0; i < V; ++i) {
      const int k = tid + i * kPrologueThreads;
      v[i] = k < K ? h[k] : 0.0f;
    }
    const float *gm = pre.gm;
    float ss = 0.0f, unused = 0.0f;
#pragma unroll
    for (int i = 0; i < V; ++i) ss += v[i] * v[i];
    cta_sum_max(ss, unused, red);
    const float r = 1.0f / sqrtf(ss / static_cast<float>(K) + eps);
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < V; ++i) {
      v[i] = (v[i] * r) * gm[i];
      amax = fmaxf(amax, fabsf(v[i]));
    }
    float unused2 = 0.0f;
    cta_sum_max(unused2, amax, red);
    const float scale = 127.0f / fmaxf(amax, 1e-5f);
    if (tid == 0) s_sm[0] = scale;
    const bool tr = trace_q && blockIdx.x == 0;
    int p = 0;
#pragma unroll
    for (int i = 0; i < V; ++i) {
      const int k = tid + i * kPrologueThreads;
      if (k < K) {
        const int qv = int8_t(quant1(v[i], scale));  // low byte, signed
        xs[k] = int8_t(qv);
        p += qv;
        if (tr) trace_q[k] = int8_t(qv);
      }
    }
    for (int k = K + tid; k < chunks * kChunkWeights; k += kPrologueThreads)
      xs[k] = 0;
    if (trace_s && blockIdx.x == 0 && tid == 0) *trace_s = scale;
    part[0] = p;
  }
};

// Prologue of every other GEMV: the previous launch wrote the fp32 values
// v[K] to normalise and, per CTA, the partial statistics (sum of v^2, max
// of |v * gamma|) over the values it wrote.  The CTA reduces the P
// partials in the same fixed order in every CTA, so every CTA gets the same
//   r = 1 / sqrt(sum / K + eps),  s = 127 / max(max * r, 1e-5),
// and quantises q = clamp(rint(((v * gamma) * r) * s)).  Rounding is
// monotone, so max * r is exactly the largest |(v * gamma) * r|.  Four
// values per thread and step (16-byte loads, one 32-bit store of codes).
template <int V4>
struct NormQuantP {
  const float *src;     // v [K], 16-byte aligned
  const float *gamma;   // [K], 16-byte aligned
  const float2 *part;   // [P]
  int P, K;
  float eps;
  int8_t *trace_q;
  float *trace_s;

  struct Pre {  // the gains are static: loaded before the wait
    float4 gm[V4];
  };
  __device__ __forceinline__ Pre pre_wait() const {
    Pre p;
#pragma unroll
    for (int i = 0; i < V4; ++i) {
      const int g = threadIdx.x + i * kPrologueThreads;
      p.gm[i] = g < (K >> 2)
                    ? __ldg(reinterpret_cast<const float4 *>(gamma) + g)
                    : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    }
    return p;
  }

  template <int MT>
  __device__ __forceinline__ void stage(const Pre &pre, const StageCtx &c,
                                        int (&part_out)[MT]) const {
    static_assert(MT == 1, "the stack runs one token per step");
    int8_t *xs = c.xs;
    float *s_sm = c.s_sm, *red = c.red;
    const int chunks = c.chunks;
    const int tid = threadIdx.x;
    const int groups = K >> 2;  // K is a multiple of 4
    // All loads are issued before the first is used (issue is in order):
    // the values, then at most kPartialsPerThread partials per thread.
    float4 v[V4];
#pragma unroll
    for (int i = 0; i < V4; ++i) {
      const int g = tid + i * kPrologueThreads;
      if (g < groups) v[i] = __ldg(reinterpret_cast<const float4 *>(src) + g);
    }
    float2 pv[kPartialsPerThread];
#pragma unroll
    for (int j = 0; j < kPartialsPerThread; ++j) {
      const int i = tid + j * kPrologueThreads;
      pv[j] = i < P ? part[i] : make_float2(0.0f, 0.0f);
    }
    float ss = 0.0f, mx = 0.0f;
#pragma unroll
    for (int j = 0; j < kPartialsPerThread; ++j) {
      ss += pv[j].x;
      mx = fmaxf(mx, pv[j].y);
    }
    for (int i = tid + kPartialsPerThread * kPrologueThreads; i < P;
         i += kPrologueThreads) {  // more producer CTAs: rare, sequential
      const float2 pe = part[i];
      ss += pe.x;
      mx = fmaxf(mx, pe.y);
    }
    cta_sum_max(ss, mx, red);  // same fixed order in every CTA
    const float4 *gm = pre.gm;
    const float r = 1.0f / sqrtf(ss / static_cast<float>(K) + eps);
    const float scale = 127.0f / fmaxf(__fmul_rn(mx, r), 1e-5f);
    if (tid == 0) s_sm[0] = scale;
    const bool tr = trace_q && blockIdx.x == 0;
    uint32_t *xw = reinterpret_cast<uint32_t *>(xs);
    int p = 0;
#pragma unroll
    for (int i = 0; i < V4; ++i) {
      const int g = tid + i * kPrologueThreads;
      if (g < groups) {
        const uint32_t word =
            pack4(quant1(__fmul_rn(__fmul_rn(v[i].x, gm[i].x), r), scale),
                  quant1(__fmul_rn(__fmul_rn(v[i].y, gm[i].y), r), scale),
                  quant1(__fmul_rn(__fmul_rn(v[i].z, gm[i].z), r), scale),
                  quant1(__fmul_rn(__fmul_rn(v[i].w, gm[i].w), r), scale));
        if (tr) {
#pragma unroll
          for (int b = 0; b < 4; ++b)
            trace_q[4 * g + b] = int8_t(word >> (8 * b));
        }
        xw[g] = word;
        p = dp4a_us(0x01010101u, word, p);
      }
    }
    for (int w = groups + tid; w < chunks * (kChunkWeights / 4);
         w += kPrologueThreads)
      xw[w] = 0u;
    if (trace_s && blockIdx.x == 0 && tid == 0) *trace_s = scale;
    part_out[0] = p;
  }
};

// Scaled bf16 output of one row: bf16((acc / s) * ws), IEEE fp32.
__device__ __forceinline__ __nv_bfloat16 scaled_bf16(int total, float s,
                                                     float ws) {
  return __float2bfloat16_rn((static_cast<float>(total) / s) * ws);
}

// Writes this CTA's partial statistics (every thread calls it).
__device__ __forceinline__ void write_partials(float2 *out, float ss, float mx,
                                               float *red) {
  if (!out) return;
  cta_sum_max(ss, mx, red);
  if (threadIdx.x == 0) out[blockIdx.x] = make_float2(ss, mx);
}

// Epilogue of wqkv: qkv[n] (bf16, scales q | k | v), and for the value rows
// the one-token attention output attn[h hd + d] = v[kv hd + d] for the
// `group` query heads h of KV head kv (fp32), with the partial statistics
// of attn against the attn_sub_norm gains.  With attn null (a stack with a
// KV cache) it writes qkv only: the attention launch that follows produces
// attn and its statistics.
struct EpiQKV {
  __nv_bfloat16 *qkv;
  float *attn;
  const __nv_bfloat16 *ws;
  WsSegments seg;
  int v_off, hd, group;
  const float *gamma_next;
  float2 *part_out;

  __device__ __forceinline__ float scale_value() const {
    return int(threadIdx.x) < seg.n_ws ? __bfloat162float(ws[threadIdx.x])
                                       : 0.0f;
  }
  // The gains of the (up to 4) query-head positions of the thread's first
  // row, if it is a value row: static, so loaded right after the wait.
  __device__ __forceinline__ float4 prefetch(const PipeArgs &a, int g_lo,
                                             int n_g) const {
    const int t = threadIdx.x;
    const int n = (g_lo + (t >> 3)) * kGroupRows + (t & 7);
    float4 p = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    if (attn && t < n_g * 8 && n < a.N && n >= v_off && group <= 4) {
      const int j = n - v_off;
      const int kv = j / hd, d = j - kv * hd;
      const float *gp = gamma_next + kv * group * hd + d;
      p.x = gp[0];
      if (group > 1) p.y = gp[hd];
      if (group > 2) p.z = gp[2 * hd];
      if (group > 3) p.w = gp[3 * hd];
    }
    return p;
  }
  template <int MT>
  __device__ __forceinline__ void finish(const PipeArgs &a, const int *tot,
                                         const int (&sx)[MT], int g_lo,
                                         int n_g, const float *s_sm,
                                         const float *ws_sm, float *red,
                                         float4 pre) const {
    float ss = 0.0f, mx = 0.0f;
    for (int t = threadIdx.x; t < n_g * 8; t += blockDim.x) {
      const int gl = t >> 3, rr = t & 7;
      const int n = (g_lo + gl) * kGroupRows + rr;
      if (n >= a.N) continue;
      int sg = 0;
#pragma unroll
      for (int i = 1; i < BW_MAX_WS; ++i)
        if (i < seg.n_ws && n >= seg.bounds[i]) sg = i;
      const __nv_bfloat16 yv =
          scaled_bf16(tot[gl * 8 + rr] - sx[0], s_sm[0], ws_sm[sg]);
      qkv[n] = yv;
      if (attn && n >= v_off) {
        const int j = n - v_off;
        const int kv = j / hd, d = j - kv * hd;
        const float yf = __bfloat162float(yv);
        const int base = kv * group * hd + d;  // position of head kv group
        // gains: prefetched for the thread's first row, else loaded together
        const bool first = t == int(threadIdx.x) && group <= 4;
        const float pv[4] = {pre.x, pre.y, pre.z, pre.w};
        float gv[kMaxGroup];
#pragma unroll
        for (int u = 0; u < kMaxGroup; ++u) {
          if (first && u < 4)
            gv[u] = pv[u];
          else
            gv[u] = u < group ? gamma_next[base + u * hd] : 0.0f;
        }
#pragma unroll
        for (int u = 0; u < kMaxGroup; ++u) {
          if (u < group) {
            attn[base + u * hd] = yf;
            ss += yf * yf;
            mx = fmaxf(mx, fabsf(__fmul_rn(yf, gv[u])));
          }
        }
        for (int u = kMaxGroup; u < group; ++u) {  // more heads per KV head
          attn[base + u * hd] = yf;
          ss += yf * yf;
          mx = fmaxf(mx, fabsf(__fmul_rn(yf, gamma_next[base + u * hd])));
        }
      }
    }
    write_partials(part_out, ss, mx, red);
  }
};

// Epilogue of wo and w2: y[n] (bf16, one scale) and the residual update
// h[n] += y[n] (fp32), with the partial statistics of the new h against the
// gains of the next RMSNorm (none after the last layer).  h[n] and the gain
// of the thread's first row are loaded right after the dependency wait.
struct EpiResid {
  __nv_bfloat16 *y;
  float *h;
  const __nv_bfloat16 *ws;
  const float *gamma_next;  // or null
  float2 *part_out;         // or null
  int *pos_advance;         // or null: the KV position, advanced once

  __device__ __forceinline__ float scale_value() const {
    return threadIdx.x == 0 ? __bfloat162float(ws[0]) : 0.0f;
  }
  __device__ __forceinline__ float4 prefetch(const PipeArgs &a, int g_lo,
                                             int n_g) const {
    const int t = threadIdx.x;
    const int n = (g_lo + (t >> 3)) * kGroupRows + (t & 7);
    if (t >= n_g * 8 || n >= a.N) return make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    return make_float4(h[n], gamma_next ? gamma_next[n] : 0.0f, 0.0f, 0.0f);
  }
  template <int MT>
  __device__ __forceinline__ void finish(const PipeArgs &a, const int *tot,
                                         const int (&sx)[MT], int g_lo,
                                         int n_g, const float *s_sm,
                                         const float *ws_sm, float *red,
                                         float4 pre) const {
    float ss = 0.0f, mx = 0.0f;
    for (int t = threadIdx.x; t < n_g * 8; t += blockDim.x) {
      const int gl = t >> 3, rr = t & 7;
      const int n = (g_lo + gl) * kGroupRows + rr;
      if (n >= a.N) continue;
      const __nv_bfloat16 yv =
          scaled_bf16(tot[gl * 8 + rr] - sx[0], s_sm[0], ws_sm[0]);
      y[n] = yv;
      const bool first = t == int(threadIdx.x);  // prefetched row
      const float hv = first ? pre.x : h[n];
      const float hn = hv + __bfloat162float(yv);
      h[n] = hn;
      if (gamma_next) {
        ss += hn * hn;
        mx = fmaxf(mx, fabsf(__fmul_rn(hn, first ? pre.y : gamma_next[n])));
      }
    }
    write_partials(part_out, ss, mx, red);
    // The last launch of a step: every attention launch of the step has
    // completed (each launch waits for the one before it), so the next
    // token's position can be published.
    if (pos_advance && blockIdx.x == 0 && threadIdx.x == 0) *pos_advance += 1;
  }
};

// Epilogue of w13, streamed with paired row groups (gate group j, then up
// group j): gu[f] and gu[F + f] (bf16, scales gate | up), and the gated
// product g[f] = relu(gate)^2 * up (fp32, exact for bf16 inputs) with its
// partial statistics against the ffn_sub_norm gains.  F is a multiple of 8.
struct EpiGate {
  __nv_bfloat16 *gu;
  float *gated;
  const __nv_bfloat16 *ws;
  int F;
  const float *gamma_next;
  float2 *part_out;

  __device__ __forceinline__ float scale_value() const {
    return threadIdx.x < 2 ? __bfloat162float(ws[threadIdx.x]) : 0.0f;
  }
  __device__ __forceinline__ float4 prefetch(const PipeArgs &, int g_lo,
                                             int n_g) const {
    const int t = threadIdx.x;
    if (t >= (n_g >> 1) * 8) return make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    const int f = ((g_lo >> 1) + (t >> 3)) * kGroupRows + (t & 7);
    return make_float4(gamma_next[f], 0.0f, 0.0f, 0.0f);
  }
  template <int MT>
  __device__ __forceinline__ void finish(const PipeArgs &a, const int *tot,
                                         const int (&sx)[MT], int g_lo,
                                         int n_g, const float *s_sm,
                                         const float *ws_sm, float *red,
                                         float4 pre) const {
    (void)a;
    float ss = 0.0f, mx = 0.0f;
    // g_lo and n_g are even: the CTA holds whole (gate, up) pairs.
    for (int t = threadIdx.x; t < (n_g >> 1) * 8; t += blockDim.x) {
      const int jl = t >> 3, rr = t & 7;
      const int f = ((g_lo >> 1) + jl) * kGroupRows + rr;
      const __nv_bfloat16 yg =
          scaled_bf16(tot[(2 * jl) * 8 + rr] - sx[0], s_sm[0], ws_sm[0]);
      const __nv_bfloat16 yu =
          scaled_bf16(tot[(2 * jl + 1) * 8 + rr] - sx[0], s_sm[0], ws_sm[1]);
      gu[f] = yg;
      gu[F + f] = yu;
      const float g = __bfloat162float(yg);
      const float r = g > 0.0f ? g : 0.0f;
      const float v = __fmul_rn(__fmul_rn(r, r), __bfloat162float(yu));
      gated[f] = v;
      ss += v * v;
      const float gn = t == int(threadIdx.x) ? pre.x : gamma_next[f];
      mx = fmaxf(mx, fabsf(__fmul_rn(v, gn)));
    }
    write_partials(part_out, ss, mx, red);
  }
};

// Partial statistics per launch: at most one entry per CTA; a launch has at
// most n_groups / kPipeMinGroupsPerCta + 1 <= 1025 CTAs for N <= 16384.
constexpr int kMaxPartials = 2048;

template <class Pro, class Epi>
cudaError_t launch_one(const uint8_t *w, int N, int K, int pair_half,
                       const Pro &pro, const Epi &epi, cudaStream_t cs,
                       int *grid) {
  PipeArgs a{};
  a.w = w;
  a.N = N;
  a.chunks = chunks_per_row(K);
  a.n_groups = int(padded_rows(N) / kGroupRows);
  a.pair_half = pair_half;
  a.err = device_error_word();
  if (!a.err) return cudaErrorInvalidSymbol;
  return launch_pipe<1>(a, pro, epi, cs, grid);
}

// First GEMV of a step: the prologue normalises h itself.
template <class Epi>
cudaError_t launch_first(const uint8_t *w, int N, int K, const float *h,
                         const float *gamma, float eps, int8_t *tq, float *ts,
                         const Epi &epi, cudaStream_t cs, int *grid) {
  if (K <= 8 * kPrologueThreads)
    return launch_one(w, N, K, 0, NormQuantH<8>{h, gamma, K, eps, tq, ts},
                      epi, cs, grid);
  if (K <= 16 * kPrologueThreads)
    return launch_one(w, N, K, 0, NormQuantH<16>{h, gamma, K, eps, tq, ts},
                      epi, cs, grid);
  return launch_one(w, N, K, 0, NormQuantH<32>{h, gamma, K, eps, tq, ts},
                    epi, cs, grid);
}

// Every other GEMV: the prologue quantises what the previous launch wrote.
template <class Epi>
cudaError_t launch_next(const uint8_t *w, int N, int K, int pair_half,
                        const float *src, const float *gamma,
                        const float2 *part, int P, float eps, int8_t *tq,
                        float *ts, const Epi &epi, cudaStream_t cs,
                        int *grid) {
  if (K <= 8 * kPrologueThreads)
    return launch_one(w, N, K, pair_half,
                      NormQuantP<2>{src, gamma, part, P, K, eps, tq, ts}, epi,
                      cs, grid);
  if (K <= 16 * kPrologueThreads)
    return launch_one(w, N, K, pair_half,
                      NormQuantP<4>{src, gamma, part, P, K, eps, tq, ts}, epi,
                      cs, grid);
  return launch_one(w, N, K, pair_half,
                    NormQuantP<8>{src, gamma, part, P, K, eps, tq, ts}, epi,
                    cs, grid);
}

WsSegments segments(const int *bounds, int n) {
  WsSegments sg{};
  sg.n_ws = n;
  for (int i = 0; i <= n; ++i) sg.bounds[i] = bounds[i];
  return sg;
}

}  // namespace
}  // namespace bw

using namespace bw;

struct bw_stack {
  bw_stack_desc d;
  std::vector<const uint8_t *> wqkv, wo, w13, w2;
  std::vector<const bw_bf16 *> ws;
  std::vector<const float *> gammas;
  int hd, qkv_n, v_off, group;
  // device scratch
  float *h;                           // residual stream [dim]
  __nv_bfloat16 *qkv, *o, *gu, *dn;   // GEMV outputs
  float *attn, *gated;                // inputs of attn_sub_norm, ffn_sub_norm
  float2 *part;                       // [2][kMaxPartials] partial statistics
  // KV cache (kv_S > 0): [n_layers][Hkv][kv_S][hd] bf16 keys and values,
  // the position of the next token, the attention workspace.
  int kv_S;
  float theta;
  __nv_bfloat16 *kc, *vc;
  int *pos;
  void *attn_ws;
  size_t kv_layer_elems;
  // One captured step per context bucket: graph b serves the tokens whose
  // context (position + 1) is at most graph_len[b] (0: any), its attention
  // launches sized for that; host_pos counts the tokens since the last reset
  // and picks the graph (the kernels read the position on the device).
  static constexpr int kMaxGraphs = 3;
  int n_graphs;
  int graph_len[kMaxGraphs];
  cudaGraphExec_t exec[kMaxGraphs];
  long long host_pos;
  // Stacks without a KV cache run as one persistent kernel per call
  // (bw_decoder.cu): its per-layer pointer table, exchange buffers and
  // control words.
  bool persistent;
  void *dec_table;
  void *dec_xch;
  unsigned int *dec_ctl;
};

namespace {

// Context buckets of a stack with a KV cache (positions + 1), below the
// cache size; a last bucket takes every context.
constexpr int kStackBuckets[2] = {128, 1024};
static_assert(2 + 1 <= bw_stack::kMaxGraphs, "one graph per bucket");

bw_status cuda_err(cudaError_t e) {
  if (e == cudaSuccess) return BW_OK;
  record_cuda_error(int(e));
  return BW_ERR_CUDA;
}

// Device-to-device copy used only when a trace is requested.
cudaError_t trace_copy(void *dst, const void *src, size_t bytes,
                       cudaStream_t cs) {
  if (!dst) return cudaSuccess;
  return cudaMemcpyAsync(dst, src, bytes, cudaMemcpyDeviceToDevice, cs);
}

#define BW_TRY(expr)                             \
  do {                                           \
    bw_status st_ = (expr);                      \
    if (st_ != BW_OK) return st_;                \
  } while (0)
#define BW_TRY_CUDA(expr) BW_TRY(cuda_err(expr))

// One decode step over all layers on fixed buffers: st->h holds the step's
// input on entry and its output on exit.  Each launch's epilogue writes the
// values the next launch normalises, with per-CTA partial statistics in one
// of two alternating buffers (a launch reads the previous launch's buffer
// and writes the other).
bw_status run_step(bw_stack *st, cudaStream_t cs, const bw_stack_trace *tr,
                   int max_len) {
  const bw_stack_desc &d = st->d;
  const int dim = d.dim, ffn = d.ffn;
  const int b_qkv[4] = {0, d.n_heads * st->hd,
                        (d.n_heads + d.n_kv_heads) * st->hd, st->qkv_n};
  const WsSegments seg_qkv = segments(b_qkv, 3);
  float2 *pin = st->part + kMaxPartials;  // read by the next launch
  float2 *pout = st->part;                // written by the next launch
  int P = 0;                              // CTAs of the previous launch
  int grid = 0;
  auto flip = [&]() {
    float2 *t = pin;
    pin = pout;
    pout = t;
    P = grid;
  };
  for (int l = 0; l < d.n_layers; ++l) {
    const float *g = st->gammas[l];
    const __nv_bfloat16 *ws =
        reinterpret_cast<const __nv_bfloat16 *>(st->ws[l]);
    const bool last = l == d.n_layers - 1;
    const bool rec = tr && tr->layer == l;
    if (rec) BW_TRY_CUDA(trace_copy(tr->h_in, st->h, dim * 4, cs));
    // qkv = W2A8(wqkv, quant(attention_norm(h))); attn = value heads (one
    // token) or the attention over the cache (next launch)
    const bool kv = st->kv_S > 0;
    const EpiQKV e_qkv{st->qkv,    kv ? nullptr : st->attn, ws,
                       seg_qkv,    st->v_off,               st->hd,
                       st->group,  kv ? nullptr : g + dim,  kv ? nullptr : pout};
    if (l == 0)
      BW_TRY_CUDA(launch_first(st->wqkv[l], st->qkv_n, dim, st->h, g, d.eps,
                               rec ? tr->q_attn : nullptr,
                               rec ? tr->s_attn : nullptr, e_qkv, cs, &grid));
    else
      BW_TRY_CUDA(launch_next(st->wqkv[l], st->qkv_n, dim, 0, st->h, g, pin,
                              P, d.eps, rec ? tr->q_attn : nullptr,
                              rec ? tr->s_attn : nullptr, e_qkv, cs, &grid));
    flip();
    if (rec) BW_TRY_CUDA(trace_copy(tr->qkv, st->qkv, st->qkv_n * 2, cs));
    if (kv) {
      // attn = attention of the step's token over layer l's cache (the key
      // and value appended at the current position), with the statistics
      // of attn_sub_norm per KV head
      AttnLaunch al{};
      al.qkv = st->qkv;
      al.pos = st->pos;
      al.kc = st->kc + size_t(l) * st->kv_layer_elems;
      al.vc = st->vc + size_t(l) * st->kv_layer_elems;
      al.out = st->attn;
      al.workspace = st->attn_ws;
      al.H = d.n_heads;
      al.Hkv = d.n_kv_heads;
      al.S = st->kv_S;
      al.theta = st->theta;
      al.norm_gamma = g + dim;
      al.norm_part = pout;
      // The position is advanced by the last launch of the previous step
      // and rows before it were appended by earlier steps; the launch
      // before this one (the wqkv GEMV) released its dependents only after
      // its own dependency wait, so all of that has completed when this
      // launch starts: its copies may start before its wait.
      al.past_ready = 1;
      al.max_len = max_len;
      BW_TRY_CUDA(launch_attn(al, cs));
      grid = d.n_kv_heads;
      flip();
    }
    if (rec) BW_TRY_CUDA(trace_copy(tr->attn, st->attn, dim * 4, cs));
    // o = W2A8(wo, quant(attn_sub_norm(attn))); h += o
    BW_TRY_CUDA(launch_next(
        st->wo[l], dim, dim, 0, st->attn, g + dim, pin, P, d.eps,
        rec ? tr->q_o : nullptr, rec ? tr->s_o : nullptr,
        EpiResid{st->o, st->h, ws + 3, g + 2 * dim, pout}, cs, &grid));
    flip();
    if (rec) {
      BW_TRY_CUDA(trace_copy(tr->o, st->o, dim * 2, cs));
      BW_TRY_CUDA(trace_copy(tr->h_mid, st->h, dim * 4, cs));
    }
    // gu = W2A8(w13, quant(ffn_norm(h))); gated = relu(gate)^2 up
    BW_TRY_CUDA(launch_next(
        st->w13[l], 2 * ffn, dim, ffn / kGroupRows, st->h, g + 2 * dim, pin,
        P, d.eps, rec ? tr->q_ffn : nullptr, rec ? tr->s_ffn : nullptr,
        EpiGate{st->gu, st->gated, ws + 4, ffn, g + 3 * dim, pout}, cs,
        &grid));
    flip();
    if (rec) BW_TRY_CUDA(trace_copy(tr->gu, st->gu, 2 * ffn * 2, cs));
    // down = W2A8(w2, quant(ffn_sub_norm(gated))); h += down
    const float *g_next = last ? nullptr : st->gammas[l + 1];
    BW_TRY_CUDA(launch_next(
        st->w2[l], dim, ffn, 0, st->gated, g + 3 * dim, pin, P, d.eps,
        rec ? tr->q_down : nullptr, rec ? tr->s_down : nullptr,
        EpiResid{st->dn, st->h, ws + 6, g_next, last ? nullptr : pout,
                 last && st->kv_S > 0 ? st->pos : nullptr},
        cs, &grid));
    flip();
    if (rec) BW_TRY_CUDA(trace_copy(tr->down, st->dn, dim * 2, cs));
  }
  return BW_OK;
}

// One persistent-kernel launch over `steps` steps (stacks without a cache).
bw_status run_decoder(bw_stack *st, const float *h_in, int steps,
                      float *h_out, const bw_stack_trace *tr,
                      cudaStream_t cs) {
  DecoderLaunch dl{};
  dl.table = st->dec_table;
  dl.n_layers = st->d.n_layers;
  dl.steps = steps;
  dl.dim = st->d.dim;
  dl.ffn = st->d.ffn;
  dl.n_heads = st->d.n_heads;
  dl.n_kv = st->d.n_kv_heads;
  dl.eps = st->d.eps;
  dl.h_in = h_in;
  dl.h_out = h_out;
  dl.xch = st->dec_xch;
  dl.ctl = st->dec_ctl;
  dl.trace = tr;
  return cuda_err(launch_decoder(dl, cs));
}

void free_stack(bw_stack *st) {
  if (!st) return;
  cudaFree(st->dec_table);
  cudaFree(st->dec_xch);
  cudaFree(st->dec_ctl);
  for (int b = 0; b < st->n_graphs; ++b) cudaGraphExecDestroy(st->exec[b]);
  cudaFree(st->h);
  cudaFree(st->attn);
  cudaFree(st->gated);
  cudaFree(st->part);
  cudaFree(st->qkv);
  cudaFree(st->o);
  cudaFree(st->gu);
  cudaFree(st->dn);
  cudaFree(st->kc);
  cudaFree(st->vc);
  cudaFree(st->pos);
  cudaFree(st->attn_ws);
  delete st;
}

bw_status stack_create(const bw_stack_desc *desc, int kv_S, float theta,
                       bw_stack **out) {
  if (!desc || !out) return BW_ERR_INVALID_ARG;
  *out = nullptr;
  const bw_stack_desc &d = *desc;
  if (d.n_layers < 1 || d.dim < 4 || d.ffn < 4 || d.n_heads < 1 ||
      d.n_kv_heads < 1 || !(d.eps >= 0.0f))
    return BW_ERR_INVALID_ARG;
  if (d.dim % d.n_heads != 0 || d.n_heads % d.n_kv_heads != 0)
    return BW_ERR_UNSUPPORTED_SHAPE;
  if (d.dim % 4 != 0 || d.ffn % 8 != 0 || d.dim > kMaxGlueK ||
      d.ffn > kMaxGlueK)
    return BW_ERR_UNSUPPORTED_SHAPE;
  if (!d.wqkv || !d.wo || !d.w13 || !d.w2 || !d.ws || !d.gammas)
    return BW_ERR_INVALID_ARG;
  for (int l = 0; l < d.n_layers; ++l) {
    if (!d.wqkv[l] || !d.wo[l] || !d.w13[l] || !d.w2[l] || !d.ws[l] ||
        !d.gammas[l])
      return BW_ERR_INVALID_ARG;
    auto a16 = [](const void *p) {
      return reinterpret_cast<uintptr_t>(p) % 16 == 0;
    };
    if (!a16(d.wqkv[l]) || !a16(d.wo[l]) || !a16(d.w13[l]) || !a16(d.w2[l]) ||
        reinterpret_cast<uintptr_t>(d.ws[l]) % 2 != 0 ||
        !a16(d.gammas[l]))
      return BW_ERR_MISALIGNED;
  }
  if (kv_S > 0) {
    bw_status ks = check_attn(d.n_heads, d.n_kv_heads, d.dim / d.n_heads, kv_S);
    if (ks != BW_OK) return ks;
    if (!(theta > 0.0f) || !(theta < 3.0e38f)) return BW_ERR_INVALID_ARG;
  } else if (kv_S < 0) {
    return BW_ERR_INVALID_ARG;
  }
  bw_stack *st = new (std::nothrow) bw_stack();
  if (!st) return BW_ERR_INVALID_ARG;
  st->d = d;
  st->wqkv.assign(d.wqkv, d.wqkv + d.n_layers);
  st->wo.assign(d.wo, d.wo + d.n_layers);
  st->w13.assign(d.w13, d.w13 + d.n_layers);
  st->w2.assign(d.w2, d.w2 + d.n_layers);
  st->ws.assign(d.ws, d.ws + d.n_layers);
  st->gammas.assign(d.gammas, d.gammas + d.n_layers);
  st->d.wqkv = st->d.wo = st->d.w13 = st->d.w2 = nullptr;
  st->d.ws = nullptr;
  st->d.gammas = nullptr;
  st->hd = d.dim / d.n_heads;
  st->qkv_n = (d.n_heads + 2 * d.n_kv_heads) * st->hd;
  st->v_off = (d.n_heads + d.n_kv_heads) * st->hd;
  st->group = d.n_heads / d.n_kv_heads;
  cudaError_t e = cudaSuccess;
  auto alloc = [&](void **p, size_t bytes) {
    if (e == cudaSuccess) e = cudaMalloc(p, bytes);
  };
  alloc(reinterpret_cast<void **>(&st->h), size_t(d.dim) * 4);
  alloc(reinterpret_cast<void **>(&st->qkv), size_t(st->qkv_n) * 2);
  alloc(reinterpret_cast<void **>(&st->o), size_t(d.dim) * 2);
  alloc(reinterpret_cast<void **>(&st->gu), size_t(2 * d.ffn) * 2);
  alloc(reinterpret_cast<void **>(&st->dn), size_t(d.dim) * 2);
  alloc(reinterpret_cast<void **>(&st->attn), size_t(d.dim) * 4);
  alloc(reinterpret_cast<void **>(&st->gated), size_t(d.ffn) * 4);
  alloc(reinterpret_cast<void **>(&st->part),
        size_t(2) * kMaxPartials * sizeof(float2));
  if (e == cudaSuccess) e = cudaMemset(st->h, 0, size_t(d.dim) * 4);
  size_t ws_bytes = 0;
  if (kv_S > 0) {
    st->kv_S = kv_S;
    st->theta = theta;
    st->kv_layer_elems = size_t(d.n_kv_heads) * kv_S * st->hd;
    const size_t cache = size_t(d.n_layers) * st->kv_layer_elems * 2;
    ws_bytes = attn_workspace_bytes(d.n_heads, d.n_kv_heads, st->hd, kv_S);
    alloc(reinterpret_cast<void **>(&st->kc), cache);
    alloc(reinterpret_cast<void **>(&st->vc), cache);
    alloc(reinterpret_cast<void **>(&st->pos), sizeof(int));
    alloc(&st->attn_ws, ws_bytes);
    if (e == cudaSuccess) e = cudaMemset(st->kc, 0, cache);
    if (e == cudaSuccess) e = cudaMemset(st->vc, 0, cache);
    if (e == cudaSuccess) e = cudaMemset(st->pos, 0, sizeof(int));
    if (e == cudaSuccess) e = cudaMemset(st->attn_ws, 0, ws_bytes);
  }
  if (e != cudaSuccess) {
    free_stack(st);
    return cuda_err(e);
  }
  if (kv_S == 0 &&
      decoder_fits(d.dim, d.ffn, d.n_heads, d.n_kv_heads, d.n_layers)) {
    // One persistent kernel per call: the pointer table, the exchange
    // buffers (zeroed: epoch 0 is never used) and the control words.
    st->persistent = true;
    const unsigned int ctl0[4] = {1u, 0u, 0u, 0u};
    alloc(&st->dec_table, decoder_table_bytes(d.n_layers));
    alloc(&st->dec_xch, decoder_xch_bytes(d.dim, d.ffn));
    alloc(reinterpret_cast<void **>(&st->dec_ctl), sizeof(ctl0));
    if (e == cudaSuccess)
      e = decoder_upload_table(st->dec_table, d.n_layers, st->wqkv.data(),
                               st->wo.data(), st->w13.data(), st->w2.data(),
                               st->ws.data(), st->gammas.data());
    if (e == cudaSuccess)
      e = cudaMemset(st->dec_xch, 0, decoder_xch_bytes(d.dim, d.ffn));
    if (e == cudaSuccess)
      e = cudaMemcpy(st->dec_ctl, ctl0, sizeof(ctl0), cudaMemcpyHostToDevice);
    if (e != cudaSuccess) {
      free_stack(st);
      return cuda_err(e);
    }
    // One step on zero input performs every one-time set-up.
    bw_status bs = run_decoder(st, st->h, 1, st->attn, nullptr, nullptr);
    if (bs == BW_OK) bs = cuda_err(cudaDeviceSynchronize());
    if (bs != BW_OK) {
      free_stack(st);
      return bs;
    }
    *out = st;
    return BW_OK;
  }
  // Capture one decode step as a graph on a private stream (after one eager
  // run on zero input, which also performs every one-time set-up); with a
  // cache, one graph per context bucket (up to 128 and 1024 positions, then
  // any), so that short contexts run attention launches of fewer, smaller
  // CTAs.
  int lens[bw_stack::kMaxGraphs];
  int n_lens = 0;
  if (kv_S > 0)
    for (int b : kStackBuckets)
      if (b < kv_S) lens[n_lens++] = b;
  lens[n_lens++] = 0;
  cudaStream_t cap = nullptr;
  e = cudaStreamCreateWithFlags(&cap, cudaStreamNonBlocking);
  bw_status bs = e == cudaSuccess ? run_step(st, cap, nullptr, 0) : cuda_err(e);
  if (bs == BW_OK) e = cudaStreamSynchronize(cap);
  for (int b = 0; b < n_lens && bs == BW_OK && e == cudaSuccess; ++b) {
    cudaGraph_t graph = nullptr;
    bool ok = false;
    if (cudaStreamBeginCapture(cap, cudaStreamCaptureModeRelaxed) ==
        cudaSuccess) {
      bw_status rs = run_step(st, cap, nullptr, lens[b]);
      cudaError_t ee = cudaStreamEndCapture(cap, &graph);
      ok = rs == BW_OK && ee == cudaSuccess &&
           cudaGraphInstantiate(&st->exec[st->n_graphs], graph, 0) ==
               cudaSuccess;
      if (graph) cudaGraphDestroy(graph);
    }
    cudaGetLastError();  // a failed capture leaves eager launches
    if (!ok) break;
    st->graph_len[st->n_graphs++] = lens[b];
  }
  // Without every graph the steps run eagerly (still sized per bucket).
  if (st->n_graphs != n_lens) {
    for (int b = 0; b < st->n_graphs; ++b) cudaGraphExecDestroy(st->exec[b]);
    st->n_graphs = 0;
  }
  if (cap) cudaStreamDestroy(cap);
  if (bs != BW_OK) {
    free_stack(st);
    return bs;
  }
  if (kv_S > 0) {
    // The set-up step advanced the position and wrote row 0: start the
    // sequence at position 0 (rows at and past the position are never read).
    e = cudaMemset(st->pos, 0, sizeof(int));
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    if (e != cudaSuccess) {
      free_stack(st);
      return cuda_err(e);
    }
  }
  *out = st;
  return BW_OK;
}

}  // namespace

extern "C" {

bw_status bw_stack_create(const bw_stack_desc *desc, bw_stack **out) {
  return stack_create(desc, 0, 0.0f, out);
}

bw_status bw_stack_create_kv(const bw_stack_desc *desc, int max_positions,
                             float theta, bw_stack **out) {
  if (max_positions < 1) return BW_ERR_INVALID_ARG;
  return stack_create(desc, max_positions, theta, out);
}

bw_status bw_stack_read_kv(const bw_stack *st, int layer, bw_bf16 *k_out,
                           bw_bf16 *v_out, bw_stream_t stream) {
  if (!st || st->kv_S < 1 || layer < 0 || layer >= st->d.n_layers ||
      !k_out || !v_out)
    return BW_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(k_out) % 2 != 0 ||
      reinterpret_cast<uintptr_t>(v_out) % 2 != 0)
    return BW_ERR_MISALIGNED;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  const size_t bytes = st->kv_layer_elems * 2;
  const size_t off = size_t(layer) * st->kv_layer_elems;
  BW_TRY_CUDA(cudaMemcpyAsync(k_out, st->kc + off, bytes,
                              cudaMemcpyDeviceToDevice, cs));
  BW_TRY_CUDA(cudaMemcpyAsync(v_out, st->vc + off, bytes,
                              cudaMemcpyDeviceToDevice, cs));
  return BW_OK;
}

bw_status bw_stack_reset_kv(bw_stack *st, bw_stream_t stream) {
  if (!st || st->kv_S < 1) return BW_ERR_INVALID_ARG;
  BW_TRY_CUDA(cudaMemsetAsync(st->pos, 0, sizeof(int),
                              reinterpret_cast<cudaStream_t>(stream)));
  st->host_pos = 0;
  return BW_OK;
}

bw_status bw_layer_stack(bw_stack *st, const float *h_in, int steps,
                         float *h_out, const bw_stack_trace *trace,
                         bw_stream_t stream) {
  if (!st || !h_in || !h_out || steps < 1) return BW_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(h_in) % 4 != 0 ||
      reinterpret_cast<uintptr_t>(h_out) % 4 != 0)
    return BW_ERR_MISALIGNED;
  if (trace && (trace->layer < 0 || trace->layer >= st->d.n_layers))
    return BW_ERR_INVALID_ARG;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  if (st->persistent) return run_decoder(st, h_in, steps, h_out, trace, cs);
  const size_t row = size_t(st->d.dim) * 4;
  for (int t = 0; t < steps; ++t) {
    // the step's bucket: the first whose contexts include this token's
    int len = 0;
    int b = 0;
    if (st->kv_S > 0) {
      const long long want = st->host_pos + 1;
      for (int lb : kStackBuckets)
        if (lb < st->kv_S && want <= lb) {
          len = lb;
          break;
        }
      while (b + 1 < st->n_graphs && st->graph_len[b] != len) ++b;
    }
    BW_TRY_CUDA(cudaMemcpyAsync(st->h, h_in + size_t(t) * st->d.dim, row,
                                cudaMemcpyDeviceToDevice, cs));
    if ((trace && t == steps - 1) || st->n_graphs == 0)
      BW_TRY(run_step(st, cs, t == steps - 1 ? trace : nullptr, len));
    else
      BW_TRY_CUDA(cudaGraphLaunch(st->exec[b], cs));
    BW_TRY_CUDA(cudaMemcpyAsync(h_out + size_t(t) * st->d.dim, st->h, row,
                                cudaMemcpyDeviceToDevice, cs));
    ++st->host_pos;
  }
  return BW_OK;
}

void bw_stack_destroy(bw_stack *st) { free_stack(st); }

}  // extern "C"
