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
// One layer, M = 1:
//   h <- h + down(prev layer)            (fused into the first glue kernel)
//   (q, s) <- quant(rmsnorm(h) * g_attn)              -> qkv = W2A8(wqkv)
//   (q, s) <- quant(rmsnorm(attn(qkv)) * g_attn_sub)  -> o   = W2A8(wo)
//   h <- h + o; (q, s) <- quant(rmsnorm(h) * g_ffn)   -> gu  = W2A8(w13)
//   (q, s) <- quant(rmsnorm(relu(gate)^2 up) * g_sub) -> down = W2A8(w2)
// attn() is attention over a one-token context: the softmax of one score is
// 1, so query head h returns the value vector of KV head h / (heads / kv).
//
// Each glue step is one single-CTA kernel (1024 threads, up to 8 values
// per thread kept in registers between the two reductions); the GEMVs are
// the TMA-streamed kernels.  All launches use programmatic dependent
// launch, and one decode step is captured once as a CUDA graph.
#include <cstdlib>
#include <new>
#include <vector>

#include "bw_internal.cuh"

namespace bw {
namespace {

constexpr int kGlueThreads = 1024;
constexpr int kMaxGlueK = 8 * kGlueThreads;

__device__ __forceinline__ void pdl_enter() {
  asm volatile("griddepcontrol.launch_dependents;");
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

// Deterministic block reductions (fixed shuffle tree, then warp 0).
__device__ __forceinline__ float block_sum(float v, float *scratch) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  __syncthreads();
  if ((threadIdx.x & 31) == 0) scratch[threadIdx.x >> 5] = v;
  __syncthreads();
  float t = 0.0f;
  for (int w = 0; w < int(blockDim.x >> 5); ++w) t += scratch[w];
  return t;
}

__device__ __forceinline__ float block_max(float v, float *scratch) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1)
    v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  __syncthreads();
  if ((threadIdx.x & 31) == 0) scratch[threadIdx.x >> 5] = v;
  __syncthreads();
  float t = 0.0f;
  for (int w = 0; w < int(blockDim.x >> 5); ++w) t = fmaxf(t, scratch[w]);
  return t;
}

__device__ __forceinline__ int8_t quant1(float x, float scale) {
  return static_cast<int8_t>(
      static_cast<int>(fminf(fmaxf(rintf(x * scale), -128.0f), 127.0f)));
}

// Element loaders of the three glue steps.
struct ResidualLoad {  // x[k] (+ bf16 add[k]), fp32
  const float *x;
  const __nv_bfloat16 *add;
  __device__ float operator()(int k) const {
    float v = x[k];
    if (add) v = v + __bfloat162float(add[k]);
    return v;
  }
};

struct AttnLoad {  // value head of query head k / hd
  const __nv_bfloat16 *qkv;
  int v_off, hd, group;
  __device__ float operator()(int k) const {
    const int h = k / hd;
    return __bfloat162float(qkv[v_off + (h / group) * hd + (k - h * hd)]);
  }
};

struct Relu2Load {  // relu(gate)^2 * up, exact in fp32 for bf16 inputs
  const __nv_bfloat16 *gu;
  int F;
  __device__ float operator()(int k) const {
    const float g = __bfloat162float(gu[k]);
    const float u = __bfloat162float(gu[F + k]);
    const float r = g > 0.0f ? g : 0.0f;
    return r * r * u;
  }
};

// v = load(k); optionally h_out[k] = v; then
// n = (v * (1 / sqrt(mean(v^2) + eps))) * gamma, s = 127 / max(absmax n, 1e-5),
// q = clamp(rint(n * s), -128, 127).  One CTA, fp32.
template <class Load, int V>
__global__ void __launch_bounds__(kGlueThreads)
norm_quant_kernel(Load load, const float *__restrict__ gamma, int K,
                  float eps, float *h_out, int8_t *__restrict__ q,
                  float *__restrict__ s) {
  __shared__ float scratch[32];
  pdl_enter();
  float v[V];
  float ss = 0.0f;
#pragma unroll
  for (int i = 0; i < V; ++i) {
    const int k = threadIdx.x + i * kGlueThreads;
    v[i] = k < K ? load(k) : 0.0f;
    ss += v[i] * v[i];
  }
  if (h_out) {
#pragma unroll
    for (int i = 0; i < V; ++i) {
      const int k = threadIdx.x + i * kGlueThreads;
      if (k < K) h_out[k] = v[i];
    }
  }
  ss = block_sum(ss, scratch);
  const float r = 1.0f / sqrtf(ss / static_cast<float>(K) + eps);
  float amax = 0.0f;
#pragma unroll
  for (int i = 0; i < V; ++i) {
    const int k = threadIdx.x + i * kGlueThreads;
    if (k < K) {
      v[i] = (v[i] * r) * gamma[k];
      amax = fmaxf(amax, fabsf(v[i]));
    }
  }
  amax = block_max(amax, scratch);
  const float scale = 127.0f / fmaxf(amax, 1e-5f);
  if (threadIdx.x == 0) *s = scale;
#pragma unroll
  for (int i = 0; i < V; ++i) {
    const int k = threadIdx.x + i * kGlueThreads;
    if (k < K) q[k] = quant1(v[i], scale);
  }
}

// h += down (the residual of the last layer).
__global__ void __launch_bounds__(kGlueThreads)
residual_kernel(float *h, const __nv_bfloat16 *down, int n) {
  pdl_enter();
  for (int k = threadIdx.x; k < n; k += blockDim.x)
    h[k] = h[k] + __bfloat162float(down[k]);
}

cudaLaunchConfig_t glue_config(cudaStream_t stream, cudaLaunchAttribute *attr) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(1);
  cfg.blockDim = dim3(kGlueThreads);
  cfg.stream = stream;
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cfg;
}

template <class Load>
cudaError_t launch_norm_quant(const Load &load, const float *gamma, int K,
                              float eps, float *h_out, int8_t *q, float *s,
                              cudaStream_t stream) {
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = glue_config(stream, attr);
  const int v = (K + kGlueThreads - 1) / kGlueThreads;
  if (v <= 1)
    return cudaLaunchKernelEx(&cfg, norm_quant_kernel<Load, 1>, load, gamma,
                              K, eps, h_out, q, s);
  if (v <= 2)
    return cudaLaunchKernelEx(&cfg, norm_quant_kernel<Load, 2>, load, gamma,
                              K, eps, h_out, q, s);
  if (v <= 4)
    return cudaLaunchKernelEx(&cfg, norm_quant_kernel<Load, 4>, load, gamma,
                              K, eps, h_out, q, s);
  return cudaLaunchKernelEx(&cfg, norm_quant_kernel<Load, 8>, load, gamma, K,
                            eps, h_out, q, s);
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
  float *h;
  int8_t *q;
  float *s;
  __nv_bfloat16 *qkv, *o, *gu, *dn;
  cudaGraphExec_t exec;
  bool have_graph;
};

namespace {

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
// input on entry and its output on exit.
bw_status run_step(bw_stack *st, cudaStream_t cs, const bw_stack_trace *tr) {
  const bw_stack_desc &d = st->d;
  const int dim = d.dim, ffn = d.ffn;
  const int b_qkv[4] = {0, d.n_heads * st->hd,
                        (d.n_heads + d.n_kv_heads) * st->hd, st->qkv_n};
  const int b_dim[2] = {0, dim};
  const int b_13[3] = {0, ffn, 2 * ffn};
  const bw_bf16 *qkv = reinterpret_cast<bw_bf16 *>(st->qkv);
  for (int l = 0; l < d.n_layers; ++l) {
    const float *g = st->gammas[l];
    const bw_bf16 *ws = st->ws[l];
    const bool rec = tr && tr->layer == l;
    // attention_norm(h + down of the previous layer)
    BW_TRY_CUDA(launch_norm_quant(
        ResidualLoad{st->h, l ? st->dn : nullptr}, g, dim, d.eps, st->h,
        st->q, st->s, cs));
    if (rec) {
      BW_TRY_CUDA(trace_copy(tr->h_in, st->h, dim * 4, cs));
      BW_TRY_CUDA(trace_copy(tr->q_attn, st->q, dim, cs));
      BW_TRY_CUDA(trace_copy(tr->s_attn, st->s, 4, cs));
    }
    BW_TRY(gemv_internal(st->q, st->wqkv[l], st->s, ws, b_qkv, 3, 1,
                         st->qkv_n, dim, reinterpret_cast<bw_bf16 *>(st->qkv),
                         cs));
    if (rec) BW_TRY_CUDA(trace_copy(tr->qkv, qkv, st->qkv_n * 2, cs));
    // attn_sub_norm(one-token attention)
    BW_TRY_CUDA(launch_norm_quant(
        AttnLoad{st->qkv, st->v_off, st->hd, st->group}, g + dim, dim, d.eps,
        nullptr, st->q, st->s, cs));
    if (rec) {
      BW_TRY_CUDA(trace_copy(tr->q_o, st->q, dim, cs));
      BW_TRY_CUDA(trace_copy(tr->s_o, st->s, 4, cs));
    }
    BW_TRY(gemv_internal(st->q, st->wo[l], st->s, ws + 3, b_dim, 1, 1, dim,
                         dim, reinterpret_cast<bw_bf16 *>(st->o), cs));
    if (rec) BW_TRY_CUDA(trace_copy(tr->o, st->o, dim * 2, cs));
    // ffn_norm(h + o)
    BW_TRY_CUDA(launch_norm_quant(ResidualLoad{st->h, st->o}, g + 2 * dim,
                                  dim, d.eps, st->h, st->q, st->s, cs));
    if (rec) {
      BW_TRY_CUDA(trace_copy(tr->h_mid, st->h, dim * 4, cs));
      BW_TRY_CUDA(trace_copy(tr->q_ffn, st->q, dim, cs));
      BW_TRY_CUDA(trace_copy(tr->s_ffn, st->s, 4, cs));
    }
    BW_TRY(gemv_internal(st->q, st->w13[l], st->s, ws + 4, b_13, 2, 1,
                         2 * ffn, dim, reinterpret_cast<bw_bf16 *>(st->gu),
                         cs));
    if (rec) BW_TRY_CUDA(trace_copy(tr->gu, st->gu, 2 * ffn * 2, cs));
    // ffn_sub_norm(relu(gate)^2 * up)
    BW_TRY_CUDA(launch_norm_quant(Relu2Load{st->gu, ffn}, g + 3 * dim, ffn,
                                  d.eps, nullptr, st->q, st->s, cs));
    if (rec) {
      BW_TRY_CUDA(trace_copy(tr->q_down, st->q, ffn, cs));
      BW_TRY_CUDA(trace_copy(tr->s_down, st->s, 4, cs));
    }
    BW_TRY(gemv_internal(st->q, st->w2[l], st->s, ws + 6, b_dim, 1, 1, dim,
                         ffn, reinterpret_cast<bw_bf16 *>(st->dn), cs));
    if (rec) BW_TRY_CUDA(trace_copy(tr->down, st->dn, dim * 2, cs));
  }
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = glue_config(cs, attr);
  BW_TRY_CUDA(cudaLaunchKernelEx(&cfg, residual_kernel, st->h,
                                 static_cast<const __nv_bfloat16 *>(st->dn),
                                 dim));
  return BW_OK;
}

void free_stack(bw_stack *st) {
  if (!st) return;
  if (st->have_graph) cudaGraphExecDestroy(st->exec);
  cudaFree(st->h);
  cudaFree(st->q);
  cudaFree(st->s);
  cudaFree(st->qkv);
  cudaFree(st->o);
  cudaFree(st->gu);
  cudaFree(st->dn);
  delete st;
}

}  // namespace

extern "C" {

bw_status bw_stack_create(const bw_stack_desc *desc, bw_stack **out) {
  if (!desc || !out) return BW_ERR_INVALID_ARG;
  *out = nullptr;
  const bw_stack_desc &d = *desc;
  if (d.n_layers < 1 || d.dim < 4 || d.ffn < 4 || d.n_heads < 1 ||
      d.n_kv_heads < 1 || !(d.eps >= 0.0f))
    return BW_ERR_INVALID_ARG;
  if (d.dim % d.n_heads != 0 || d.n_heads % d.n_kv_heads != 0)
    return BW_ERR_UNSUPPORTED_SHAPE;
  if (d.dim % 4 != 0 || d.ffn % 4 != 0 || d.dim > kMaxGlueK ||
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
        reinterpret_cast<uintptr_t>(d.gammas[l]) % 4 != 0)
      return BW_ERR_MISALIGNED;
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
  const int qmax = d.dim > d.ffn ? d.dim : d.ffn;
  cudaError_t e = cudaSuccess;
  auto alloc = [&](void **p, size_t bytes) {
    if (e == cudaSuccess) e = cudaMalloc(p, bytes);
  };
  alloc(reinterpret_cast<void **>(&st->h), size_t(d.dim) * 4);
  alloc(reinterpret_cast<void **>(&st->q), size_t(qmax));
  alloc(reinterpret_cast<void **>(&st->s), 16);
  alloc(reinterpret_cast<void **>(&st->qkv), size_t(st->qkv_n) * 2);
  alloc(reinterpret_cast<void **>(&st->o), size_t(d.dim) * 2);
  alloc(reinterpret_cast<void **>(&st->gu), size_t(2 * d.ffn) * 2);
  alloc(reinterpret_cast<void **>(&st->dn), size_t(d.dim) * 2);
  if (e == cudaSuccess) e = cudaMemset(st->h, 0, size_t(d.dim) * 4);
  if (e != cudaSuccess) {
    free_stack(st);
    return cuda_err(e);
  }
  // Capture one decode step as a graph on a private stream (after one eager
  // run on zero input, which also performs every one-time set-up).
  cudaStream_t cap = nullptr;
  e = cudaStreamCreateWithFlags(&cap, cudaStreamNonBlocking);
  bw_status bs = e == cudaSuccess ? run_step(st, cap, nullptr) : cuda_err(e);
  if (bs == BW_OK) e = cudaStreamSynchronize(cap);
  if (bs == BW_OK && e == cudaSuccess) {
    cudaGraph_t graph = nullptr;
    e = cudaStreamBeginCapture(cap, cudaStreamCaptureModeRelaxed);
    if (e == cudaSuccess) {
      bw_status rs = run_step(st, cap, nullptr);
      cudaError_t ee = cudaStreamEndCapture(cap, &graph);
      if (rs == BW_OK && ee == cudaSuccess &&
          cudaGraphInstantiate(&st->exec, graph, 0) == cudaSuccess)
        st->have_graph = true;
      if (graph) cudaGraphDestroy(graph);
    }
    cudaGetLastError();  // a failed capture leaves eager launches
  }
  if (cap) cudaStreamDestroy(cap);
  if (bs != BW_OK) {
    free_stack(st);
    return bs;
  }
  *out = st;
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
  const size_t row = size_t(st->d.dim) * 4;
  for (int t = 0; t < steps; ++t) {
    BW_TRY_CUDA(cudaMemcpyAsync(st->h, h_in + size_t(t) * st->d.dim, row,
                                cudaMemcpyDeviceToDevice, cs));
    if ((trace && t == steps - 1) || !st->have_graph)
      BW_TRY(run_step(st, cs, t == steps - 1 ? trace : nullptr));
    else
      BW_TRY_CUDA(cudaGraphLaunch(st->exec, cs));
    BW_TRY_CUDA(cudaMemcpyAsync(h_out + size_t(t) * st->d.dim, st->h, row,
                                cudaMemcpyDeviceToDevice, cs));
  }
  return BW_OK;
}

void bw_stack_destroy(bw_stack *st) { free_stack(st); }

}  // extern "C"
