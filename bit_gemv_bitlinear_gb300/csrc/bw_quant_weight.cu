// bw_quant_weight.cu -- absmean ternarisation of fp32 weights into the
// canonical 2-bit codes and one bf16 scale per weight-scale segment.
//
// The checkpoint conversion of "BitNet GPU 推理框架：从零构建 W2A8 的 2-bit 大模型
// CUDA GEMV 内核", §4.2: s = 1 / max(mean |W|, 1e-5), w = clamp(round(W s), -1,
// 1), ws = bf16(1 / s), one scale per projection (here per segment of rows,
// the same segments the GEMV's ws_bounds name).  The page leaves the
// precision to the framework's dtype; here: |W| summed in fp64 per segment,
// the mean (sum / count, fp64) rounded to fp32, s, W s and 1 / s in fp32,
// round to nearest even, ws rounded to nearest even bf16.  The fp64 sum is
// accumulated in a different order than a sequential sum; its rounding can
// change the fp32 mean only when the mean lies within a few fp64 rounding
// steps of an fp32 rounding boundary.
//
// Offline: two kernels (the segment sums, one fp64 atomic per block; then
// one thread per output byte), scratch from cudaMallocAsync, and the call
// synchronises its stream, like the repack.
#include <algorithm>

#include "bw_internal.cuh"

namespace bw {
namespace {

constexpr int kQwThreads = 256;
constexpr int kQwVecPerThread = 8;  // float4 per thread and pass of kernel 1

__device__ __forceinline__ double block_sum(double v, double *red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) red[warp] = v;
  __syncthreads();
  v = 0.0;
  if (warp == 0) {
    v = lane < int(blockDim.x >> 5) ? red[lane] : 0.0;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  }
  return v;  // valid in thread 0
}

// sums[i] += sum of |W| over rows [bounds[i], bounds[i+1]) (blockIdx.y = i):
// the segment is one contiguous run of float4 (K % 4 == 0, W 16-byte aligned).
__global__ void __launch_bounds__(kQwThreads)
absmean_sum_kernel(const float4 *W, int K4, WsSegments seg, double *sums) {
  __shared__ double red[kQwThreads / 32];
  const int i = blockIdx.y;
  const int64_t lo = int64_t(seg.bounds[i]) * K4;
  const int64_t hi = int64_t(seg.bounds[i + 1]) * K4;
  double acc = 0.0;
  for (int64_t v = lo + int64_t(blockIdx.x) * blockDim.x + threadIdx.x; v < hi;
       v += int64_t(gridDim.x) * blockDim.x) {
    const float4 w = __ldg(W + v);
    acc += double(fabsf(w.x)) + double(fabsf(w.y)) + double(fabsf(w.z)) +
           double(fabsf(w.w));
  }
  acc = block_sum(acc, red);
  if (threadIdx.x == 0) atomicAdd(&sums[i], acc);
}

__device__ __forceinline__ float segment_scale(const double *sums, int i,
                                               const WsSegments &seg, int K) {
  const double count = double(seg.bounds[i + 1] - seg.bounds[i]) * double(K);
  float mean = float(sums[i] / count);
  mean = fmaxf(mean, 1e-5f);
  return 1.0f / mean;
}

__device__ __forceinline__ uint32_t ternary_code(float w, float s) {
  float v = rintf(__fmul_rn(w, s));  // nearest, ties to even
  v = fminf(fmaxf(v, -1.0f), 1.0f);
  return uint32_t(int(v) + 1);
}

// One thread per canonical byte (row n, weights 4j .. 4j+3); element 4j+t
// at bits 2t.  Block 0 also writes the bf16 scales.
__global__ void __launch_bounds__(kQwThreads)
ternarise_kernel(const float4 *W, int N, int K4, WsSegments seg,
                 const double *sums, uint8_t *canon, __nv_bfloat16 *ws) {
  if (blockIdx.x == 0 && int(threadIdx.x) < seg.n_ws) {
    const float s = segment_scale(sums, threadIdx.x, seg, 4 * K4);
    ws[threadIdx.x] = __float2bfloat16_rn(1.0f / s);
  }
  const int64_t total = int64_t(N) * K4;
  for (int64_t b = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; b < total;
       b += int64_t(gridDim.x) * blockDim.x) {
    const int n = int(b / K4);
    int sg = 0;
#pragma unroll
    for (int i = 1; i < BW_MAX_WS; ++i)
      if (i < seg.n_ws && n >= seg.bounds[i]) sg = i;
    const float s = segment_scale(sums, sg, seg, 4 * K4);
    const float4 w = __ldg(W + b);
    canon[b] = uint8_t(ternary_code(w.x, s) | (ternary_code(w.y, s) << 2) |
                       (ternary_code(w.z, s) << 4) |
                       (ternary_code(w.w, s) << 6));
  }
}

}  // namespace

cudaError_t launch_quant_weight(const float *W, int N, int K,
                                const WsSegments &seg, uint8_t *canon,
                                __nv_bfloat16 *ws, cudaStream_t stream) {
  double *sums = nullptr;
  cudaError_t e = cudaMallocAsync(reinterpret_cast<void **>(&sums),
                                  sizeof(double) * BW_MAX_WS, stream);
  if (e != cudaSuccess) return e;
  e = cudaMemsetAsync(sums, 0, sizeof(double) * BW_MAX_WS, stream);
  const int K4 = K / 4;
  const float4 *W4 = reinterpret_cast<const float4 *>(W);
  if (e == cudaSuccess) {
    // blocks per segment: enough for the largest, at most 1024
    int64_t most = 0;
    for (int i = 0; i < seg.n_ws; ++i)
      most = std::max<int64_t>(most, int64_t(seg.bounds[i + 1] - seg.bounds[i]) * K4);
    const int64_t per_block = int64_t(kQwThreads) * kQwVecPerThread;
    const unsigned bx = unsigned(std::min<int64_t>(1024, (most + per_block - 1) / per_block));
    absmean_sum_kernel<<<dim3(bx, unsigned(seg.n_ws)), kQwThreads, 0, stream>>>(
        W4, K4, seg, sums);
    e = cudaGetLastError();
  }
  if (e == cudaSuccess) {
    const int64_t total = int64_t(N) * K4;
    const unsigned blocks = unsigned(std::min<int64_t>(
        8 * 1024, std::max<int64_t>(1, (total + kQwThreads - 1) / kQwThreads)));
    ternarise_kernel<<<blocks, kQwThreads, 0, stream>>>(W4, N, K4, seg, sums,
                                                         canon, ws);
    e = cudaGetLastError();
  }
  const cudaError_t ef = cudaFreeAsync(sums, stream);
  if (e == cudaSuccess) e = ef;
  if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
  return e;
}

}  // namespace bw
