// bw_gemv_mma.cu -- the W2A8 product for batched activations (M >= 8) on
// tensor cores.
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
// gives the exact integer in any order.
//
// Design:
//  * mma.sync m16n8k16 (fp16 in, fp32 accumulate).  A = 16 weight rows x 16
//    k, B = 16 k x 8 tokens, D = 16 rows x 8 tokens.  A warp owns 16 rows
//    (two 8-row groups of the device layout) and all tokens of the tile, so
//    every A fragment is decoded once and used for M/8 MMAs.
//  * A fragment straight from the packed words in registers: thread (g, t)
//    needs codes (row g | g+8, k = 2t, 2t+1, 2t+8, 2t+9) of a 16-k word;
//    with the word interleave of the layout these sit in byte pair 2(t&1)
//    at slots t/2 and t/2 + 2, so one shift, two masks, a byte permute that
//    builds fp16(1024 + c) and one fp16 subtract of 1025 give two weights
//    c - 1 per 32-bit register.
//  * Activations: the CTA converts each K slice of x (int8) to fp16 once
//    (x + 128 as the low byte of fp16(1024 + u), minus 1152) into a padded
//    shared tile, double-buffered; B fragments are conflict-free 32-bit
//    shared loads.
//  * The CTA's weight rows are one contiguous run (8 row groups): one bulk
//    L2 prefetch before the programmatic-launch dependency wait, then
//    128-bit loads, one slice ahead.
#include <cuda_fp16.h>

#include "bw_internal.cuh"

namespace bw {
namespace {

constexpr int kMmaWarps = 4;         // 4 warps x 16 rows = 64 rows per CTA
constexpr int kRowsPerCta = 16 * kMmaWarps;
constexpr int kSlice = 256;          // k per staged activation slice
constexpr int kXStride = kSlice + 8; // halves per staged row (+16 bytes)

__device__ __forceinline__ void pdl_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;");
}
__device__ __forceinline__ void prefetch_l2(const void *p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ uint4 ld_weights16(const uint8_t *p) {
  uint4 v;
  asm("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
      : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
      : "l"(p));
  return v;
}

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

// Two codes (bits 0-1 of bytes 0 and 1 of m) -> fp16x2 of (code - 1).
__device__ __forceinline__ uint32_t decode_pair(uint32_t m) {
  // bytes [c0, 0x64, c1, 0x64] = fp16(1024 + c0), fp16(1024 + c1)
  return hsub2(prmt(m, 0x64646464u, 0x4140u), 0x64016401u);  // - 1025
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

// Stage activation rows [0, 8 NT) x k in [k0, k0 + kSlice) as fp16 (zero
// beyond K and beyond the tile's rows).
template <int NT>
__device__ __forceinline__ void stage_x(const GemvArgs &a, int rows, int k0,
                                        __half *xs) {
  constexpr int MT = 8 * NT;
  constexpr int kWords = kSlice / 4;
  for (int i = threadIdx.x; i < MT * kWords; i += blockDim.x) {
    const int m = i / kWords;
    const int kk = (i % kWords) * 4;
    const int k = k0 + kk;
    uint32_t v = 0u;
    if (m < rows && k < a.K)
      v = __ldg(reinterpret_cast<const unsigned int *>(a.x + size_t(m) * a.x_ld +
                                                       k));
    *reinterpret_cast<uint2 *>(xs + m * kXStride + kk) = int8x4_to_f16(v);
  }
}

template <int NT, bool ACC_OUT>
__global__ void __launch_bounds__(kMmaWarps * 32)
gemv_w2a8_mma_kernel(const GemvArgs a, int rows) {
  constexpr int MT = 8 * NT;
  extern __shared__ __align__(16) uint8_t smem[];
  __half *xs = reinterpret_cast<__half *>(smem);  // [2][MT][kXStride]
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  const int group0 = blockIdx.x * (kRowsPerCta / kGroupRows);
  const size_t group_bytes = size_t(a.chunks) * kGroupChunkBytes;

  // The CTA's weight rows are contiguous: ask L2 for them before the wait.
  if (threadIdx.x == 0) {
    const int g_end = min(group0 + kRowsPerCta / kGroupRows, a.n_groups);
    size_t len = size_t(g_end - group0) * group_bytes;
    const uint8_t *p = a.w + size_t(group0) * group_bytes;
    for (size_t o = 0; o < len; o += 65536)
      prefetch_l2(p + o, uint32_t(min(len - o, size_t(65536))));
  }
  pdl_wait();
  pdl_trigger();

  const int ga = group0 + 2 * warp;  // groups of rows g (ga) and g + 8 (gb)
  const bool live_a = ga < a.n_groups;
  const bool live_b = ga + 1 < a.n_groups;
  const uint8_t *wa = a.w + size_t(ga) * group_bytes + g * kChunkBytes;
  const uint8_t *wb = wa + group_bytes;
  const int shift = 16 * (t & 1) + 2 * (t >> 1);

  float acc[NT][4];
#pragma unroll
  for (int j = 0; j < NT; ++j)
#pragma unroll
    for (int i = 0; i < 4; ++i) acc[j][i] = 0.0f;

  const int kpad = a.chunks * kChunkWeights;
  const int n_slices = (kpad + kSlice - 1) / kSlice;
  stage_x<NT>(a, rows, 0, xs);
  __syncthreads();

  for (int sl = 0; sl < n_slices; ++sl) {
    __half *cur = xs + (sl & 1) * (MT * kXStride);
    // Weights of this slice: 4 chunks (16 k-steps) of rows g and g + 8.
    uint4 wra[kSlice / 64], wrb[kSlice / 64];
#pragma unroll
    for (int c = 0; c < kSlice / 64; ++c) {
      const int j = sl * (kSlice / 64) + c;
      const bool live = j < a.chunks;
      wra[c] = (live && live_a) ? ld_weights16(wa + size_t(j) * kGroupChunkBytes)
                                : make_uint4(0x55555555u, 0x55555555u,
                                             0x55555555u, 0x55555555u);
      wrb[c] = (live && live_b) ? ld_weights16(wb + size_t(j) * kGroupChunkBytes)
                                : make_uint4(0x55555555u, 0x55555555u,
                                             0x55555555u, 0x55555555u);
    }
    if (sl + 1 < n_slices)
      stage_x<NT>(a, rows, (sl + 1) * kSlice,
                  xs + ((sl + 1) & 1) * (MT * kXStride));

#pragma unroll
    for (int c = 0; c < kSlice / 64; ++c) {
      const uint32_t wda[4] = {wra[c].x, wra[c].y, wra[c].z, wra[c].w};
      const uint32_t wdb[4] = {wrb[c].x, wrb[c].y, wrb[c].z, wrb[c].w};
#pragma unroll
      for (int w4 = 0; w4 < 4; ++w4) {
        const uint32_t ha = wda[w4] >> shift;
        const uint32_t hb = wdb[w4] >> shift;
        uint32_t af[4];
        af[0] = decode_pair(ha & 0x0303u);         // row g,   k 2t, 2t+1
        af[1] = decode_pair(hb & 0x0303u);         // row g+8, k 2t, 2t+1
        af[2] = decode_pair((ha >> 4) & 0x0303u);  // row g,   k 2t+8, 2t+9
        af[3] = decode_pair((hb >> 4) & 0x0303u);  // row g+8, k 2t+8, 2t+9
        const int kk = c * 64 + w4 * 16;  // k offset inside the slice
#pragma unroll
        for (int j = 0; j < NT; ++j) {
          const __half *xr = cur + (8 * j + g) * kXStride + kk + 2 * t;
          const uint32_t b0 = *reinterpret_cast<const uint32_t *>(xr);
          const uint32_t b1 = *reinterpret_cast<const uint32_t *>(xr + 8);
          mma16816(acc[j], af, b0, b1);
        }
      }
    }
    __syncthreads();
  }

  // D fragment: acc[j][0..1] = rows g, tokens 8j + 2t (+1);
  //             acc[j][2..3] = row g + 8, same tokens.
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    const int n = (ga + half) * kGroupRows + g;
    if (n >= a.N) continue;
    int seg = 0;
#pragma unroll
    for (int i = 1; i < BW_MAX_WS; ++i)
      if (i < a.seg.n_ws && n >= a.seg.bounds[i]) seg = i;
    const float wsv = ACC_OUT ? 0.0f : __bfloat162float(a.ws[seg]);
#pragma unroll
    for (int j = 0; j < NT; ++j) {
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int m = 8 * j + 2 * t + e;
        if (m >= rows) continue;
        const int total = __float2int_rn(acc[j][2 * half + e]);
        if (ACC_OUT) {
          static_cast<int *>(a.out)[size_t(m) * a.out_ld + n] = total;
        } else {
          const float scaled = static_cast<float>(total) / a.s[m];
          static_cast<__nv_bfloat16 *>(a.out)[size_t(m) * a.out_ld + n] =
              __float2bfloat16_rn(scaled * wsv);
        }
      }
    }
  }
}

template <int NT, bool ACC>
cudaError_t launch_nt(const GemvArgs &a, int rows, cudaStream_t stream) {
  const size_t smem = size_t(2) * (8 * NT) * kXStride * sizeof(__half);
  static bool configured[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!configured[dev]) {
    e = cudaFuncSetAttribute(gemv_w2a8_mma_kernel<NT, ACC>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             int(smem));
    if (e != cudaSuccess) return e;
    configured[dev] = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((a.n_groups * kGroupRows + kRowsPerCta - 1) / kRowsPerCta);
  cfg.blockDim = dim3(kMmaWarps * 32);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, gemv_w2a8_mma_kernel<NT, ACC>, a, rows);
}

}  // namespace

int mma_tile_rows(int left) {
  return left >= 64 ? 64 : (left > 32 ? 64 : (left > 16 ? 32 : (left > 8 ? 16 : 8)));
}

cudaError_t launch_gemv_mma(const GemvArgs &a, int rows, bool acc_out,
                            cudaStream_t stream) {
  const int tile = mma_tile_rows(rows);
  if (tile == 8)
    return acc_out ? launch_nt<1, true>(a, rows, stream)
                   : launch_nt<1, false>(a, rows, stream);
  if (tile == 16)
    return acc_out ? launch_nt<2, true>(a, rows, stream)
                   : launch_nt<2, false>(a, rows, stream);
  if (tile == 32)
    return acc_out ? launch_nt<4, true>(a, rows, stream)
                   : launch_nt<4, false>(a, rows, stream);
  return acc_out ? launch_nt<8, true>(a, rows, stream)
                 : launch_nt<8, false>(a, rows, stream);
}

}  // namespace bw
