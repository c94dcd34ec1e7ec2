// bw_gemv.cu -- W2A8 ternary GEMV on CUDA cores for sm_103a.
//
// Computes acc[m][n] = sum_k w[n][k] * x[m][k] exactly in int32 and either
// stores acc or the bf16 epilogue y = bf16((acc / s[m]) * ws[seg(n)]).
// Source: "BitNet GPU 推理框架：从零构建 W2A8 的 2-bit 大模型 CUDA GEMV 内核",
// §5.2 (2-bit decode into int8 lanes), §5.3 (dp4a dot product, shuffle
// reduction, scale epilogue), §4.2 (one weight scale per sub-projection).
//
// Design (differs from the page's sm_80 kernel, which decodes each code to a
// signed int8 with lop3 + a byte-wise subtract):
//  * Codes stay unsigned, c = w + 1 in {0,1,2}.  sum_k w x = sum_k c x - sum_k x,
//    and sum_k x is computed once per lane, so a decoded operand costs one
//    AND: slot i of a 32-bit word is masked in place (c << 2i per byte) and fed
//    to an unsigned-by-signed dp4a; the factor 4^i is removed once at the end
//    ((((a3 >> 2) + a2) >> 2) + a1) >> 2) + a0, exact because a_i is a multiple
//    of 4^i.  One LOP3 + one IDP4A per four weights.
//  * Lane (q, r) of a warp handles row r of an 8-row group and chunk q of a
//    quad of 16-byte chunks, so one warp load is one contiguous 512-byte run
//    of the device layout (128-bit loads, L1 bypassed: every byte is used by
//    exactly one lane).
//  * A lane keeps the int8 activations of its chunks in registers for the
//    whole CTA, so no shared-memory traffic sits on the weight stream.
//  * Partial sums: 2 shuffle rounds across the 4 chunk lanes of a row, then a
//    fixed-order sum over warps in shared memory (integer: order-free).
#include "bw_internal.cuh"

namespace bw {
namespace {

// d = c + sum_b a.u8[b] * b.s8[b]
__device__ __forceinline__ int dp4a_us(uint32_t a, uint32_t b, int c) {
  int d;
  asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

// 16-byte load of streamed weights: read-only path, not kept in L1.
__device__ __forceinline__ uint4 ld_weights16(const uint8_t *p) {
  uint4 v;
  asm("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
      : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
      : "l"(p));
  return v;
}

template <int MT, int RG, int JB, bool ACC_OUT>
__global__ void __launch_bounds__(512)
gemv_w2a8_kernel(const GemvArgs a) {
  extern __shared__ int red[];  // [warps][MT][RG * 8]
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int warps = blockDim.x >> 5;
  const int q = lane >> 3;  // chunk inside the quad
  const int r = lane & 7;   // row inside the group
  const int g0 = blockIdx.x * RG;

  int acc[MT][RG][4];
  int sx[MT];
#pragma unroll
  for (int m = 0; m < MT; ++m) {
    sx[m] = 0;
#pragma unroll
    for (int g = 0; g < RG; ++g)
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[m][g][i] = 0;
  }

  for (int pass = 0; pass < a.passes; ++pass) {
    int chunk[JB];
    bool live[JB];
#pragma unroll
    for (int jb = 0; jb < JB; ++jb) {
      chunk[jb] = ((pass * warps + warp) * JB + jb) * 4 + q;
      live[jb] = chunk[jb] < a.chunks;
    }

    // Weights first: they do not depend on anything else.
    uint4 wv[RG][JB];
#pragma unroll
    for (int g = 0; g < RG; ++g) {
#pragma unroll
      for (int jb = 0; jb < JB; ++jb) {
        const int grp = g0 + g;
        if (live[jb] && grp < a.n_groups) {
          const size_t off =
              (size_t(grp) * a.chunks + chunk[jb]) * kGroupChunkBytes +
              r * kChunkBytes;
          wv[g][jb] = ld_weights16(a.w + off);
        } else {
          wv[g][jb] = make_uint4(0u, 0u, 0u, 0u);
        }
      }
    }

    // Activations of this lane's chunks (zero beyond K).
    uint32_t xr[MT][JB][16];
#pragma unroll
    for (int m = 0; m < MT; ++m) {
      const int8_t *xrow = a.x + size_t(m) * a.x_ld;
#pragma unroll
      for (int jb = 0; jb < JB; ++jb) {
        const int k0 = chunk[jb] * kChunkWeights;
        if (a.vec_x) {
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            uint4 v = make_uint4(0u, 0u, 0u, 0u);
            if (live[jb] && k0 + 16 * u < a.K)
              v = __ldg(reinterpret_cast<const uint4 *>(xrow + k0 + 16 * u));
            xr[m][jb][4 * u + 0] = v.x;
            xr[m][jb][4 * u + 1] = v.y;
            xr[m][jb][4 * u + 2] = v.z;
            xr[m][jb][4 * u + 3] = v.w;
          }
        } else {
#pragma unroll
          for (int u = 0; u < 16; ++u) {
            uint32_t v = 0u;
            if (live[jb] && k0 + 4 * u < a.K)
              v = __ldg(reinterpret_cast<const unsigned int *>(xrow + k0 +
                                                               4 * u));
            xr[m][jb][u] = v;
          }
        }
#pragma unroll
        for (int u = 0; u < 16; ++u)
          sx[m] = dp4a_us(0x01010101u, xr[m][jb][u], sx[m]);
      }
    }

    // Word t of a chunk holds k in [16t, 16t+16); slot i (bits 2i of each
    // byte) holds k = 16t + 4i + byte, which pairs with activation word 4t+i.
#pragma unroll
    for (int g = 0; g < RG; ++g) {
#pragma unroll
      for (int jb = 0; jb < JB; ++jb) {
        const uint32_t wd[4] = {wv[g][jb].x, wv[g][jb].y, wv[g][jb].z,
                                wv[g][jb].w};
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          const uint32_t c0 = wd[t] & 0x03030303u;
          const uint32_t c1 = wd[t] & 0x0c0c0c0cu;
          const uint32_t c2 = wd[t] & 0x30303030u;
          const uint32_t c3 = wd[t] & 0xc0c0c0c0u;
#pragma unroll
          for (int m = 0; m < MT; ++m) {
            acc[m][g][0] = dp4a_us(c0, xr[m][jb][4 * t + 0], acc[m][g][0]);
            acc[m][g][1] = dp4a_us(c1, xr[m][jb][4 * t + 1], acc[m][g][1]);
            acc[m][g][2] = dp4a_us(c2, xr[m][jb][4 * t + 2], acc[m][g][2]);
            acc[m][g][3] = dp4a_us(c3, xr[m][jb][4 * t + 3], acc[m][g][3]);
          }
        }
      }
    }
  }

  // Remove the slot scales and the code offset, then reduce.
#pragma unroll
  for (int m = 0; m < MT; ++m) {
#pragma unroll
    for (int g = 0; g < RG; ++g) {
      int p = ((((acc[m][g][3] >> 2) + acc[m][g][2]) >> 2) + acc[m][g][1]) >> 2;
      p += acc[m][g][0] - sx[m];
      p += __shfl_xor_sync(0xffffffffu, p, 8);
      p += __shfl_xor_sync(0xffffffffu, p, 16);
      if (q == 0) red[(warp * MT + m) * (RG * 8) + g * 8 + r] = p;
    }
  }
  __syncthreads();

  constexpr int kOuts = MT * RG * 8;
  for (int t = threadIdx.x; t < kOuts; t += blockDim.x) {
    const int m = t / (RG * 8);
    const int rr = t % (RG * 8);
    int total = 0;
    for (int w = 0; w < warps; ++w) total += red[(w * MT + m) * (RG * 8) + rr];
    const int n = g0 * 8 + rr;
    if (n >= a.N) continue;
    if (ACC_OUT) {
      static_cast<int *>(a.out)[size_t(m) * a.out_ld + n] = total;
    } else {
      int seg = 0;  // unrolled over the fixed maximum: no local-memory copy
#pragma unroll
      for (int i = 1; i < BW_MAX_WS; ++i)
        if (i < a.seg.n_ws && n >= a.seg.bounds[i]) seg = i;
      const float scaled = static_cast<float>(total) / a.s[m];
      const float v = scaled * __bfloat162float(a.ws[seg]);
      static_cast<__nv_bfloat16 *>(a.out)[size_t(m) * a.out_ld + n] =
          __float2bfloat16_rn(v);
    }
  }
}

template <int MT, int RG, int JB>
cudaError_t launch_tmpl(const GemvPlan &p, const GemvArgs &a, bool acc_out,
                        cudaStream_t stream) {
  const size_t smem = size_t(p.warps) * MT * RG * 8 * sizeof(int);
  if (acc_out)
    gemv_w2a8_kernel<MT, RG, JB, true>
        <<<p.grid, p.warps * 32, smem, stream>>>(a);
  else
    gemv_w2a8_kernel<MT, RG, JB, false>
        <<<p.grid, p.warps * 32, smem, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace

GemvPlan plan_gemv(int mt, int N, int K, int num_sms) {
  GemvPlan p{};
  p.mt = mt;
  const int chunks = chunks_per_row(K);
  const int quads = (chunks + 3) / 4;
  const int max_jb = mt == 1 ? 4 : (mt == 2 ? 2 : 1);
  constexpr int kMaxWarps = 16;

  // Chunk quads per warp: the fewest idle quads with at most 16 warps.
  p.jb = 0;
  int best_waste = 1 << 30;
  for (int jb = 1; jb <= max_jb; ++jb) {
    const int w = (quads + jb - 1) / jb;
    if (w > kMaxWarps) continue;
    const int waste = w * jb - quads;
    if (waste < best_waste) {
      best_waste = waste;
      p.jb = jb;
      p.warps = w;
    }
  }
  if (p.jb == 0) {  // K too long for one pass: 16 warps, several passes
    p.jb = max_jb;
    p.warps = kMaxWarps;
  }
  p.passes = (quads + p.warps * p.jb - 1) / (p.warps * p.jb);

  // Row groups per CTA: the largest that still gives two CTAs per SM.
  const int64_t groups = padded_rows(N) / kGroupRows;
  // (register budget: weight and activation registers grow with rg * jb)
  int max_rg = mt == 4 ? 1 : (mt == 2 ? 2 : 4);
  while (max_rg > 1 && max_rg * p.jb > 8) max_rg /= 2;
  p.rg = 1;
  for (int rg = max_rg; rg > 1; rg /= 2) {
    if ((groups + rg - 1) / rg >= 2 * int64_t(num_sms)) {
      p.rg = rg;
      break;
    }
  }
  p.grid = int((groups + p.rg - 1) / p.rg);
  return p;
}

cudaError_t launch_gemv(const GemvPlan &p, const GemvArgs &a, bool acc_out,
                        cudaStream_t stream) {
#define BW_CASE(MT_, RG_, JB_)                                   \
  if (p.mt == MT_ && p.rg == RG_ && p.jb == JB_)                 \
    return launch_tmpl<MT_, RG_, JB_>(p, a, acc_out, stream);
  BW_CASE(1, 1, 1) BW_CASE(1, 1, 2) BW_CASE(1, 1, 3) BW_CASE(1, 1, 4)
  BW_CASE(1, 2, 1) BW_CASE(1, 2, 2) BW_CASE(1, 2, 3) BW_CASE(1, 2, 4)
  BW_CASE(1, 4, 1) BW_CASE(1, 4, 2)
  BW_CASE(2, 1, 1) BW_CASE(2, 1, 2) BW_CASE(2, 2, 1) BW_CASE(2, 2, 2)
  BW_CASE(4, 1, 1)
#undef BW_CASE
  return cudaErrorInvalidConfiguration;
}

}  // namespace bw
