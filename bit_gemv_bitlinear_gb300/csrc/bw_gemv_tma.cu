// bw_gemv_tma.cu -- the public W2A8 ternary GEMV (M < 8): the TMA-streamed
// pipe kernel of bw_pipe.cuh fed with staged int8 activations.
//
// Same product and epilogue as bw_gemv.cu (acc = sum_k w x exactly in int32,
// y = bf16((acc / s[m]) * ws[seg(n)])).  Source: "BitNet GPU 推理框架：从零构建
// W2A8 的 2-bit 大模型 CUDA GEMV 内核", §5.2 (2-bit decode), §5.3 (dp4a dot
// product, shuffle reduction, scale epilogue), §4.2 (weight-scale segments).
//
// Design for sm_103a (details in bw_pipe.cuh):
//  * The packed weights are the only large operand and each byte is used
//    once, so they are streamed HBM -> shared memory with 1-D TMA bulk copies
//    (cp.async.bulk, completion counted in bytes on an mbarrier); the bytes
//    in flight per SM are set by the shared-memory buffers, not by registers
//    or warps.
//  * A CTA owns k consecutive row groups (k as small as the resident CTAs
//    allow, so every CTA but the last has the same work); its 8 warps split
//    the CTA's chunks into 8 equal runs and each warp streams its run in
//    pieces of up to 4 KB through its own 2-slot ring, issuing its own
//    copies.  Partial row sums meet in shared memory (int32 atomics, exact in
//    any order); one epilogue per CTA scales and stores the rows.
//  * Lane (q, r): row r of the group, chunks j = q (mod 4).  One 128-bit
//    shared load gives 64 codes (a contiguous 512-byte warp access, no bank
//    conflict); the int8 activations, staged in shared memory, come as
//    four 128-bit broadcast loads per chunk.  Where each warp's run is at
//    most one row long, every warp stages only the activations of its own
//    run (stage_warp) and no CTA barrier follows the dependency wait;
//    otherwise the CTA stages the whole row once (stage).  Decode = one AND per 4 codes
//    (unsigned codes c = w + 1 masked in place, unsigned x signed dp4a); the
//    4^i slot factor and the sum_k x offset are removed once per row.
//  * Every mbarrier wait is bounded (clock64); on time-out the kernel sets
//    the library's device error word and stops; the host reads it with
//    bw_device_error().  Before leaving, the issuing lane waits (bounded)
//    for the copies it issued.
//  * Programmatic dependent launch: the first pieces are requested before
//    griddepcontrol.wait (the packed weights are static once bw_repack has
//    returned); activations, scales and outputs are touched after it.
#include <atomic>

#include "bw_pipe.cuh"

namespace bw {

__device__ unsigned int g_device_error;  // time-out bits, see bw.h

namespace {

using namespace pipe;

// Ring slots per warp for the public GEMV: measured in one call against 2
// slots, 3 give 2.5 % more on the decode-shape sweep and 2.4 % on 55296 x
// 5120 (the layer stack keeps 2: its heavier prologues prefer the third CTA
// per SM).
constexpr int kGemvSlots = 3;

// Failure-detection self-test: a wait that nothing can complete (the
// barrier expects two arrivals and gets one) must run out, report bit 8 in
// the device error word and return, leaving the context usable.
__global__ void selftest_wait_kernel(long long limit) {
  __shared__ uint64_t bar;
  if (threadIdx.x != 0) return;
  mbar_init(&bar, 2);
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  mbar_arrive(&bar);
  if (!mbar_wait(&bar, 0u, limit)) atomicOr(&g_device_error, 8u);
}

// Prologue: the MT int8 activation rows x[m][0..K) (row stride x_ld) and,
// in bf16 mode, their scales s[m].  All loads of a row are independent; K is
// a multiple of 4, and x rows are 16-byte aligned when vec_x is set.
struct StageInt8 {
  const int8_t *x;
  const float *s;  // null in accumulator mode
  int x_ld, K, vec_x;
  int rows;                  // activation rows of this launch
  const void *ws;            // weight scales (null in accumulator mode)

  // Every input may come from the preceding kernel, so nothing is read
  // before the dependency wait.  The lines of x, s and ws are only
  // prefetched into L2 (a hint that returns no data: L2 is the point of
  // coherence, so the loads after the wait still see the final values),
  // one line per thread across the grid.
  struct Pre {};
  __device__ __forceinline__ Pre pre_wait() const {
    const char *lo = reinterpret_cast<const char *>(x);
    const char *hi = lo + size_t(rows - 1) * x_ld + K;  // end of the last row
    const size_t base = reinterpret_cast<size_t>(lo) & ~size_t(127);
    const int lines = int((reinterpret_cast<size_t>(hi) - base + 127) / 128);
    const int stride = gridDim.x * blockDim.x;
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < lines + 2;
         i += stride) {
      const void *p = i == lines ? static_cast<const void *>(s)
                      : i == lines + 1
                          ? ws
                          : static_cast<const void *>(
                                lo + (i == 0 ? 0 : size_t(i) * 128 -
                                                       (reinterpret_cast<size_t>(lo) - base)));
      if (p) asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
    }
    return Pre{};
  }

  // Per-warp staging (PipeArgs::per_warp_x): a warp loads only the chunks
  // its run covers -- [a_lo, a_lo + len_a) of a row, then [0, len_b) (the
  // start of the next row group's) -- into its own region (row stride
  // xrow_w), in that order, and returns the two segments' sums per row; it
  // needs 16-byte aligned rows.
  static constexpr bool kPerWarpX = true;
  __host__ __device__ bool per_warp_capable() const { return vec_x != 0; }
  template <int MT>
  __device__ __forceinline__ void stage_warp(const Pre &, int8_t *xw,
                                             uint32_t xrow_w, int a_lo,
                                             int len_a, int len_b,
                                             float *s_sm, int (&xsum_a)[MT],
                                             int (&xsum_b)[MT]) const {
    constexpr int kBatch = 4;
    const int lane = threadIdx.x & 31;
    const float sv = (s && threadIdx.x < MT) ? s[threadIdx.x] : 0.0f;
    const int nv = (len_a + len_b) * 4;  // 16-byte vectors of a row
    const int va = len_a * 4;            // of them in the first segment
    const int kv = K / 16;               // vectors inside K (K % 16 == 0)
#pragma unroll
    for (int m = 0; m < MT; ++m) {
      const uint4 *src = reinterpret_cast<const uint4 *>(x + size_t(m) * x_ld);
      uint4 *dst = reinterpret_cast<uint4 *>(xw + m * xrow_w);
      int pa = 0, pb = 0;
      for (int v0 = lane; v0 < nv; v0 += kBatch * 32) {
        uint4 x4[kBatch];
#pragma unroll
        for (int b = 0; b < kBatch; ++b) {
          const int v = v0 + b * 32;
          const int gv = v < va ? a_lo * 4 + v : v - va;  // vector of the row
          x4[b] = (v < nv && gv < kv) ? __ldg(src + gv)
                                      : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int b = 0; b < kBatch; ++b) {
          const int v = v0 + b * 32;
          if (v < nv) {
            dst[v] = x4[b];
            int t = dp4a_us(0x01010101u, x4[b].x, 0);
            t = dp4a_us(0x01010101u, x4[b].y, t);
            t = dp4a_us(0x01010101u, x4[b].z, t);
            t = dp4a_us(0x01010101u, x4[b].w, t);
            if (v < va)
              pa += t;
            else
              pb += t;
          }
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        pa += __shfl_xor_sync(0xffffffffu, pa, o);
        pb += __shfl_xor_sync(0xffffffffu, pb, o);
      }
      xsum_a[m] = pa;
      xsum_b[m] = pb;
    }
    if (s && threadIdx.x < MT) s_sm[threadIdx.x] = sv;
  }

  template <int MT>
  __device__ __forceinline__ void stage(const Pre &, const StageCtx &c,
                                        int (&part)[MT]) const {
    // Every load is issued before the first shared-memory store that needs
    // one (issue is in order): the scale, then up to kBatch vectors per row
    // and thread at a time.
    constexpr int kBatch = 4;
    const float sv = (s && threadIdx.x < MT) ? s[threadIdx.x] : 0.0f;
    const int tid = threadIdx.x, nthreads = blockDim.x;
#pragma unroll
    for (int m = 0; m < MT; ++m) {
      int p = 0;
      int8_t *dst = c.xs + m * c.xrow;
      if (vec_x) {
        const uint4 *src = reinterpret_cast<const uint4 *>(x + size_t(m) * x_ld);
        const int nv = c.chunks * 4;
        for (int v0 = tid; v0 < nv; v0 += kBatch * nthreads) {
          uint4 x4[kBatch];
#pragma unroll
          for (int b = 0; b < kBatch; ++b) {
            const int v = v0 + b * nthreads;
            x4[b] = (v < nv && 16 * v < K) ? __ldg(src + v)
                                           : make_uint4(0u, 0u, 0u, 0u);
          }
#pragma unroll
          for (int b = 0; b < kBatch; ++b) {
            const int v = v0 + b * nthreads;
            if (v < nv) {
              reinterpret_cast<uint4 *>(dst)[v] = x4[b];
              p = dp4a_us(0x01010101u, x4[b].x, p);
              p = dp4a_us(0x01010101u, x4[b].y, p);
              p = dp4a_us(0x01010101u, x4[b].z, p);
              p = dp4a_us(0x01010101u, x4[b].w, p);
            }
          }
        }
      } else {
        const unsigned int *src =
            reinterpret_cast<const unsigned int *>(x + size_t(m) * x_ld);
        const int nw = c.chunks * 16;
        for (int w0 = tid; w0 < nw; w0 += kBatch * nthreads) {
          uint32_t xv[kBatch];
#pragma unroll
          for (int b = 0; b < kBatch; ++b) {
            const int wd = w0 + b * nthreads;
            xv[b] = (wd < nw && 4 * wd < K) ? __ldg(src + wd) : 0u;
          }
#pragma unroll
          for (int b = 0; b < kBatch; ++b) {
            const int wd = w0 + b * nthreads;
            if (wd < nw) {
              reinterpret_cast<uint32_t *>(dst)[wd] = xv[b];
              p = dp4a_us(0x01010101u, xv[b], p);
            }
          }
        }
      }
      part[m] = p;
    }
    if (s && threadIdx.x < MT) c.s_sm[threadIdx.x] = sv;
  }
};

template <int MT, bool ACC>
cudaError_t launch_instance(const GemvArgs &g, cudaStream_t stream) {
  PipeArgs a{};
  a.w = g.w;
  a.N = g.N;
  a.chunks = g.chunks;
  a.n_groups = g.n_groups;
  a.slots = kGemvSlots;
  a.err = device_error_word();
  if (!a.err) return cudaErrorInvalidSymbol;
  const StageInt8 pro{g.x, ACC ? nullptr : g.s, g.x_ld, g.K, g.vec_x, MT,
                      ACC ? nullptr : static_cast<const void *>(g.ws)};
  const EpiOut<ACC> epi{g.out, g.out_ld, g.ws, g.seg};
  return launch_pipe<MT>(a, pro, epi, stream);
}

}  // namespace

// Cached per device: every launch needs the address and the lookup costs a
// runtime call.  Threads racing on the first lookup store the same value, so
// the cache is a relaxed atomic.  Like the other per-device state of the
// library (SM counts, kernel attributes), it assumes the device is not reset
// with cudaDeviceReset while the library is loaded (bw.h says so).
unsigned int *device_error_word() {
  static std::atomic<unsigned int *> word[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64)
    return nullptr;
  unsigned int *w = word[dev].load(std::memory_order_relaxed);
  if (!w) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_device_error) != cudaSuccess) return nullptr;
    w = static_cast<unsigned int *>(p);
    word[dev].store(w, std::memory_order_relaxed);
  }
  return w;
}

bool pipe_fits(int mt, int K) {
  if (mt != 1 && mt != 2 && mt != 4) return false;
  // The activations are staged whole: K too long for shared memory goes to
  // the register-streamed kernel.
  return pipe_smem_bytes(mt, chunks_per_row(K), kPipeSlotChunks,
                         kGemvSlots, kPipeMaxGroupsPerCta) <= 227u * 1024u;
}

cudaError_t launch_gemv_pipe(const GemvArgs &a, int mt, bool acc_out,
                             cudaStream_t stream) {
  if (mt == 1)
    return acc_out ? launch_instance<1, true>(a, stream)
                   : launch_instance<1, false>(a, stream);
  if (mt == 2)
    return acc_out ? launch_instance<2, true>(a, stream)
                   : launch_instance<2, false>(a, stream);
  if (mt == 4)
    return acc_out ? launch_instance<4, true>(a, stream)
                   : launch_instance<4, false>(a, stream);
  return cudaErrorInvalidConfiguration;
}

cudaError_t launch_selftest_wait(cudaStream_t stream) {
  int dev = 0, khz = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess)
    e = cudaDeviceGetAttribute(&khz, cudaDevAttrClockRate, dev);
  if (e != cudaSuccess) return e;
  const long long limit = (long long)(khz > 0 ? khz : 2000000) * 10;  // ~10 ms
  selftest_wait_kernel<<<1, 32, 0, stream>>>(limit);
  return cudaGetLastError();
}

cudaError_t read_device_error(cudaStream_t stream, unsigned int *out) {
  const unsigned int zero = 0;
  cudaError_t e = cudaMemcpyFromSymbolAsync(out, g_device_error,
                                            sizeof(unsigned int), 0,
                                            cudaMemcpyDeviceToHost, stream);
  if (e == cudaSuccess)
    e = cudaMemcpyToSymbolAsync(g_device_error, &zero, sizeof(unsigned int),
                                0, cudaMemcpyHostToDevice, stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
  return e;
}

}  // namespace bw
