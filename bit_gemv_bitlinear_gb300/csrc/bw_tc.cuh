// bw_tc.cuh -- inline-PTX helpers shared by the tcgen05 kernels
// (bw_gemv_tc.cu, bw_gemm.cu): tensor-memory allocation, MMA issue and
// commit, tiled TMA loads, shared-memory matrix and instruction
// descriptors, tensor-memory loads and stores, the 2-bit weight decode into
// fp16 operands, the epilogues' corrected-reciprocal division and 16-byte
// shared-memory load, and the host-side tensor-map encoder.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_fp16.h>

#include "bw_pipe.cuh"

namespace bw {
namespace {

using namespace pipe;

// ---- tcgen05 / proxy helpers -------------------------------------------

__device__ __forceinline__ void tmem_alloc(uint32_t *slot, uint32_t cols) {
  asm volatile(
      "tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
          smem_addr(slot)),
      "r"(cols)
      : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::
                   : "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t cols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(
                   taddr),
               "r"(cols)
               : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D (tmem) (+)= A (tmem) * B (smem descriptor); M = 128, kind::f16.
__device__ __forceinline__ void tc_mma(uint32_t d, uint32_t a, uint64_t bdesc,
                                       uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d),
      "r"(a), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrives on `bar` once every tcgen05.mma issued so far by this thread is
// complete.
__device__ __forceinline__ void tc_commit(uint64_t *bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 "
      "[%0];" ::"r"(smem_addr(bar))
      : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
  asm volatile(
      "{\n\t.reg .b64 st;\n\t"
      "mbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(smem_addr(bar))
      : "memory");
}

__device__ __forceinline__ void fence_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// 2-D tiled bulk copy of one box of `map` at element coordinates (c0, c1);
// completes `bytes` = the box size on `bar` (out-of-range elements are
// zero-filled and still counted).
__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map,
                                            int c0, int c1, uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_"
      "tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1),
      "r"(smem_addr(bar))
      : "memory");
}

// True in one lane of the (converged) warp: the lowest active one.
__device__ __forceinline__ bool elect_one() {
  uint32_t p;
  asm volatile(
      "{\n\t.reg .pred e;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "selp.u32 %0, 1, 0, e;\n\t}"
      : "=r"(p));
  return p != 0;
}

// Warp-uniform bounded wait (all lanes call it).
__device__ __forceinline__ bool warp_wait(uint64_t *bar, uint32_t parity) {
  return __all_sync(0xffffffffu, mbar_wait(bar, parity));
}

// Shared-memory matrix descriptor: K-major rows of 128 bytes with the
// 128-byte swizzle, 8-row groups 1024 bytes apart.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t addr) {
  uint64_t d = uint64_t((addr >> 4) & 0x3FFFu);
  d |= uint64_t(1) << 16;             // leading byte offset (unused here)
  d |= uint64_t(1024 >> 4) << 32;     // stride byte offset
  d |= uint64_t(1) << 46;             // descriptor version
  d |= uint64_t(2) << 61;             // 128-byte swizzle
  return d;
}

// Instruction descriptor, kind::f16: fp16 A and B (K-major), fp32 D,
// M = 128, N = n.
__host__ __device__ constexpr uint32_t tc_idesc(int n) {
  return (1u << 4) | (uint32_t(n >> 3) << 17) | (uint32_t(128 >> 4) << 24);
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
      "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, "
      "%31, %32};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]),
      "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]),
      "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]), "r"(v[16]), "r"(v[17]),
      "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]),
      "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]), "r"(v[28]), "r"(v[29]),
      "r"(v[30]), "r"(v[31])
      : "memory");
}

__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// 4 consecutive accumulator columns of this warp's 32 lanes; the load and
// its wait are one asm statement, so no use of the values can be scheduled
// before the wait.
__device__ __forceinline__ void tmem_ld4(uint32_t taddr, float (&v)[4]) {
  uint32_t r[4];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0, %1, %2, %3}, [%4];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 4; ++i) v[i] = __uint_as_float(r[i]);
}

// a / s rounded to nearest even, from r = RN(1 / s): two correction steps
// of the product a r by its exact residual (fma).  The first brings the
// quotient within one ulp of a / s, so the second residual is exact and,
// by P. Markstein's theorem on the final step of division (IBM J. Res.
// Dev. 34(1), 1990), the second correction is the correctly rounded
// quotient.  Valid for an integer |a| <= 2^24 and s, r in [2^-60, 2^60]
// (no intermediate leaves the normal range); the caller divides otherwise.
// Five FMA-pipe instructions instead of a division per output.
__device__ __forceinline__ float div_by_recip(float a, float s, float r) {
  const float q0 = a * r;
  const float q1 = fmaf(fmaf(-q0, s, a), r, q0);
  return fmaf(fmaf(-q1, s, a), r, q1);
}

// 16 bytes of shared memory.  Volatile (kept in order with the barriers and
// tensor-memory loads around it) but without a memory clobber, so that the
// compiler need not order it against the epilogue's global stores.
__device__ __forceinline__ float4 lds4(const void *p) {
  float4 v;
  asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(smem_addr(p)));
  return v;
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t s) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(s));
  return d;
}

// One packed word (16 weights) -> 8 columns of fp16x2 (c 4^sl 2^-24), in
// the pair order of the file header: column j = (byte b = j >> 2, slot
// sl = j & 3), code bits 8 b + 2 sl (+16 for the high half) kept in place
// (bytes 1 and 3 shifted down by 8).
__device__ __forceinline__ void decode_word(uint32_t w, uint32_t *col) {
  const uint32_t v = w >> 8;
  col[0] = w & 0x00030003u;
  col[1] = w & 0x000C000Cu;
  col[2] = w & 0x00300030u;
  col[3] = w & 0x00C000C0u;
  col[4] = v & 0x00030003u;
  col[5] = v & 0x000C000Cu;
  col[6] = v & 0x00300030u;
  col[7] = v & 0x00C000C0u;
}

__device__ __forceinline__ uint32_t hfma2(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

// Column scale 4^-r and -1152 4^-r as fp16x2 (r = slot of the column).
__device__ __forceinline__ uint32_t col_scale(int r) {
  return r == 0 ? 0x3C003C00u : r == 1 ? 0x34003400u : r == 2 ? 0x2C002C00u
                                                               : 0x24002400u;
}
__device__ __forceinline__ uint32_t col_bias(int r) {
  return r == 0 ? 0xE480E480u : r == 1 ? 0xDC80DC80u : r == 2 ? 0xD480D480u
                                                               : 0xCC80CC80u;
}

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static std::atomic<PFN_cuTensorMapEncodeTiled_v12000> cached{nullptr};
  PFN_cuTensorMapEncodeTiled_v12000 fn = cached.load(std::memory_order_relaxed);
  if (!fn) {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                         cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess) {
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
      cached.store(fn, std::memory_order_relaxed);
    }
  }
  return fn;
}

// Row-major 2-D tensor: d1 rows of d0 elements, rows `pitch` bytes apart;
// boxes of b1 rows x b0 elements; out-of-range elements read as zero.  With
// CU_TENSOR_MAP_SWIZZLE_128B a box row must be 128 bytes and lands in
// shared memory with its 16-byte pieces permuted by the row index mod 8 (the
// layout of the tcgen05 128-byte swizzle).
bool encode_2d(CUtensorMap *map, CUtensorMapDataType type, const void *base,
               uint64_t d0, uint64_t d1, uint64_t pitch, uint32_t b0,
               uint32_t b1,
               CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_NONE) {
  PFN_cuTensorMapEncodeTiled_v12000 fn = tensor_map_encoder();
  if (!fn) return false;
  const cuuint64_t dims[2] = {d0, d1};
  const cuuint64_t strides[1] = {pitch};
  const cuuint32_t box[2] = {b0, b1};
  const cuuint32_t elem[2] = {1, 1};
  return fn(map, type, 2, const_cast<void *>(base), dims, strides, box, elem,
            CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace
}  // namespace bw
