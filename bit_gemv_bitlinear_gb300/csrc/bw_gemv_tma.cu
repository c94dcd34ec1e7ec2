// bw_gemv_tma.cu -- the W2A8 ternary GEMV streamed by TMA bulk copies.
//
// Same product and epilogue as bw_gemv.cu (acc = sum_k w x exactly in int32,
// y = bf16((acc / s[m]) * ws[seg(n)])).  Source: "BitNet GPU 推理框架：从零构建
// W2A8 的 2-bit 大模型 CUDA GEMV 内核", §5.2 (2-bit decode), §5.3 (dp4a dot
// product, shuffle reduction, scale epilogue), §4.2 (weight-scale segments).
//
// Design for sm_103a:
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
//    conflict); the int8 activations, staged once in shared memory, come as
//    four 128-bit broadcast loads per chunk.  Decode = one AND per 4 codes
//    (unsigned codes c = w + 1 masked in place, unsigned x signed dp4a); the
//    4^i slot factor and the sum_k x offset are removed once per row.
//  * Every mbarrier wait is bounded (clock64); on time-out the kernel sets
//    the library's device error word and stops; the host reads it with
//    bw_device_error().  Before leaving, the issuing lane waits (bounded)
//    for the copies it issued.
//  * Programmatic dependent launch: the first ring fills are issued before
//    griddepcontrol.wait (the packed weights are static once bw_repack has
//    returned); activations, scales and outputs are touched after it, and
//    the scales are staged in shared memory with the activations so that no
//    global load sits in the epilogue.
#include "bw_internal.cuh"

namespace bw {

__device__ unsigned int g_device_error;  // time-out bits, see bw.h

namespace {

constexpr long long kWaitLimitCycles = 2000000000LL;  // about one second

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)),
               "r"(count)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(
                   smem_addr(bar))
               : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar,
                                                      uint32_t bytes) {
  asm volatile(
      "mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(
          smem_addr(bar)),
      "r"(bytes)
      : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar,
                                              uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return done != 0;
}

// Wait for the phase of `parity` to complete, for at most `limit` cycles
// (about a second by default).
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity,
                                          long long limit = kWaitLimitCycles) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity))
    if (clock64() - t0 > limit) return false;
  return true;
}

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

__device__ __forceinline__ void bulk_copy_g2s(void *dst, const void *src,
                                              uint32_t bytes, uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes "
      "[%0], [%1], %2, [%3];" ::"r"(smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}

__device__ __forceinline__ void pdl_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;");
}

__device__ __forceinline__ int dp4a_us(uint32_t a, uint32_t b, int c) {
  int d;
  asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

// Activations in shared memory: row m, chunk j (64 int8 values) at byte
// m xrow + 64 j, zero beyond K.
__host__ __device__ inline uint32_t xs_row_bytes(int chunks) {
  return uint32_t(chunks) * 64u;
}

// Stages the MT activation rows (zero beyond K) in shared memory and
// returns this thread's share of sum_k x[m][k] in part[m].  All loads of a
// row are independent; K is a multiple of 4.
template <int MT>
__device__ __forceinline__ void stage_x(const GemvArgs &a, int8_t *xs,
                                        uint32_t xrow, int tid, int nthreads,
                                        int (&part)[MT]) {
#pragma unroll
  for (int m = 0; m < MT; ++m) {
    int p = 0;
    int8_t *dst = xs + m * xrow;
    if (a.vec_x) {
      const uint4 *src =
          reinterpret_cast<const uint4 *>(a.x + size_t(m) * a.x_ld);
      for (int v = tid; v < a.chunks * 4; v += nthreads) {
        uint4 x4 = make_uint4(0u, 0u, 0u, 0u);
        if (16 * v < a.K) x4 = __ldg(src + v);
        reinterpret_cast<uint4 *>(dst)[v] = x4;
        p = dp4a_us(0x01010101u, x4.x, p);
        p = dp4a_us(0x01010101u, x4.y, p);
        p = dp4a_us(0x01010101u, x4.z, p);
        p = dp4a_us(0x01010101u, x4.w, p);
      }
    } else {
      const unsigned int *src =
          reinterpret_cast<const unsigned int *>(a.x + size_t(m) * a.x_ld);
      for (int wd = tid; wd < a.chunks * 16; wd += nthreads) {
        uint32_t v = 0u;
        if (4 * wd < a.K) v = __ldg(src + wd);
        reinterpret_cast<uint32_t *>(dst)[wd] = v;
        p = dp4a_us(0x01010101u, v, p);
      }
    }
    part[m] = p;
  }
}

// Products of one chunk: 16 bytes of packed codes (row r, 64 weights) at
// wp against the 64 activations of each row m at xp + m xrow.
template <int MT>
__device__ __forceinline__ void dot_chunk(const uint8_t *wp, const int8_t *xp,
                                          uint32_t xrow, int (&acc)[MT][4]) {
  const uint4 wv = *reinterpret_cast<const uint4 *>(wp);
  const uint32_t wd[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
  for (int t = 0; t < 4; ++t) {
    const uint32_t c0w = wd[t] & 0x03030303u;
    const uint32_t c1w = wd[t] & 0x0c0c0c0cu;
    const uint32_t c2w = wd[t] & 0x30303030u;
    const uint32_t c3w = wd[t] & 0xc0c0c0c0u;
#pragma unroll
    for (int m = 0; m < MT; ++m) {
      // activation words 4t..4t+3 of the chunk: k = 64j + 16t + 4i + b
      const uint4 xv = *reinterpret_cast<const uint4 *>(xp + m * xrow + 16 * t);
      acc[m][0] = dp4a_us(c0w, xv.x, acc[m][0]);
      acc[m][1] = dp4a_us(c1w, xv.y, acc[m][1]);
      acc[m][2] = dp4a_us(c2w, xv.z, acc[m][2]);
      acc[m][3] = dp4a_us(c3w, xv.w, acc[m][3]);
    }
  }
}

// Dot products of `chunks` consecutive chunks of one row group held in
// shared memory at wbase, the first being chunk c0 of the row: lane (q, r)
// takes chunks 4 pq + q of row r.  acc[m][i] collects slot i (codes scaled
// by 4^i) against activation row m.  Two pointers advance by constants;
// only the last, partial quad is predicated.
template <int MT>
__device__ __forceinline__ void dot_row_group(const uint8_t *wbase,
                                              const int8_t *xs, uint32_t xrow,
                                              int c0, int chunks, int q,
                                              int r, int (&acc)[MT][4]) {
  const uint8_t *wp = wbase + q * kGroupChunkBytes + r * kChunkBytes;
  const int8_t *xp = xs + (c0 + q) * kChunkWeights;
  const int quads = chunks >> 2;
#pragma unroll 2
  for (int pq = 0; pq < quads; ++pq) {
    dot_chunk<MT>(wp, xp, xrow, acc);
    wp += 4 * kGroupChunkBytes;
    xp += 4 * kChunkWeights;
  }
  if (q < (chunks & 3)) dot_chunk<MT>(wp, xp, xrow, acc);
}

// Remove the slot factors: (((a3/4 + a2)/4 + a1)/4 + a0, exact because a_i is
// a multiple of 4^i; then sum the 4 chunk lanes of the row.
__device__ __forceinline__ int fold_row(const int (&a)[4]) {
  int v = ((((a[3] >> 2) + a[2]) >> 2) + a[1]) >> 2;
  v += a[0];
  v += __shfl_xor_sync(0xffffffffu, v, 8);
  v += __shfl_xor_sync(0xffffffffu, v, 16);
  return v;
}

// Epilogue of one output; s_sm / ws_sm are the scales staged in shared
// memory (fp32 copies of s[m] and of the bf16 weight scales).
template <int MT, bool ACC_OUT>
__device__ __forceinline__ void store_row(const GemvArgs &a, int n, int m,
                                          int total, const float *s_sm,
                                          const float *ws_sm) {
  if (ACC_OUT) {
    static_cast<int *>(a.out)[size_t(m) * a.out_ld + n] = total;
  } else {
    int seg = 0;
#pragma unroll
    for (int i = 1; i < BW_MAX_WS; ++i)
      if (i < a.seg.n_ws && n >= a.seg.bounds[i]) seg = i;
    const float scaled = static_cast<float>(total) / s_sm[m];
    const float v = scaled * ws_sm[seg];
    static_cast<__nv_bfloat16 *>(a.out)[size_t(m) * a.out_ld + n] =
        __float2bfloat16_rn(v);
  }
}

// ---------------------------------------------------------------------------
// Balanced per-warp pipelines (pipe mode).
//
// CTA b owns the k consecutive row groups b k .. b k + k - 1 (the last CTA
// may own fewer); its 8 warps split the CTA's k C chunks into 8 contiguous,
// equal runs.  A warp walks its run in pieces of at most `slot_chunks`
// chunks that never cross a row-group boundary; each piece is one bulk copy
// into the next slot of the warp's own ring of `slots` slots.  Lane 0 of the
// warp issues the copies: the first `slots` pieces before
// griddepcontrol.wait, then piece i + slots into the slot of piece i as soon
// as the warp has read it, so each warp keeps slots - 1 pieces in flight
// whatever the other warps do.  When a piece ends a row group or the run, the
// warp folds its partial sums and adds them (int32, exact in any order) to
// the CTA's row totals in shared memory; one epilogue per CTA then scales
// and stores the k * 8 rows.  Every warp has the same amount of work and
// every CTA but the last the same number of groups, so no tail of the grid
// runs on a few warps with few bytes in flight.
struct PipeLayout {
  uint32_t ring, xs, sums, tot, bars, total;
};

// sums: [MT] activation scales s, [BW_MAX_WS] weight scales (as fp32),
// [warps][MT] per-warp activation sums; tot: [k][MT][8] row totals.
__host__ __device__ inline PipeLayout pipe_layout(int mt, int chunks,
                                                  int slot_chunks, int slots,
                                                  int warps, int k) {
  PipeLayout l;
  l.ring = 0;
  l.xs = uint32_t(warps * slots * slot_chunks) * kGroupChunkBytes;
  l.sums = l.xs + uint32_t(mt) * xs_row_bytes(chunks);
  const uint32_t sums_bytes = uint32_t((mt + BW_MAX_WS + warps * mt) * 4);
  l.tot = (l.sums + sums_bytes + 15) / 16 * 16;
  l.bars = l.tot + uint32_t(k * mt * 8 * 4);
  l.total = l.bars + uint32_t(warps * slots * 8);
  return l;
}

constexpr int kPipeWarps = 8;
constexpr int kPipeMaxGroupsPerCta = 256;
constexpr int kPipeMinGroupsPerCta = 2;  // fewer CTAs staging x for small N

// Orders this warp's earlier generic-proxy reads of a slot before the
// bulk copy (async proxy) that overwrites it.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Position in a warp's run: chunk u of the CTA's range = chunk c of the
// CTA's row group g.
struct RunCursor {
  int u, g, c;
  __device__ __forceinline__ int piece(int ks, int chunks, int end) const {
    return min(min(ks, chunks - c), end - u);
  }
  __device__ __forceinline__ void advance(int len, int chunks) {
    u += len;
    c += len;
    if (c == chunks) {
      c = 0;
      ++g;
    }
  }
};

template <int MT, bool ACC_OUT>
__global__ void __launch_bounds__(kPipeWarps * 32)
gemv_w2a8_pipe_kernel(const GemvArgs a, const TmaPlan p) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int KS = p.slot_chunks;
  const int R = p.slots;
  const int C = a.chunks;
  const int k = p.groups_per_cta;
  const uint32_t slot_bytes = uint32_t(KS) * kGroupChunkBytes;
  const uint32_t xrow = xs_row_bytes(C);
  const PipeLayout L = pipe_layout(MT, C, KS, R, kPipeWarps, k);
  uint8_t *ring = smem + L.ring + size_t(warp) * R * slot_bytes;
  int8_t *xs = reinterpret_cast<int8_t *>(smem + L.xs);
  float *s_sm = reinterpret_cast<float *>(smem + L.sums);
  float *ws_sm = s_sm + MT;
  int *sx_part = reinterpret_cast<int *>(ws_sm + BW_MAX_WS);  // [warps][MT]
  int *tot = reinterpret_cast<int *>(smem + L.tot);           // [k][MT][8]
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + L.bars) + warp * R;

  const int g_lo = int(blockIdx.x) * k;
  const int n_g = min(k, a.n_groups - g_lo);
  const int U = n_g * C;  // chunks of this CTA (k C <= 256 * 384)
  const int run_lo = U * warp / kPipeWarps;
  const int run_hi = U * (warp + 1) / kPipeWarps;
  const uint8_t *wcta = a.w + size_t(g_lo) * C * kGroupChunkBytes;

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
                  wcta + (size_t(iss.g) * C + iss.c) * kGroupChunkBytes,
                  bytes, &full[slot]);
    iss.advance(len, C);
    ++issued;
  };
  if (lane == 0) {
    for (int s = 0; s < R; ++s) mbar_init(&full[s], 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    // The weights are static once written (bw_repack synchronises its
    // stream): the first pieces are requested before the dependency wait.
    for (int s = 0; s < R && iss.u < run_hi; ++s) issue_next(s);
  }
  for (int t = threadIdx.x; t < n_g * MT * 8; t += blockDim.x) tot[t] = 0;
  pdl_wait();

  if (!ACC_OUT) {
    if (threadIdx.x < MT) s_sm[threadIdx.x] = a.s[threadIdx.x];
    if (threadIdx.x >= 32 && threadIdx.x < 32 + a.seg.n_ws)
      ws_sm[threadIdx.x - 32] = __bfloat162float(a.ws[threadIdx.x - 32]);
  }
  int part[MT];
  stage_x<MT>(a, xs, xrow, threadIdx.x, int(blockDim.x), part);
#pragma unroll
  for (int m = 0; m < MT; ++m) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
      part[m] += __shfl_xor_sync(0xffffffffu, part[m], o);
    if (lane == 0) sx_part[warp * MT + m] = part[m];
  }
  __syncthreads();  // activations staged, totals zeroed, barriers set up
  pdl_trigger();    // dependents may start their prologue on free SM slots

  const int q = lane >> 3;  // chunk residue (relative to the piece) mod 4
  const int r = lane & 7;   // row inside the group
  int acc[MT][4];
#pragma unroll
  for (int m = 0; m < MT; ++m)
#pragma unroll
    for (int t = 0; t < 4; ++t) acc[m][t] = 0;
  bool ok = true;
  int consumed = 0, slot = 0;
  uint32_t phase = 0;
  while (cur.u < run_hi) {
    // warp-uniform outcome before any full-mask shuffle below
    if (!__all_sync(0xffffffffu, mbar_wait(&full[slot], phase))) {
      ok = false;
      break;
    }
    const int len = cur.piece(KS, C, run_hi);
    dot_row_group<MT>(ring + size_t(slot) * slot_bytes, xs, xrow, cur.c, len,
                      q, r, acc);
    __syncwarp();
    if (lane == 0 && iss.u < run_hi) {  // piece consumed + R: this slot
      fence_proxy_async_smem();
      issue_next(slot);
    }
    const int g = cur.g;
    cur.advance(len, C);
    ++consumed;
    if (cur.c == 0 || cur.u == run_hi) {  // row group or run finished
#pragma unroll
      for (int m = 0; m < MT; ++m) {
        const int v = fold_row(acc[m]);
        if (q == 0) atomicAdd(&tot[(g * MT + m) * 8 + r], v);
#pragma unroll
        for (int t = 0; t < 4; ++t) acc[m][t] = 0;
      }
    }
    if (++slot == R) {
      slot = 0;
      phase ^= 1u;
    }
  }
  if (!ok && lane == 0) {
    atomicOr(&g_device_error, 4u);
    // copies still in flight land before the CTA may leave
    for (int i = consumed; i < issued; ++i)
      if (!mbar_wait(&full[i % R], uint32_t(i / R) & 1u))
        atomicOr(&g_device_error, 2u);
  }
  __syncthreads();  // every partial sum is in `tot`

  int sx[MT];  // sum_k x[m][k] over the whole row
#pragma unroll
  for (int m = 0; m < MT; ++m) {
    sx[m] = 0;
#pragma unroll
    for (int w = 0; w < kPipeWarps; ++w) sx[m] += sx_part[w * MT + m];
  }
  for (int t = threadIdx.x; t < n_g * 8; t += blockDim.x) {
    const int gl = t >> 3, rr = t & 7;
    const int n = (g_lo + gl) * kGroupRows + rr;
    if (n < a.N) {
#pragma unroll
      for (int m = 0; m < MT; ++m)
        store_row<MT, ACC_OUT>(a, n, m, tot[(gl * MT + m) * 8 + rr] - sx[m],
                               s_sm, ws_sm);
    }
  }
}

// Sets the opt-in shared-memory size once per device and returns how many
// CTAs of `kernel` are resident on the device at once (at least one).
template <class Kernel>
cudaError_t resident_ctas(Kernel kernel, bool *configured, int threads,
                          uint32_t smem, int64_t *resident) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!configured[dev]) {
    e = cudaFuncSetAttribute(kernel,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             227 * 1024);
    if (e != cudaSuccess) return e;
    configured[dev] = true;
  }
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, threads,
                                                    smem) != cudaSuccess ||
      per_sm < 1)
    per_sm = 1;
  *resident = int64_t(per_sm) * device_sm_count();
  return cudaSuccess;
}

// Launches `kernel` on `grid` CTAs with programmatic dependent launch.
template <class Kernel>
cudaError_t launch_pdl(Kernel kernel, int64_t grid, int threads,
                       uint32_t smem, const GemvArgs &a, const TmaPlan &p,
                       cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(grid > 0 ? grid : 1));
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, a, p);
}

template <int MT, bool ACC>
cudaError_t launch_tma_instance(const TmaPlan &plan, const GemvArgs &a,
                                cudaStream_t stream) {
  int64_t resident = 0;
  // k groups per CTA with k as small as the resident CTAs allow
  // (at most kPipeMaxGroupsPerCta; beyond that the grid runs in waves), and
  // slots no longer than a warp's run.
  static bool configured[64];
  TmaPlan p = plan;
  // k from the residency at k = 1, then once more at that k (the row
  // totals grow with k).
  int64_t k = 1;
  for (int pass = 0; pass < 2; ++pass) {
    const PipeLayout Lk = pipe_layout(MT, a.chunks, p.slot_chunks, p.slots,
                                      p.consumers, int(k));
    cudaError_t e = resident_ctas(gemv_w2a8_pipe_kernel<MT, ACC>, configured,
                                  p.consumers * 32, Lk.total, &resident);
    if (e != cudaSuccess) return e;
    k = (a.n_groups + resident - 1) / resident;
    if (k > kPipeMaxGroupsPerCta) k = kPipeMaxGroupsPerCta;
    if (k < kPipeMinGroupsPerCta) k = kPipeMinGroupsPerCta;
  }
  const int64_t grid = (a.n_groups + k - 1) / k;
  const int64_t run = (k * a.chunks + p.consumers - 1) / p.consumers;
  if (run < p.slot_chunks) p.slot_chunks = int(run < 1 ? 1 : run);
  p.groups_per_cta = int(k);
  const PipeLayout L = pipe_layout(MT, a.chunks, p.slot_chunks, p.slots,
                                   p.consumers, p.groups_per_cta);
  return launch_pdl(gemv_w2a8_pipe_kernel<MT, ACC>, grid, p.consumers * 32,
                    L.total, a, p, stream);
}

}  // namespace

bool plan_gemv_tma(int mt, int N, int K, int num_sms, TmaPlan *p) {
  (void)N;
  (void)num_sms;
  if (mt != 1 && mt != 2 && mt != 4) return false;
  // Pieces of up to 4 KB, two slots per warp: 64 KB of ring per 8-warp CTA,
  // about three CTAs per SM for K <= 8192.
  p->consumers = kPipeWarps;
  p->slot_chunks = 32;
  p->slots = 2;
  p->groups_per_cta = 0;  // chosen at launch from the resident CTAs
  // The activations are staged whole: K too long for shared memory goes to
  // the register-streamed kernel.
  const PipeLayout L = pipe_layout(mt, chunks_per_row(K), p->slot_chunks,
                                   p->slots, p->consumers,
                                   kPipeMaxGroupsPerCta);
  return L.total <= 227u * 1024u;
}

cudaError_t launch_gemv_tma(const TmaPlan &p, const GemvArgs &a, int mt,
                            bool acc_out, cudaStream_t stream) {
  if (mt == 1)
    return acc_out ? launch_tma_instance<1, true>(p, a, stream)
                   : launch_tma_instance<1, false>(p, a, stream);
  if (mt == 2)
    return acc_out ? launch_tma_instance<2, true>(p, a, stream)
                   : launch_tma_instance<2, false>(p, a, stream);
  if (mt == 4)
    return acc_out ? launch_tma_instance<4, true>(p, a, stream)
                   : launch_tma_instance<4, false>(p, a, stream);
  return cudaErrorInvalidConfiguration;
}

cudaError_t launch_selftest_wait(cudaStream_t stream) {
  int khz = 0;
  cudaError_t e = cudaDeviceGetAttribute(&khz, cudaDevAttrClockRate, 0);
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
