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
//    (cp.async.bulk, completion counted in bytes on an mbarrier) into a ring
//    of `stages` buffers.  One producer lane keeps the ring full; the bytes
//    in flight per SM are set by the ring size, not by registers or warps.
//  * A stage is S whole row groups (contiguous in the device layout).
//    Consumer warps form teams of S warps; team t takes every T-th stage of
//    the CTA and warp u of the team the u-th row group of it, i.e. a warp
//    owns all of K for 8 rows: no cross-warp reduction, no CTA barrier in
//    the loop.
//  * Lane (q, r): row r of the group, chunks j = q (mod 4).  One 128-bit
//    shared load gives 64 codes (a contiguous 512-byte warp access, no bank
//    conflict); the int8 activations, staged once in shared memory, come as
//    four 128-bit broadcast loads per chunk.  Decode = one AND per 4 codes
//    (unsigned codes c = w + 1 masked in place, unsigned x signed dp4a); the
//    4^i slot factor and the sum_k x offset are removed once per row.
//  * A warp keeps its totals for 4 row groups in the 4 lane quarters and
//    runs one 32-lane epilogue for those 32 rows.
//  * Every mbarrier wait is bounded (clock64); on time-out the kernel sets
//    the library's device error word and stops; the host reads it with
//    bw_device_error().  Before leaving, the producer waits (bounded) for
//    the copies it issued.
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

__device__ __forceinline__ void prefetch_l2(const void *p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void pdl_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;");
}

// Barrier among the consumer warps only (the producer warp never joins).
__device__ __forceinline__ void consumer_sync(int consumer_threads) {
  asm volatile("bar.sync 1, %0;" ::"r"(consumer_threads) : "memory");
}

__device__ __forceinline__ int dp4a_us(uint32_t a, uint32_t b, int c) {
  int d;
  asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

// Shared-memory carve-up of one CTA (all offsets 16-byte aligned).
struct SmemLayout {
  uint32_t ring, xs, sums, red, bars, total;
};

// sums: [MT] spare, [consumers][MT] per-warp activation sums, 1 abort flag,
//       [MT] activation scales s, [BW_MAX_WS] weight scales (as fp32);
// red: [2][consumers][MT][8] row partials of the K-split mode.
__host__ __device__ inline SmemLayout smem_layout(int mt, int kpad,
                                                  uint32_t stage_bytes,
                                                  int stages, int consumers) {
  SmemLayout l;
  l.ring = 0;
  l.xs = l.ring + stage_bytes * uint32_t(stages);
  l.sums = l.xs + uint32_t(mt * kpad);
  const uint32_t sums_bytes =
      uint32_t((mt + consumers * mt + 1 + mt + BW_MAX_WS) * 4);
  l.red = (l.sums + sums_bytes + 15) / 16 * 16;
  const uint32_t red_bytes = uint32_t(2 * consumers * mt * 8 * 4);
  l.bars = (l.red + red_bytes + 15) / 16 * 16;
  l.total = l.bars + uint32_t(2 * stages * 8);
  return l;
}

// Dot products of one row group held in shared memory, over the chunk quads
// pq = first, first + step, ...: lane (q, r) takes chunk 4 pq + q of row r.
// acc[m][i] collects slot i (codes scaled by 4^i) against activation row m.
template <int MT>
__device__ __forceinline__ void dot_row_group(const uint8_t *wbase,
                                              const int8_t *xs, int kpad,
                                              int chunks, int q, int r,
                                              int first, int step,
                                              int (&acc)[MT][4]) {
  const int quads = (chunks + 3) / 4;
#pragma unroll 2
  for (int pq = first; pq < quads; pq += step) {
    const int j = 4 * pq + q;
    if (j < chunks) {
      const uint4 wv = *reinterpret_cast<const uint4 *>(
          wbase + j * kGroupChunkBytes + r * kChunkBytes);
      const uint32_t wd[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        const uint32_t c0 = wd[t] & 0x03030303u;
        const uint32_t c1 = wd[t] & 0x0c0c0c0cu;
        const uint32_t c2 = wd[t] & 0x30303030u;
        const uint32_t c3 = wd[t] & 0xc0c0c0c0u;
#pragma unroll
        for (int m = 0; m < MT; ++m) {
          // activation words 4t..4t+3 of chunk j: k = 64j + 16t + 4i + b
          const uint4 xv = *reinterpret_cast<const uint4 *>(
              xs + m * kpad + j * kChunkWeights + 16 * t);
          acc[m][0] = dp4a_us(c0, xv.x, acc[m][0]);
          acc[m][1] = dp4a_us(c1, xv.y, acc[m][1]);
          acc[m][2] = dp4a_us(c2, xv.z, acc[m][2]);
          acc[m][3] = dp4a_us(c3, xv.w, acc[m][3]);
        }
      }
    }
  }
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

template <int MT, bool ACC_OUT>
__global__ void __launch_bounds__(288)
gemv_w2a8_tma_kernel(const GemvArgs a, const TmaPlan p) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int warps = blockDim.x >> 5;
  const int consumers = warps - 1;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int S = p.groups_per_stage;
  const int NS = p.stages;
  const int kpad = a.chunks * kChunkWeights;
  const uint32_t group_bytes = uint32_t(a.chunks) * kGroupChunkBytes;
  const uint32_t stage_bytes = uint32_t(S) * group_bytes;
  const SmemLayout L = smem_layout(MT, kpad, stage_bytes, NS, consumers);
  uint8_t *ring = smem + L.ring;
  int8_t *xs = reinterpret_cast<int8_t *>(smem + L.xs);
  int *sx_part = reinterpret_cast<int *>(smem + L.sums) + MT;  // [cons][MT]
  volatile int *abort_flag = sx_part + consumers * MT;
  float *s_sm = reinterpret_cast<float *>(sx_part + consumers * MT + 1);
  float *ws_sm = s_sm + MT;
  int *red = reinterpret_cast<int *>(smem + L.red);
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + L.bars);
  uint64_t *empty = full + NS;

  const int n_stages = (a.n_groups + S - 1) / S;
  const int grid = gridDim.x;
  const int n_local = (n_stages - int(blockIdx.x) + grid - 1) / grid;

  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], p.split ? 1u : uint32_t(S));
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();  // barriers initialised before any copy or wait

  // The first ring fills start before the dependency on earlier work
  // resolves: the weights are static once written (bw_repack synchronises
  // its stream), so only the activations and scales -- which the preceding
  // kernel may produce -- wait for griddepcontrol.wait.
  auto fill = [&](int i) {
    const int s = i % NS;
    const int g0 = (int(blockIdx.x) + i * grid) * S;
    const int g1 = min(g0 + S, a.n_groups);
    const uint32_t bytes = uint32_t(g1 - g0) * group_bytes;
    mbar_arrive_expect_tx(&full[s], bytes);
    bulk_copy_g2s(ring + size_t(s) * stage_bytes,
                  a.w + size_t(g0) * group_bytes, bytes, &full[s]);
  };
  const int early = NS < n_local ? NS : n_local;
  if (warp == consumers && lane == 0) {
    for (int i = 0; i < early; ++i) fill(i);
    for (int i = early; i < n_local && i < 2 * NS; ++i) {  // next ones: L2
      const int g0 = (int(blockIdx.x) + i * grid) * S;
      const int g1 = min(g0 + S, a.n_groups);
      prefetch_l2(a.w + size_t(g0) * group_bytes,
                  uint32_t(g1 - g0) * group_bytes);
    }
  }
  pdl_wait();

  if (warp == consumers) {
    // ---------------------------------------------------------- producer
    pdl_trigger();
    if (lane == 0) {
      int issued = early;
      bool ok = true;
      for (int i = early; i < n_local; ++i) {
        const int s = i % NS;
        if (!mbar_wait(&empty[s], uint32_t((i / NS) - 1) & 1u)) {
          ok = false;
          break;
        }
        fill(i);
        ++issued;
      }
      if (!ok) atomicOr(&g_device_error, 1u);
      // Every issued copy has landed before this thread leaves (normally
      // the consumers have already waited for them; after a time-out they
      // may not have).
      for (int i = max(0, issued - NS); i < issued; ++i)
        if (!mbar_wait(&full[i % NS], uint32_t(i / NS) & 1u))
          atomicOr(&g_device_error, 2u);
    }
    return;
  }

  // ------------------------------------------------------------- consumers
  const int cthreads = consumers * 32;
  // Stage the scales, the activations (zero beyond K) and the per-warp
  // activation sums; all loads are issued before any is used.
  if (!ACC_OUT) {
    if (threadIdx.x < MT) s_sm[threadIdx.x] = a.s[threadIdx.x];
    if (threadIdx.x >= 32 && threadIdx.x < 32 + a.seg.n_ws)
      ws_sm[threadIdx.x - 32] = __bfloat162float(a.ws[threadIdx.x - 32]);
  }
#pragma unroll
  for (int m = 0; m < MT; ++m) {
    int part = 0;
    if (a.vec_x) {
      const uint4 *xrow = reinterpret_cast<const uint4 *>(a.x + size_t(m) * a.x_ld);
      uint4 *dst = reinterpret_cast<uint4 *>(xs + m * kpad);
      for (int v = threadIdx.x; v < kpad / 16; v += cthreads) {
        uint4 x4 = make_uint4(0u, 0u, 0u, 0u);
        if (16 * v < a.K) x4 = __ldg(xrow + v);
        dst[v] = x4;
        part = dp4a_us(0x01010101u, x4.x, part);
        part = dp4a_us(0x01010101u, x4.y, part);
        part = dp4a_us(0x01010101u, x4.z, part);
        part = dp4a_us(0x01010101u, x4.w, part);
      }
    } else {
      const unsigned int *xrow =
          reinterpret_cast<const unsigned int *>(a.x + size_t(m) * a.x_ld);
      uint32_t *dst = reinterpret_cast<uint32_t *>(xs + m * kpad);
      for (int wd = threadIdx.x; wd < kpad / 4; wd += cthreads) {
        uint32_t v = 0u;
        if (4 * wd < a.K) v = __ldg(xrow + wd);
        dst[wd] = v;
        part = dp4a_us(0x01010101u, v, part);
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
      part += __shfl_xor_sync(0xffffffffu, part, o);
    if (lane == 0) sx_part[warp * MT + m] = part;
  }
  if (threadIdx.x == 0) *abort_flag = 0;
  consumer_sync(cthreads);
  int sx[MT];  // sum_k x[m][k] over the whole row
#pragma unroll
  for (int m = 0; m < MT; ++m) {
    sx[m] = 0;
    for (int w = 0; w < consumers; ++w) sx[m] += sx_part[w * MT + m];
  }
  pdl_trigger();  // dependents may start their prologue on free SM slots

  const int q = lane >> 3;  // chunk residue mod 4
  const int r = lane & 7;   // row inside the group

  if (p.split) {
    // One row group per stage; consumer warp w takes chunk quads w, w + 8,
    // ...; row partials meet in shared memory (double-buffered by stage
    // parity, one consumer barrier per stage).
    for (int i = 0; i < n_local; ++i) {
      const int s = i % NS;
      const bool ok =
          __all_sync(0xffffffffu, mbar_wait(&full[s], uint32_t(i / NS) & 1u));
      if (!ok && lane == 0) {
        atomicOr(&g_device_error, 4u);
        *abort_flag = 1;
      }
      int acc[MT][4];
#pragma unroll
      for (int m = 0; m < MT; ++m)
#pragma unroll
        for (int t = 0; t < 4; ++t) acc[m][t] = 0;
      if (ok)
        dot_row_group<MT>(ring + size_t(s) * stage_bytes, xs, kpad, a.chunks,
                          q, r, warp, consumers, acc);
      int *rb = red + (i & 1) * (consumers * MT * 8);
#pragma unroll
      for (int m = 0; m < MT; ++m) {
        const int v = fold_row(acc[m]);
        if (q == 0) rb[(warp * MT + m) * 8 + r] = v;
      }
      // every warp reaches this barrier, also after a time-out
      consumer_sync(cthreads);
      if (*abort_flag) break;
      if (threadIdx.x == 0) mbar_arrive(&empty[s]);  // stage fully read
      if (warp == 0 && lane < 8) {
        const int n = (int(blockIdx.x) + i * grid) * kGroupRows + lane;
        if (n < a.N) {
#pragma unroll
          for (int m = 0; m < MT; ++m) {
            int total = -sx[m];
            for (int w = 0; w < consumers; ++w)
              total += rb[(w * MT + m) * 8 + lane];
            store_row<MT, ACC_OUT>(a, n, m, total, s_sm, ws_sm);
          }
        }
      }
    }
    return;
  }

  // One warp per row group: teams of S warps take every T-th stage.
  const int teams = consumers / S;
  const int team = warp / S;
  const int member = warp % S;

  int my_group = -1;  // row group whose totals this lane keeps
  int my_tot[MT];
#pragma unroll
  for (int m = 0; m < MT; ++m) my_tot[m] = 0;
  int handled = 0;

  auto epilogue = [&]() {
    const int n = my_group * kGroupRows + r;
    if (my_group >= 0 && n < a.N) {
#pragma unroll
      for (int m = 0; m < MT; ++m)
        store_row<MT, ACC_OUT>(a, n, m, my_tot[m], s_sm, ws_sm);
    }
    my_group = -1;
  };

  for (int i = team; i < n_local; i += teams) {
    const int s = i % NS;
    // warp-uniform outcome before any full-mask shuffle below
    if (!__all_sync(0xffffffffu, mbar_wait(&full[s], uint32_t(i / NS) & 1u))) {
      if (lane == 0) atomicOr(&g_device_error, 4u);
      break;
    }
    const int grp = (int(blockIdx.x) + i * grid) * S + member;
    int tot[MT];
#pragma unroll
    for (int m = 0; m < MT; ++m) tot[m] = 0;
    if (grp < a.n_groups) {
      int acc[MT][4];
#pragma unroll
      for (int m = 0; m < MT; ++m)
#pragma unroll
        for (int t = 0; t < 4; ++t) acc[m][t] = 0;
      dot_row_group<MT>(
          ring + size_t(s) * stage_bytes + size_t(member) * group_bytes, xs,
          kpad, a.chunks, q, r, 0, 1, acc);
#pragma unroll
      for (int m = 0; m < MT; ++m) tot[m] = fold_row(acc[m]) - sx[m];
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);
    if (q == (handled & 3)) {
      my_group = grp;
#pragma unroll
      for (int m = 0; m < MT; ++m) my_tot[m] = tot[m];
    }
    ++handled;
    if ((handled & 3) == 0) epilogue();
  }
  if (handled & 3) epilogue();
}

template <int MT, bool ACC>
cudaError_t launch_tma_instance(const TmaPlan &p, const GemvArgs &a,
                                cudaStream_t stream) {
  const int kpad = a.chunks * kChunkWeights;
  const uint32_t stage_bytes =
      uint32_t(p.groups_per_stage) * uint32_t(a.chunks) * kGroupChunkBytes;
  const SmemLayout L =
      smem_layout(MT, kpad, stage_bytes, p.stages, p.consumers);
  static bool configured[64];  // per device: the opt-in smem attribute
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!configured[dev]) {
    e = cudaFuncSetAttribute(gemv_w2a8_tma_kernel<MT, ACC>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             227 * 1024);
    if (e != cudaSuccess) return e;
    configured[dev] = true;
  }
  const int threads = (p.consumers + 1) * 32;
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(
          &per_sm, gemv_w2a8_tma_kernel<MT, ACC>, threads, L.total) !=
          cudaSuccess ||
      per_sm < 1)
    per_sm = 1;
  const int n_stages =
      (a.n_groups + p.groups_per_stage - 1) / p.groups_per_stage;
  const int resident = per_sm * device_sm_count();
  const int grid = n_stages < resident ? n_stages : resident;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid > 0 ? grid : 1);
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = L.total;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, gemv_w2a8_tma_kernel<MT, ACC>, a, p);
}

}  // namespace

bool plan_gemv_tma(int mt, int N, int K, int num_sms, TmaPlan *p) {
  const int chunks = chunks_per_row(K);
  const uint32_t group_bytes = uint32_t(chunks) * kGroupChunkBytes;
  constexpr uint32_t kStageTarget = 24 * 1024;
  constexpr uint32_t kRingBudget = 96 * 1024;   // two CTAs fit in one SM
  constexpr uint32_t kSplitBudget = 48 * 1024;  // four CTAs fit in one SM
  if (mt != 1 && mt != 2 && mt != 4) return false;
  if (group_bytes > kRingBudget / 2) return false;  // K too long: other path
  p->consumers = 8;
  const int64_t groups = padded_rows(N) / kGroupRows;
  // Few row groups (up to four per SM): split each row group's K across all
  // consumer warps, so no warp walks a whole row alone and every CTA
  // finishes its one or two row groups at about the same time.
  if (groups <= 4 * int64_t(num_sms)) {
    p->split = 1;
    p->groups_per_stage = 1;
    const int stages = int(kSplitBudget / group_bytes);
    p->stages = stages < 2 ? 2 : (stages > 4 ? 4 : stages);
    return true;
  }
  // Many row groups: one warp per row group, S row groups per stage, with S
  // small enough that every CTA (about two per SM) still gets eight stages,
  // one per consumer team at least.
  p->split = 0;
  int S = 1;
  while (S < p->consumers && 2 * S * group_bytes <= kStageTarget &&
         groups / (2 * S) >= 16 * int64_t(num_sms))
    S *= 2;
  p->groups_per_stage = S;
  const int stages = int(kRingBudget / (uint32_t(S) * group_bytes));
  p->stages = stages < 2 ? 2 : (stages > 8 ? 8 : stages);
  return true;
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
