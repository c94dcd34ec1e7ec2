// bw_gemv_lut.cu -- the W2A8 GEMV with pre-summed activation tables: the GPU
// restatement of the table-lookup kernels of the microcontroller pages.
//
// Source: "BitNet на микроконтроллерах: как устроен запуск 1.58-битной LLM на
// кластере ESP32-S3", sections "LUT-компиляция" (lut_ctor: the activations of
// a pair of weights are pre-summed into a 16-entry table indexed by the two
// weights' codes) and "Ядро qgemm_lut" (the product as a sum of table
// lookups).  Same result as bw_gemv_w2a8: acc = sum_k w x exactly in int32,
// then the same epilogue.  It exists to compare the table method with the
// dp4a decode on this GPU (bw.h, bw_gemv_w2a8_lut).
//
// Restated for this library's device layout and its pipe kernel
// (bw_pipe.cuh):
//  * In a 32-bit word of codes, byte b holds elements b, b+4, b+8, b+12 of
//    the word's 16 weights at slots 0..3 (the word interleave), so each 4-bit
//    nibble holds the codes of one pair (e, e+4).  The prologue builds, per
//    pair and activation row, the 16 sums
//        T[n] = (n mod 4 - 1) x[e] + (n div 4 - 1) x[e+4],   n = c_e + 4 c_{e+4}
//    (code 3 never occurs: bw_repack rejects it), 32 pairs per 64-weight
//    chunk, 1 KB (plus a bank-spreading pad) of shared memory per chunk of K
//    and row.
//  * The dot product is one table read per nibble, 8 reads and adds per word
//    of 16 weights, where the dp4a decode spends 4 ANDs and 4 dp4a.  For one
//    row the entries are int16.  For 2 and 4 rows, an entry holds every row's
//    value as a uint16 biased by 256, packed in one 32- or 64-bit word: one
//    read serves all rows and one 32-bit add accumulates two of them (the 32
//    reads of a chunk sum to less than 2^16 per half, so no carry crosses
//    into the other half; the bias is removed per chunk).
//  * The weight streaming, the work split, the reduction and the epilogue
//    are the dp4a GEMV's (same kernel template), so a measured difference is
//    the inner loop's.  The rings keep 2 slots per warp to leave room for the
//    tables.
#include "bw_pipe.cuh"

namespace bw {
namespace {

using namespace pipe;

constexpr int kLutSlots = 2;
constexpr int kLutBias = 256;                  // |T| <= 254
// Tables of one chunk and row: 32 pairs x 16 entries x 16 bits = 1 KB, plus
// a pad so that the tables of the 4 consecutive chunks a warp reads at once
// start on different banks (unpadded they map to the same banks): 32 bytes
// for one row (a pair table spans 8 banks), 16 for two (16 banks); none for
// four, whose pair tables span all 32 banks (and whose tables must fit).
constexpr uint32_t kLutTableBytes = 32 * 16 * 2;
template <int MT>
constexpr uint32_t lut_pad() {
  return MT == 1 ? 32u : (MT == 2 ? 16u : 0u);
}

// Prologue: the pair tables of the MT activation rows (zero beyond K) and
// their scales.  The tables already hold signed weights, so the code-sum
// correction of the dp4a path is zero.
template <uint32_t kTabBytes>
struct StageLut {
  const int8_t *x;
  const float *s;  // null in accumulator mode
  int x_ld, K;

  struct Pre {};
  __device__ __forceinline__ Pre pre_wait() const { return Pre{}; }

  template <int MT>
  __device__ __forceinline__ void stage(const Pre &, const StageCtx &c,
                                        int (&part)[MT]) const {
    const float sv = (s && threadIdx.x < MT) ? s[threadIdx.x] : 0.0f;
    const int pairs = c.chunks * 32;
    uint4 *tab = reinterpret_cast<uint4 *>(c.xs);
    constexpr int kChunkVecs = int(kTabBytes) * MT / 16;
    for (int pi = threadIdx.x; pi < pairs; pi += blockDim.x) {
      // pair pi = (chunk j, word t, nibble p): elements e0 = b + 8h and
      // e0 + 4 of word t, b = p mod 4, h = p div 4
      const int j = pi >> 5, t = (pi >> 3) & 3, p = pi & 7;
      const int k0 = 64 * j + 16 * t + (p & 3) + 8 * (p >> 2);
      const int k1 = k0 + 4;
      int x0[MT], x1[MT];
#pragma unroll
      for (int m = 0; m < MT; ++m) {
        x0[m] = k0 < K ? int(x[size_t(m) * x_ld + k0]) : 0;
        x1[m] = k1 < K ? int(x[size_t(m) * x_ld + k1]) : 0;
      }
      // 16 entries x MT rows of 16 bits: 2 MT vectors of 16 bytes
      uint32_t words[8 * MT];
#pragma unroll
      for (int n = 0; n < 16; ++n) {
#pragma unroll
        for (int m = 0; m < MT; ++m) {
          const int v = ((n & 3) - 1) * x0[m] + ((n >> 2) - 1) * x1[m];
          const uint32_t h =
              MT == 1 ? (uint32_t(v) & 0xffffu) : uint32_t(v + kLutBias);
          const int idx = n * MT + m;  // 16-bit element index
          if ((idx & 1) == 0)
            words[idx >> 1] = h;
          else
            words[idx >> 1] |= h << 16;
        }
      }
#pragma unroll
      for (int v = 0; v < 2 * MT; ++v)
        tab[size_t(pi >> 5) * kChunkVecs + (pi & 31) * 2 * MT + v] =
            make_uint4(words[4 * v], words[4 * v + 1], words[4 * v + 2],
                       words[4 * v + 3]);
    }
    if (s && threadIdx.x < MT) c.s_sm[threadIdx.x] = sv;
#pragma unroll
    for (int m = 0; m < MT; ++m) part[m] = 0;
  }
};

// The table-lookup dot product.  acc[m][0] collects row m's sum (the other
// three accumulators of the dp4a layout stay zero).
template <uint32_t kTabBytes>
struct DotLut {
  static constexpr uint32_t kXsChunkBytes = kTabBytes;

  template <int MT>
  __device__ __forceinline__ static void chunk(const uint8_t *wp,
                                               const uint8_t *tc,
                                               int (&acc)[MT][4]) {
    const uint4 wv = *reinterpret_cast<const uint4 *>(wp);
    const uint32_t wd[4] = {wv.x, wv.y, wv.z, wv.w};
    if (MT == 1) {
      const int16_t *t16 = reinterpret_cast<const int16_t *>(tc);
      int a = 0;
#pragma unroll
      for (int t = 0; t < 4; ++t)
#pragma unroll
        for (int p = 0; p < 8; ++p) {
          const int n = int((wd[t] >> (8 * (p & 3) + 4 * (p >> 2))) & 15u);
          a += t16[(t * 8 + p) * 16 + n];
        }
      acc[0][0] += a;
    } else if (MT == 2) {
      const uint32_t *t32 = reinterpret_cast<const uint32_t *>(tc);
      uint32_t pk = 0;
#pragma unroll
      for (int t = 0; t < 4; ++t)
#pragma unroll
        for (int p = 0; p < 8; ++p) {
          const int n = int((wd[t] >> (8 * (p & 3) + 4 * (p >> 2))) & 15u);
          pk += t32[(t * 8 + p) * 16 + n];
        }
      acc[0][0] += int(pk & 0xffffu) - 32 * kLutBias;
      acc[1 % MT][0] += int(pk >> 16) - 32 * kLutBias;
    } else {
      const uint2 *t64 = reinterpret_cast<const uint2 *>(tc);
      uint32_t pa = 0, pb = 0;
#pragma unroll
      for (int t = 0; t < 4; ++t)
#pragma unroll
        for (int p = 0; p < 8; ++p) {
          const int n = int((wd[t] >> (8 * (p & 3) + 4 * (p >> 2))) & 15u);
          const uint2 v = t64[(t * 8 + p) * 16 + n];
          pa += v.x;
          pb += v.y;
        }
      acc[0][0] += int(pa & 0xffffu) - 32 * kLutBias;
      acc[1 % MT][0] += int(pa >> 16) - 32 * kLutBias;
      acc[2 % MT][0] += int(pb & 0xffffu) - 32 * kLutBias;
      acc[3 % MT][0] += int(pb >> 16) - 32 * kLutBias;
    }
  }

  // Lane (q, r) takes chunks c0 + q, c0 + q + 4, ... of row r (as the dp4a
  // policy does).
  template <int MT>
  __device__ __forceinline__ static void run(const uint8_t *wbase,
                                             const int8_t *xs, uint32_t,
                                             int c0, int chunks, int q, int r,
                                             int (&acc)[MT][4]) {
    const uint8_t *wp = wbase + q * kGroupChunkBytes + r * kChunkBytes;
    const uint8_t *tc = reinterpret_cast<const uint8_t *>(xs) +
                        size_t(c0 + q) * kTabBytes * MT;
    const int quads = chunks >> 2;
#pragma unroll 1
    for (int pq = 0; pq < quads; ++pq) {
      chunk<MT>(wp, tc, acc);
      wp += 4 * kGroupChunkBytes;
      tc += 4 * kTabBytes * MT;
    }
    if (q < (chunks & 3)) chunk<MT>(wp, tc, acc);
  }

  __device__ __forceinline__ static int fold(const int (&a)[4]) {
    int v = a[0];
    v += __shfl_xor_sync(0xffffffffu, v, 8);
    v += __shfl_xor_sync(0xffffffffu, v, 16);
    return v;
  }
};

template <int MT, bool ACC>
cudaError_t launch_lut_instance(const GemvArgs &g, cudaStream_t stream) {
  PipeArgs a{};
  a.w = g.w;
  a.N = g.N;
  a.chunks = g.chunks;
  a.n_groups = g.n_groups;
  a.slots = kLutSlots;
  a.err = device_error_word();
  if (!a.err) return cudaErrorInvalidSymbol;
  constexpr uint32_t kBytes = kLutTableBytes + lut_pad<MT>();
  const StageLut<kBytes> pro{g.x, ACC ? nullptr : g.s, g.x_ld, g.K};
  const EpiOut<ACC> epi{g.out, g.out_ld, g.ws, g.seg};
  return launch_pipe<MT, StageLut<kBytes>, EpiOut<ACC>, DotLut<kBytes>>(
      a, pro, epi, stream);
}

}  // namespace

bool lut_fits(int mt, int N, int K) {
  if (mt != 1 && mt != 2 && mt != 4) return false;
  const int sms = device_sm_count();
  if (sms <= 0) return false;
  // the tables allow one CTA per SM: k = ceil(groups / SMs) groups per CTA
  const int64_t groups = padded_rows(N) / kGroupRows;
  int64_t k = (groups + sms - 1) / sms;
  if (k < kPipeMinGroupsPerCta) k = kPipeMinGroupsPerCta;
  if (k > kPipeMaxGroupsPerCta) k = kPipeMaxGroupsPerCta;
  const uint32_t pad = mt == 1 ? lut_pad<1>() : (mt == 2 ? lut_pad<2>()
                                                            : lut_pad<4>());
  return pipe_smem_bytes(mt, chunks_per_row(K), kPipeSlotChunks, kLutSlots,
                         int(k), kLutTableBytes + pad) <= 227u * 1024u;
}

cudaError_t launch_gemv_lut(const GemvArgs &a, int mt, bool acc_out,
                            cudaStream_t stream) {
  if (mt == 1)
    return acc_out ? launch_lut_instance<1, true>(a, stream)
                   : launch_lut_instance<1, false>(a, stream);
  if (mt == 2)
    return acc_out ? launch_lut_instance<2, true>(a, stream)
                   : launch_lut_instance<2, false>(a, stream);
  if (mt == 4)
    return acc_out ? launch_lut_instance<4, true>(a, stream)
                   : launch_lut_instance<4, false>(a, stream);
  return cudaErrorInvalidConfiguration;
}

}  // namespace bw
