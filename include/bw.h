/*
 * bw.h -- C ABI of libbw, a GB300 (sm_103a) library for the BitNet b1.58
 * ternary-weight x int8-activation (W2A8) linear layer at decode.
 *
 * Sources (page title and section):
 *   [W2A8] "BitNet GPU 推理框架：从零构建 W2A8 的 2-bit 大模型 CUDA GEMV 内核":
 *          §2.2 the kernel's C interface (int8 activations, 4:1 packed ternary
 *          weights, bf16 output, activation scale s, weight scales ws, M, N,
 *          K, stream); §5.1/§5.2 packing, permutation and word interleave;
 *          §5.3 dp4a dot product, shuffle reduction and the scale epilogue;
 *          §六 item 3 the per-row absmax activation quantisation;
 *          §一 and §4.1 the BitNet-2B decoder layer the stack chains.
 *   [ESP]  "Յոթ ESP32-S3 տախտակ ... 1,58 բիթանոց լեզվական մոդել", section
 *          "1,58 բիթ մեկ կշռի համար": ternary weights, four per byte.
 *
 * Conventions for every call:
 *   - Tensor arguments are DEVICE pointers owned by the caller; the library
 *     never frees them and keeps no reference after the call returns.
 *   - Calls are asynchronous on `stream` unless their comment says otherwise;
 *     nothing is synchronised on the GEMV path.
 *   - Arguments are validated on the host before any launch.  A failed check
 *     returns a status and launches nothing.  A launch error is returned as
 *     BW_ERR_CUDA (the CUDA error is then available from cudaGetLastError in
 *     this library's runtime instance via bw_last_cuda_error()).
 *   - bf16 values are passed as their 16-bit patterns (the upper half of an
 *     IEEE fp32 pattern), type bw_bf16; __nv_bfloat16 has the same layout.
 *   - Matrices are row-major.  Sizes are element counts.
 *   - The library keeps per-device state for the life of the process (SM
 *     counts, kernel attributes, the address of its device error word):
 *     resetting a device with cudaDeviceReset while the library is loaded
 *     is not supported.
 *
 * Canonical weight format (input of bw_repack, output of bw_unrepack):
 *   N rows of K/4 bytes; weight w[n][k] in {-1, 0, +1} is stored as the code
 *   c = w + 1 in {0, 1, 2} at bits 2t..2t+1 (t = k mod 4) of byte k/4 of row
 *   n.  Code 3 is invalid.  K must be a multiple of 4.
 *
 * Device weight layout (output of bw_repack, input of the GEMV):
 *   Rows are padded to Npad = ceil(N/8)*8 and K to Kpad = ceil(K/64)*64
 *   with code 1 (weight 0).  A 16-byte chunk holds the 64 weights of one row
 *   with k in [64j, 64j+64) (chunk j).  Its 32-bit word t (bytes 4t..4t+3)
 *   holds k in [64j+16t, 64j+16t+16); element e = k mod 16 of the word sits
 *   in byte (e mod 4) at bits 2*(e div 4) -- the [W2A8] §5.2 word interleave
 *   (field order 0,4,8,12,1,5,9,13,2,6,10,14,3,7,11,15).  Chunks are stored
 *   by groups of 8 rows: chunk (n, j) starts at byte
 *       ((n/8) * C + j) * 128 + (n mod 8) * 16,       C = Kpad/64,
 *   so the 8 rows x Kpad weights of a row group are one contiguous run of
 *   2*Kpad bytes.  Total size: bw_repack_bytes(N, K) = Npad * Kpad / 4.
 */
#ifndef BW_H
#define BW_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* cudaStream_t without requiring the CUDA headers in the caller. */
typedef struct CUstream_st *bw_stream_t;
typedef uint16_t bw_bf16;

typedef enum {
    BW_OK = 0,
    BW_ERR_INVALID_ARG = 1,       /* null pointer, negative size, bad bounds */
    BW_ERR_UNSUPPORTED_SHAPE = 2, /* a size outside the limits below        */
    BW_ERR_MISALIGNED = 3,        /* a pointer without its required alignment */
    BW_ERR_BAD_CODE = 4,          /* a canonical weight code equal to 3      */
    BW_ERR_CUDA = 5,              /* a CUDA runtime call or launch failed    */
    BW_ERR_TIMEOUT = 6            /* a bounded device-side wait gave up      */
} bw_status;

/* Limits checked by every call. */
#define BW_MAX_K 65536      /* reduction length                           */
#define BW_MAX_N (1 << 24)  /* output rows                                */
#define BW_MAX_M 4096       /* activation rows of one GEMV call           */
#define BW_MAX_WS 8         /* weight-scale segments of one GEMV call     */

/* Human-readable name of a status.  Never returns NULL. */
const char *bw_status_string(bw_status status);

/* The CUDA error code of the last BW_ERR_CUDA returned on this thread
 * (cudaSuccess = 0 if none). */
int bw_last_cuda_error(void);

/* Library version, major * 10000 + minor * 100 + patch. */
int bw_version(void);

/* ------------------------------------------------------------------------
 * bw_quant_act -- per-row absmax quantisation of activations to int8.
 * [W2A8] §六 item 3: s = 127 / max|x|, q = round(x * s) clamped to
 * [-128, 127] (round half to even, as PyTorch's round).  The absmax is
 * floored at 1e-5 so an all-zero row gives q = 0 (reading: the floor the
 * page's weight quantiser of §4.2 uses).  fp32 arithmetic throughout.
 *   x  fp32 [M][K] device, 4-byte aligned; finite values.
 *   q  int8 [M][K] device (output).
 *   s  fp32 [M]    device (output): the scale that multiplied x.
 *   1 <= M <= BW_MAX_M, 1 <= K <= BW_MAX_K.
 * ---------------------------------------------------------------------- */
bw_status bw_quant_act(const float *x, int M, int K, int8_t *q, float *s,
                       bw_stream_t stream);

/* ------------------------------------------------------------------------
 * bw_repack -- canonical ternary bytes to the device weight layout
 * (offline, once per weight; [W2A8] §5.1/§5.2 describe the page's own
 * permutation and interleave, which this layout replaces).
 *   canon   uint8 [N][K/4] device, canonical format (any alignment).
 *   packed  uint8 [bw_repack_bytes(N, K)] device, 16-byte aligned (output).
 *   1 <= N <= BW_MAX_N, 4 <= K <= BW_MAX_K, K % 4 == 0.
 * Returns BW_ERR_BAD_CODE if any code is 3 (the output is then undefined).
 * This call allocates a 4-byte status word with cudaMallocAsync on `stream`
 * and SYNCHRONISES `stream` before returning (it is not for the hot path).
 * ---------------------------------------------------------------------- */
size_t bw_repack_bytes(int N, int K);
bw_status bw_repack(const uint8_t *canon, int N, int K, uint8_t *packed,
                    bw_stream_t stream);

/* bw_repack_noalloc -- bw_repack without any device allocation, for
 * callers that are not allowed to allocate device memory (for example an
 * application whose device memory is owned by a host framework's own
 * allocator, or one running with stream-ordered memory pools disabled).
 * The pages have no counterpart: this is a library convenience, not part of
 * the method.  Same arguments, result and limits as bw_repack; sizes beyond
 * BW_MAX_N or BW_MAX_K are rejected with BW_ERR_UNSUPPORTED_SHAPE.
 *   Scratch: instead of allocating its 4-byte bad-code flag, the call uses
 *   a fixed 256-byte array inside the library (every GPU that loads the
 *   library holds it until the process exits; the repack needs one word of
 *   it whatever N and K are).  Each call looks up that array's device
 *   address on the current device.  Every call shares the array and clears
 *   the flag before use, so calls that overlap on the GPU (on different
 *   streams or from different threads) race on it and may report each
 *   other's bad codes: serialise them.  Calls no cudaMalloc, cudaFree or
 *   other allocating routine.  SYNCHRONISES `stream` before returning (it
 *   copies the flag to the host and waits for it), so it must not be called
 *   while `stream` is being captured into a graph. */
bw_status bw_repack_noalloc(const uint8_t *canon, int N, int K,
                            uint8_t *packed, bw_stream_t stream);

/* bw_unrepack -- the inverse of bw_repack: device layout to canonical bytes
 * [N][K/4] (padding is dropped).  Asynchronous; same limits as bw_repack;
 * packed must be 16-byte aligned. */
bw_status bw_unrepack(const uint8_t *packed, int N, int K, uint8_t *canon,
                      bw_stream_t stream);

/* bw_quant_weight -- absmean ternarisation of fp32 weights W [N][K] into the
 * canonical codes [N][K/4] (the input of bw_repack) and one bf16 scale per
 * weight-scale segment ([W2A8] §4.2, the checkpoint conversion): for the
 * rows of segment i, s = 1 / max(mean |W|, 1e-5), w = clamp(round(W s), -1,
 * 1) (nearest, ties to even), ws[i] = bf16(1 / s) (nearest even).  The page
 * leaves the precision open: |W| is summed in fp64 per segment, the mean
 * rounded to fp32, and s, W s and 1 / s are fp32.
 *   W          fp32 [N][K] device, 16-byte aligned.
 *   ws_bounds  int [n_ws + 1] HOST, as for bw_gemv_w2a8 (1 <= n_ws <=
 *              BW_MAX_WS).
 *   canon      uint8 [N][K/4] device (output).
 *   ws         bf16 [n_ws] device, 2-byte aligned (output).
 * Same shape limits as bw_repack.  Offline: it takes a few bytes of device
 * scratch (stream-ordered) and synchronises `stream` before returning. */
bw_status bw_quant_weight(const float *W, int N, int K, const int *ws_bounds,
                          int n_ws, uint8_t *canon, bw_bf16 *ws,
                          bw_stream_t stream);

/* ------------------------------------------------------------------------
 * bw_gemv_w2a8 -- y = bf16( (acc / s[m]) * ws[seg(n)] ),
 *                 acc[m][n] = sum_k w[n][k] * x[m][k]  (exact int32).
 * [W2A8] §2.2 (the interface: int8 x, packed int2 W, bf16 out, s, ws, M,
 * N, K, stream), §5.3 (int32 dp4a accumulation, bf16 epilogue), §4.2 (one
 * weight scale per fused sub-projection).  The page's kernel multiplies by
 * s; with s = 127/absmax (§六 item 3) the dimensionally consistent reading
 * divides, which is what this call does.  Every fp32 step is IEEE (no fast
 * math) and there is a single rounding to bf16, to nearest even.  The
 * tensor-core tiles get the correctly rounded quotient acc / s from a stored
 * RN(1 / s) and a corrected product (Markstein's final step of division),
 * and divide where s lies outside [2^-60, 2^60]; the result is the same.
 *   x          int8 [M][K] device, 4-byte aligned.
 *   packed     device weight layout from bw_repack(N, K), 16-byte aligned.
 *   s          fp32 [M] device: activation scales (as bw_quant_act writes).
 *   ws         bf16 [n_ws] device: weight scales.
 *   ws_bounds  int [n_ws + 1] HOST: 0 = b[0] < b[1] < ... < b[n_ws] = N;
 *              row n uses ws[i] for b[i] <= n < b[i+1] (e.g. the fused
 *              q|k|v projection of BitNet-2B: {0, 2560, 3200, 3840}).
 *   y          bf16 [M][N] device, 2-byte aligned (output).
 *   1 <= M <= BW_MAX_M, 1 <= N <= BW_MAX_N, 4 <= K <= BW_MAX_K, K % 4 == 0,
 *   1 <= n_ws <= BW_MAX_WS.  M < 8: activation rows in tiles of 4, 2 and
 *   1 on CUDA cores (int dp4a).  M >= 8: tiles of up to 128 rows on the
 *   tensor cores (tcgen05.mma; mma.sync where x is not 16-byte aligned or
 *   K % 16 != 0), exact in int32 as well.  The weights are streamed once
 *   per tile.
 * Ordering: the call is launched with programmatic dependent launch, so it
 * may start while the preceding work on `stream` is still running.  x, s,
 * ws and y are touched only after that work has completed; `packed` may be
 * read earlier.  So `packed` must not be written by work still in flight on
 * `stream` (weights are static once bw_repack, which synchronises, has
 * returned; order any later writer with an event or a synchronisation).
 * ---------------------------------------------------------------------- */
bw_status bw_gemv_w2a8(const int8_t *x, const uint8_t *packed, const float *s,
                       const bw_bf16 *ws, const int *ws_bounds, int n_ws,
                       int M, int N, int K, bw_bf16 *y, bw_stream_t stream);

/* bw_gemv_w2a8_acc -- the exact int32 accumulators acc[M][N] of the same
 * product, without scales (the page's exact-int32 test of §三).  acc is
 * int32 [M][N] device, 4-byte aligned.  Same limits as bw_gemv_w2a8. */
bw_status bw_gemv_w2a8_acc(const int8_t *x, const uint8_t *packed, int M,
                           int N, int K, int32_t *acc, bw_stream_t stream);

/* bw_gemv_w2a8_lut, bw_gemv_w2a8_lut_acc -- the same products as
 * bw_gemv_w2a8 and bw_gemv_w2a8_acc (identical int32 accumulators, identical
 * bf16 outputs), computed with pre-summed activation tables instead of the
 * dp4a decode: the GPU restatement of the table-lookup kernels of "BitNet на
 * микроконтроллерах: как устроен запуск 1.58-битной LLM на кластере
 * ESP32-S3" (sections "LUT-компиляция" and "Ядро qgemm_lut").  For every pair
 * of activations whose weights share a 4-bit nibble of the device layout,
 * the kernel first builds the 16 sums (c0 - 1) x0 + (c1 - 1) x1 over the
 * codes, then adds one table entry per nibble.  Same arguments, layouts,
 * ordering and limits as bw_gemv_w2a8, except that the tables of one
 * activation row take K bytes x 16 of shared memory: rows are taken in tiles
 * of 4, 2 and 1, and a tile whose tables do not fit (K above about 10000 at
 * one row, about 2600 at four) returns BW_ERR_UNSUPPORTED_SHAPE before any
 * launch.  Provided to compare the table method with the dp4a decode; the
 * dp4a path is faster on this GPU at every measured M. */
bw_status bw_gemv_w2a8_lut(const int8_t *x, const uint8_t *packed,
                           const float *s, const bw_bf16 *ws,
                           const int *ws_bounds, int n_ws, int M, int N, int K,
                           bw_bf16 *y, bw_stream_t stream);
bw_status bw_gemv_w2a8_lut_acc(const int8_t *x, const uint8_t *packed, int M,
                               int N, int K, int32_t *acc,
                               bw_stream_t stream);

/* bw_gemv_workspace_bytes -- device scratch a bw_gemv_w2a8 call of this
 * shape needs from the caller: always 0.  Every kernel reduces its partial
 * sums in shared memory (int32 atomics per CTA) and no CTA shares a row with
 * another, so there is no split-K workspace and no cross-CTA reduction
 * (the pages' kernel has none either: [W2A8] §5.3 reduces inside a block).
 * Kept so that callers that size a workspace per shape keep working. */
size_t bw_gemv_workspace_bytes(int M, int N, int K);

/* ------------------------------------------------------------------------
 * bw_gemm_w2a8, bw_gemm_w2a8_acc -- the same products as bw_gemv_w2a8 and
 * bw_gemv_w2a8_acc (identical int32 accumulators, identical bf16 outputs)
 * for prefill-sized batches of tokens.  [W2A8] §一 runs prefill and decode
 * as separate paths (the page's prefill is a BF16 matmul); this is the
 * prefill product in W2A8, with the §5.3 exact int32 accumulation and
 * epilogue and the §4.2 weight-scale segments.
 * Two launches on `stream`: the tokens are first written once into
 * `workspace` as the tensor cores' fp16 operand (plus their sums), then
 * each CTA multiplies 128 weight rows by 256 tokens over all K (tcgen05.mma,
 * M = 128, N = 256, fp32 accumulators exact by construction), so every
 * decoded weight serves 256 tokens.
 *   x, packed, s, ws, ws_bounds, n_ws, M, N, K, y, acc: as for
 *              bw_gemv_w2a8 / bw_gemv_w2a8_acc (same layouts, alignment,
 *              limits), and K <= 16384.
 *   workspace  device scratch of at least bw_gemm_workspace_bytes(M, K)
 *              bytes, 256-byte aligned, owned by the caller; overwritten.
 *              It must not be in use by work still in flight elsewhere.
 * Any M >= 1 is accepted; it pays off from a few hundred tokens (for fewer,
 * bw_gemv_w2a8 takes 64- or 128-token tiles).  Errors: BW_ERR_INVALID_ARG
 * (null pointer, bad segments, workspace too small), BW_ERR_MISALIGNED,
 * BW_ERR_UNSUPPORTED_SHAPE (K % 4 != 0, K > 16384, M, N beyond the limits),
 * BW_ERR_CUDA; nothing is launched on an error.  Ordering as for
 * bw_gemv_w2a8 (programmatic dependent launch; `packed` may be read before
 * the preceding work on `stream` completes).
 * ---------------------------------------------------------------------- */
size_t bw_gemm_workspace_bytes(int M, int K);
bw_status bw_gemm_w2a8(const int8_t *x, const uint8_t *packed, const float *s,
                       const bw_bf16 *ws, const int *ws_bounds, int n_ws,
                       int M, int N, int K, bw_bf16 *y, void *workspace,
                       size_t workspace_bytes, bw_stream_t stream);
bw_status bw_gemm_w2a8_acc(const int8_t *x, const uint8_t *packed, int M,
                           int N, int K, int32_t *acc, void *workspace,
                           size_t workspace_bytes, bw_stream_t stream);

/* ------------------------------------------------------------------------
 * Decoder layer stack: chained M=1 W2A8 GEMVs with the fp32 glue between
 * them, in the order of the BitNet b1.58 block ([W2A8] §一 model shape,
 * §4.1 fused projections and the four RMSNorms, §六 item 3 the per-token
 * quantisation before each GEMV, §六 item 1 decode replayed from a graph):
 *   h += down(previous layer)
 *   qkv  = W2A8(quant(rmsnorm(h) * g_attn),            wqkv)   3 scales
 *   o    = W2A8(quant(rmsnorm(attn(qkv)) * g_attn_sub), wo)     1 scale
 *   h   += o
 *   gu   = W2A8(quant(rmsnorm(h) * g_ffn),              w13)    2 scales
 *   down = W2A8(quant(rmsnorm(relu(gate)^2 * up) * g_ffn_sub), w2) 1 scale
 * and, after the last layer, h += down.  attn() is attention over a
 * one-token context: query head i returns the value vector of KV head
 * i / (n_heads / n_kv_heads) (the softmax of a single score is 1); q and k
 * are computed but do not change the result.  RMSNorm:
 * v * (1/sqrt(mean(v^2) + eps)) * gamma, fp32.  The residual stream h is
 * fp32; GEMV outputs are bf16.  The wo and w2 GEMVs add their outputs into
 * h (so h += down happens at the end of each layer, which is the same sum).
 * Execution of a stack without a KV cache (bw_stack_create): ONE persistent
 * cooperative kernel per bw_layer_stack call runs every step, with one CTA
 * per SM; each CTA streams its share of every GEMV's weights ahead of time
 * and receives each GEMV's input from the other CTAs through exchange
 * buffers polled with bounded waits (bw_device_error bit 32 if one runs
 * out).  It needs n_layers <= 128 and the shapes to fit one CTA per SM
 * (every BitNet-2B-sized shape does); a stack that does not fit, and a
 * stack with a KV cache, run as one kernel launch per GEMV (and one per
 * attention) instead, each step replayed from a CUDA graph.  In both, every
 * CTA reduces the norm statistics in a fixed order, so every CTA gets the
 * same codes.  The fp32 sums run in a different order than a sequential
 * loop, so results match a reference within rounding, not bit for bit.
 * ---------------------------------------------------------------------- */
typedef struct bw_stack bw_stack;

typedef struct {
    int n_layers;
    int dim;          /* model width (multiple of n_heads and of 4, <= 8192) */
    int ffn;          /* FFN width (multiple of 8, <= 8192)                  */
    int n_heads;      /* query heads                                         */
    int n_kv_heads;   /* KV heads (divides n_heads)                          */
    float eps;        /* RMSNorm epsilon                                     */
    /* Host arrays of n_layers DEVICE pointers (16-byte aligned), each a
     * device weight layout written by bw_repack:
     *   wqkv [(n_heads + 2 n_kv_heads) * dim/n_heads][dim]  (q | k | v rows)
     *   wo   [dim][dim]
     *   w13  [2 ffn][dim]                                   (gate | up rows)
     *   w2   [dim][ffn]                                                    */
    const uint8_t *const *wqkv;
    const uint8_t *const *wo;
    const uint8_t *const *w13;
    const uint8_t *const *w2;
    /* Host array of n_layers device pointers to 7 bf16 weight scales:
     * q, k, v, o, gate, up, down. */
    const bw_bf16 *const *ws;
    /* Host array of n_layers device pointers (16-byte aligned) to
     * 3 dim + ffn fp32 gains: attention_norm, attn_sub_norm, ffn_norm (dim
     * each), ffn_sub_norm. */
    const float *const *gammas;
} bw_stack_desc;

/* Optional per-stage record of one layer of the LAST step of a
 * bw_layer_stack call (device buffers; any pointer may be NULL). */
typedef struct {
    int layer;
    float *h_in;                     /* [dim] layer input (after residual) */
    int8_t *q_attn; float *s_attn;   /* [dim], [1]                         */
    bw_bf16 *qkv;                    /* [(n_heads + 2 n_kv) hd]            */
    int8_t *q_o; float *s_o;         /* [dim], [1]                         */
    bw_bf16 *o;                      /* [dim]                              */
    float *h_mid;                    /* [dim] h + o                        */
    int8_t *q_ffn; float *s_ffn;     /* [dim], [1]                         */
    bw_bf16 *gu;                     /* [2 ffn]                            */
    int8_t *q_down; float *s_down;   /* [ffn], [1]                         */
    bw_bf16 *down;                   /* [dim]                              */
    float *attn;                     /* [dim] attention output: the fp32
                                        input of attn_sub_norm             */
} bw_stack_trace;

/* Creates a stack: copies the descriptor (the pointer arrays; the weights
 * stay the caller's and must outlive the stack), allocates its device
 * scratch (about 14 dim + 8 ffn bytes of activations plus 32 KB) with
 * cudaMalloc,
 * runs one step on zero input and captures one step as a CUDA graph on a
 * private stream.  Synchronising; call it before any stream capture. */
bw_status bw_stack_create(const bw_stack_desc *desc, bw_stack **stack);

/* bw_stack_create_kv -- the same stack with grouped-query attention over a
 * KV cache in place of the one-token attention: per layer, after the wqkv
 * launch, one bw_attn_decode-style launch rotates the token's new key and
 * query heads (RoPE base theta), appends key and value at the current
 * position p of the layer's bf16 cache and attends over positions 0..p
 * ([W2A8] §一 head counts, §4.1 RoPE on adjacent pairs, §六 item 2 the
 * preallocated cache).  Five launches per layer.  The position starts at 0
 * and advances by one per decode step, so consecutive bw_layer_stack steps
 * (and calls) are consecutive tokens of one sequence; a step at position
 * max_positions or beyond sets bit 16 of the device error word and gives
 * zero attention.  Needs dim / n_heads == 128, n_heads / n_kv_heads in {1,
 * 2, 4, 8}, 1 <= max_positions <= BW_ATTN_MAX_S, theta > 0.  Allocates
 * 2 n_layers n_kv_heads max_positions 128 bf16 of cache with cudaMalloc
 * (zeroed) besides the scratch of bw_stack_create.  It captures one step per
 * context bucket (contexts up to 128 and up to 1024 positions where the
 * cache is longer, then any); the stack counts its tokens on the host (reset
 * by bw_stack_reset_kv) and replays the graph of the token's bucket, whose
 * attention launches have fewer and smaller CTAs for short contexts.  The
 * kernels read the position from device memory: write it only through this
 * API.  Synchronising; call it before any stream capture. */
bw_status bw_stack_create_kv(const bw_stack_desc *desc, int max_positions,
                             float theta, bw_stack **stack);

/* Copies layer `layer`'s key and value caches (bf16 [n_kv_heads]
 * [max_positions][128] each) into k_out and v_out (device, 2-byte aligned),
 * asynchronously on `stream`.  Only for stacks made by bw_stack_create_kv. */
bw_status bw_stack_read_kv(const bw_stack *stack, int layer, bw_bf16 *k_out,
                           bw_bf16 *v_out, bw_stream_t stream);

/* Sets the position of a KV stack back to 0 (a new sequence), on `stream`.
 * The cache rows are not cleared: rows at and past the position are never
 * read. */
bw_status bw_stack_reset_kv(bw_stack *stack, bw_stream_t stream);

/* Runs `steps` decode steps: h_out[t] = stack(h_in[t]) (fp32 [steps][dim],
 * device).  Steps are independent (no KV cache) for a stack made by
 * bw_stack_create; for one made by bw_stack_create_kv they are consecutive
 * tokens of one sequence.  Asynchronous on `stream`.  For a stack without a
 * KV cache the call is one kernel launch, which may be captured in a CUDA
 * graph and replayed (its exchange epochs live in device memory).
 * `trace` (may be NULL) records the stages of trace->layer in the last
 * step.  Calls on the same stack must not overlap (they share its scratch);
 * use one stack per concurrent stream. */
bw_status bw_layer_stack(bw_stack *stack, const float *h_in, int steps,
                         float *h_out, const bw_stack_trace *trace,
                         bw_stream_t stream);

/* Frees the scratch and the graphs (synchronises the device through
 * cudaFree).  NULL is accepted. */
void bw_stack_destroy(bw_stack *stack);

/* ------------------------------------------------------------------------
 * bw_attn_decode -- one decode step of grouped-query attention for one
 * sequence over a bf16 KV cache, in the shape of the BitNet-2B decoder
 * ([W2A8] §一: 20 query heads over 5 KV heads of 128 dims; §4.1: the
 * model's RoPE turns adjacent pairs of head dims; §六 item 2: the KV cache
 * is preallocated and attention takes a flash path).  With G = H / Hkv and
 * p = *pos:
 *   1. the new key of KV head g (k = qkv[H D + g D ..]) is rotated at
 *      position p and written to k_cache[g][p] (rounded to bf16, nearest
 *      even); the new value (qkv[(H + Hkv) D + g D ..]) is written to
 *      v_cache[g][p] as it is;
 *   2. query head h (qkv[h D ..]) is rotated at p and reads KV head h / G;
 *   3. out[h] = sum_j softmax_j(q'.k_cache[h/G][j] / sqrt(D)) v_cache[h/G][j]
 *      over j = 0..p.
 * RoPE: pair (x[2i], x[2i+1]) turns by the angle p * f_i, f_i =
 * theta^(-2i/D); f_i is rounded to fp32 and the angle is the fp32 product
 * (the pages give neither the base theta nor the precision; theta is an
 * argument).  Scores, softmax and sums are fp32.
 *   qkv       bf16 [(H + 2 Hkv) D] device, 2-byte aligned: q | k | v, the
 *             fused wqkv output of the layer.
 *   pos       int32 [1] device: the position p of the new token; read on the
 *             device, so a graph replay serves every step.  p outside
 *             [0, S) writes zeros to out, leaves the cache alone and sets
 *             bit 16 of the device error word (bw_device_error then returns
 *             BW_ERR_INVALID_ARG).
 *   k_cache, v_cache  bf16 [Hkv][S][D] device, 16-byte aligned; rows 0..p-1
 *             hold the earlier tokens (keys rotated); row p is written.
 *   out       fp32 [H][D] device, 4-byte aligned.
 *   workspace device scratch of at least bw_attn_workspace_bytes(H, Hkv, D,
 *             S) bytes, 16-byte aligned, owned by the caller.  Zero it once
 *             before its first use: it holds one counter per KV head, and
 *             every call leaves them at zero again.  Calls sharing a
 *             workspace must not overlap on the GPU.  For S <= 4096 the
 *             splits of a KV head run as one thread-block cluster and merge
 *             through distributed shared memory, leaving the workspace
 *             untouched; it is required all the same.
 *   D == 128; G in {1, 2, 4, 8}; 1 <= Hkv <= BW_ATTN_MAX_KV_HEADS;
 *   1 <= S <= BW_ATTN_MAX_S; theta > 0 (host, fp32).
 * Ordering: launched with programmatic dependent launch; every input is
 * read after the preceding work on `stream` has completed.  Asynchronous;
 * allocates nothing.
 * ---------------------------------------------------------------------- */
#define BW_ATTN_MAX_S 65536
#define BW_ATTN_MAX_KV_HEADS 64
size_t bw_attn_workspace_bytes(int H, int Hkv, int D, int S);
bw_status bw_attn_decode(const bw_bf16 *qkv, const int *pos, int H, int Hkv,
                         int D, int S, float theta, bw_bf16 *k_cache,
                         bw_bf16 *v_cache, float *out, void *workspace,
                         size_t workspace_bytes, bw_stream_t stream);

/* bw_attn_decode_ex -- bw_attn_decode with flags; flags 0 is bw_attn_decode.
 *   BW_ATTN_PAST_READY: the caller promises that *pos and rows 0..p-1 of
 *     both caches are final before the launch immediately preceding this
 *     one on `stream` starts: no work still running when that launch may
 *     start writes them.  The call then reads the position and starts
 *     copying those rows before it waits for the preceding launch (the
 *     layer's past is static during a decode step, like the weights); q|k|v
 *     and everything the call writes keep the ordering above.  A decoder
 *     meets it when the position and the earlier rows are written by the
 *     previous step and the launch before the attention releases its
 *     dependents only after its own dependency wait, as the M = 1 q|k|v
 *     GEMV (bw_gemv_w2a8) and this call do.  The position is read again
 *     after the wait and decides the result; if this CTA's rows differ, the
 *     early copies are discarded, the rows copied again and bit 128 of the
 *     device error word set.  A broken promise about the rows gives the
 *     attention over stale rows, never an access outside the caches.
 * Unknown flag bits return BW_ERR_INVALID_ARG.  Otherwise as
 * bw_attn_decode. */
#define BW_ATTN_PAST_READY 1u
bw_status bw_attn_decode_ex(const bw_bf16 *qkv, const int *pos, int H,
                            int Hkv, int D, int S, float theta,
                            bw_bf16 *k_cache, bw_bf16 *v_cache, float *out,
                            void *workspace, size_t workspace_bytes,
                            unsigned int flags, bw_stream_t stream);

/* bw_device_error -- reads and clears the library's device error word.
 * Kernels that wait on an mbarrier or poll for another CTA's data bound
 * every wait (about one second); a wait that runs out sets a bit here and
 * the kernel stops early instead of hanging (bit 2: a lane gave up waiting
 * for the copies it issued before leaving; bit 4: a warp gave up waiting
 * for a weight piece; bit 32: a CTA of the persistent decoder stack gave
 * up waiting for another CTA's output, or saw another CTA give up; bits 8
 * and 64 are the self-test's).  Bit 16: bw_attn_decode was given a position
 * outside its cache.  Bit 128: bw_attn_decode_ex with BW_ATTN_PAST_READY
 * read a different position after its dependency wait than before it (the
 * promise was broken; the call used the later one).
 * Returns BW_ERR_TIMEOUT if any bit other than 16 and 128 was set, else
 * BW_ERR_INVALID_ARG if bit 16 or 128 was, else BW_OK; *bits receives the
 * word.
 * SYNCHRONISES `stream`; not for the hot path. */
bw_status bw_device_error(unsigned int *bits, bw_stream_t stream);

/* bw_selftest_wait_timeout -- failure-detection self-test of both kinds of
 * bounded wait.  It launches (1) a one-thread kernel whose mbarrier wait
 * cannot complete (it expects two arrivals and receives one) and (2) a
 * kernel that polls, with the persistent decoder's poll routine, exchange
 * entries that nothing writes; each has a limit of about 10 ms.  Both waits
 * run out; the kernels set bits 8 and 64 of the device error word and
 * return; this call then reads and clears the word like bw_device_error and
 * returns BW_ERR_TIMEOUT (with *bits = 8 | 64) -- the expected outcome.  The
 * context stays usable.  SYNCHRONISES `stream`. */
bw_status bw_selftest_wait_timeout(unsigned int *bits, bw_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* BW_H */
