// bw_internal.cuh -- declarations shared by the translation units of libbw.
// Nothing here is visible through the C ABI (include/bw.h).
#pragma once

#include <atomic>

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "../../include/bw.h"

namespace bw {

// Device layout geometry (see the layout specification in bw.h).
constexpr int kGroupRows = 8;         // rows per row group
constexpr int kChunkWeights = 64;     // weights per 16-byte chunk
constexpr int kChunkBytes = 16;
constexpr int kGroupChunkBytes = 128; // one chunk of all 8 rows of a group

inline int64_t padded_rows(int N) { return (int64_t(N) + 7) / 8 * 8; }
inline int chunks_per_row(int K) { return (K + 63) / 64; }

// Weight-scale segments passed by value to the kernels.
struct WsSegments {
  int n_ws;
  int bounds[BW_MAX_WS + 1];
};

// Arguments of one GEMV launch over an M-tile of at most 4 rows.
struct GemvArgs {
  const int8_t *x;        // [mt][x_ld]
  const uint8_t *w;       // device layout
  const float *s;         // [mt] (bf16 mode only)
  const __nv_bfloat16 *ws;
  void *out;              // bf16 [mt][out_ld] or int32 [mt][out_ld]
  int K, N;
  int x_ld, out_ld;
  int chunks;             // C = Kpad / 64
  int n_groups;           // Npad / 8
  int passes;             // K passes of warps*jb quads each
  int vec_x;              // x rows are 16-byte aligned and K % 16 == 0
  WsSegments seg;
};

// Launch configuration chosen by the host dispatcher.
struct GemvPlan {
  int mt;      // activation rows per launch (1, 2 or 4)
  int rg;      // row groups per CTA (1, 2 or 4)
  int jb;      // chunk quads per warp and pass (1..4)
  int warps;   // warps per CTA
  int passes;  // K passes
  int grid;    // CTAs
};

// TMA-streamed GEMV (bw_gemv_tma.cu, kernel in bw_pipe.cuh) for M-tiles of
// mt = 1, 2 or 4 rows; pipe_fits() is false where the staged activations
// do not fit in shared memory.
bool pipe_fits(int mt, int K);
cudaError_t launch_gemv_pipe(const GemvArgs &args, int mt, bool acc_out,
                             cudaStream_t stream);
// Device address of the library's error word on the current device (null
// if it cannot be resolved).
unsigned int *device_error_word();
// Launches the bounded-wait self-test kernel (sets bit 8 after ~10 ms).
cudaError_t launch_selftest_wait(cudaStream_t stream);

// Reads and clears the device error word (synchronises `stream`).
cudaError_t read_device_error(cudaStream_t stream, unsigned int *bits);

// Tensor-core GEMV for batched activations (bw_gemv_mma.cu): one launch
// per tile of at most mma_tile_rows(K) activation rows (`rows` valid rows
// at args.x); mma_tile_rows is 0 where the staged tile does not fit.
constexpr int kMmaMinRows = 8;      // M at or above this uses tensor cores
constexpr int kMmaMaxK = 16384;     // fp32 partial sums stay below 2^21
int mma_tile_rows(int K);
cudaError_t launch_gemv_mma(const GemvArgs &args, int rows, bool acc_out,
                            cudaStream_t stream);
// Tensor-core GEMV on tcgen05 (bw_gemv_tc.cu): one launch per tile of at
// most kTcMaxRows activation rows (64-token tiles with deep rings, larger
// tiles with N = 128 MMAs); needs 16-byte aligned activation rows with
// K % 16 == 0 (bulk copies) and K <= kMmaMaxK.
constexpr int kTcMaxRows = 128;
bool tc_fits(const GemvArgs &args);
cudaError_t launch_gemv_tc(const GemvArgs &args, int rows, bool acc_out,
                           cudaStream_t stream);

// Prefill-sized products (bw_gemm.cu): the tokens converted once to fp16
// in the caller's workspace, then 256-token tcgen05 tiles of 128 weight
// rows; needs K <= kMmaMaxK.
size_t gemm_workspace_bytes(int M, int K);
cudaError_t launch_gemm(const GemvArgs &args, int M, bool acc_out,
                        void *workspace, cudaStream_t stream);

// Pair-table (LUT) GEMV (bw_gemv_lut.cu) for M-tiles of mt = 1, 2 or 4
// rows; lut_fits() is false where the tables do not fit in shared memory.
bool lut_fits(int mt, int N, int K);
cudaError_t launch_gemv_lut(const GemvArgs &args, int mt, bool acc_out,
                            cudaStream_t stream);

GemvPlan plan_gemv(int mt, int N, int K, int num_sms);
cudaError_t launch_gemv(const GemvPlan &plan, const GemvArgs &args,
                        bool acc_out, cudaStream_t stream);

cudaError_t launch_quant_act(const float *x, int M, int K, int8_t *q,
                             float *s, cudaStream_t stream);
cudaError_t launch_repack(const uint8_t *canon, int N, int K,
                          uint8_t *packed, unsigned int *bad,
                          cudaStream_t stream);
cudaError_t launch_unrepack(const uint8_t *packed, int N, int K,
                            uint8_t *canon, cudaStream_t stream);
// Absmean ternarisation (bw_quant_weight.cu): synchronises `stream`.
cudaError_t launch_quant_weight(const float *W, int N, int K,
                                const WsSegments &seg, uint8_t *canon,
                                __nv_bfloat16 *ws, cudaStream_t stream);

int device_sm_count();

// Decode attention (bw_attn.cu) for library-internal callers: the checks of
// bw_attn_decode are the caller's; norm_gamma / norm_part (or null) ask for
// the next RMSNorm's per-KV-head statistics of the output.
struct AttnLaunch {
  const __nv_bfloat16 *qkv;
  const int *pos;
  __nv_bfloat16 *kc, *vc;
  float *out;
  void *workspace;  // attn_workspace_bytes, zeroed before its first use
  int H, Hkv, S;
  float theta;
  const float *norm_gamma;
  float2 *norm_part;
  int past_ready;  // BW_ATTN_PAST_READY: *pos and rows < *pos final earlier
  // 0, or the longest context (p + 1) the launch must serve; a shorter one
  // lets a launch of fewer, smaller CTAs serve it (a longer position then
  // reads as outside the cache: zeros and device error bit 16).
  int max_len;
};
size_t attn_workspace_bytes(int H, int Hkv, int D, int S);  // 0: unsupported
bw_status check_attn(int H, int Hkv, int D, int S);
cudaError_t launch_attn(const AttnLaunch &l, cudaStream_t stream);

// The layer stack as one persistent kernel (bw_decoder.cu) for stacks
// without a KV cache.  The table holds the per-layer pointers
// (decoder_upload_table); the exchange buffers (decoder_xch_bytes) are
// zeroed once and the 4 control words set to {1, 0, 0, 0} once, at creation.
struct DecoderLaunch {
  const void *table;
  int n_layers, steps, dim, ffn, n_heads, n_kv;
  float eps;
  const float *h_in;   // [steps][dim]
  float *h_out;        // [steps][dim]
  void *xch;
  unsigned int *ctl;
  const bw_stack_trace *trace;  // or null
};
size_t decoder_xch_bytes(int dim, int ffn);
size_t decoder_table_bytes(int n_layers);
bool decoder_fits(int dim, int ffn, int n_heads, int n_kv, int n_layers);
cudaError_t decoder_upload_table(void *table, int n_layers,
                                 const uint8_t *const *wqkv,
                                 const uint8_t *const *wo,
                                 const uint8_t *const *w13,
                                 const uint8_t *const *w2,
                                 const bw_bf16 *const *ws,
                                 const float *const *gammas);
cudaError_t launch_decoder(const DecoderLaunch &l, cudaStream_t stream);
// Self-test of the decoder's bounded exchange poll (sets bit 64 in ~10 ms).
cudaError_t launch_selftest_poll(cudaStream_t stream);

// Remembers a CUDA error for bw_last_cuda_error() (calling thread).
void record_cuda_error(int err);

// bw_gemv_w2a8 for library-internal callers (same validation and launch).
bw_status gemv_internal(const int8_t *x, const uint8_t *packed, const float *s,
                        const bw_bf16 *ws, const int *ws_bounds, int n_ws,
                        int M, int N, int K, bw_bf16 *y, cudaStream_t stream);

}  // namespace bw
