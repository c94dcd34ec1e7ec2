// bw_attn_plan.cuh -- how one decode-attention launch splits positions
// 0..p of a KV head's cache over its CTAs (bw_attn.cu).  Integer arithmetic
// only, on the host (launch shapes) and on the device (each CTA's share of
// the position it reads), and plain C++ as well, so that a host program
// can check every share of every position without a GPU.
//
// Sources: "BitNet GPU 推理框架：从零构建 W2A8 的 2-bit 大模型 CUDA GEMV 内核",
// §六 item 2 (a preallocated KV cache; one launch per step, the position
// read on the device).
#pragma once

#include <cstdint>

#ifdef __CUDACC__
#define BW_PLAN_FN __host__ __device__ inline
#else
#define BW_PLAN_FN inline
#endif

namespace bw {

// ---- workspace kernel: splits merged through the caller's workspace ----
constexpr int kAttnChunk = 160;         // positions per split, at most
constexpr int kAttnMinChunk = 64;       // positions per used split, at least
constexpr int kAttnSoloMax = 128;       // contexts one CTA per head finishes

BW_PLAN_FN int max_splits(int S) {
  return (S + kAttnMinChunk - 1) / kAttnMinChunk;
}

// One CTA per SM over the KV heads where the cache is long enough, within
// [ceil(S / kAttnChunk), ceil(S / kAttnMinChunk)].
inline int attn_splits(int S, int Hkv, int sms) {
  const int lo = (S + kAttnChunk - 1) / kAttnChunk;
  const int hi = max_splits(S);
  int n = sms / Hkv;
  if (n > hi) n = hi;
  if (n < lo) n = lo;
  return n < 1 ? 1 : n;
}

// A CTA's share of positions 0..p: n_eff splits in use, positions
// [j0, j0 + n) for this CTA (n = 0: none); valid: p lies in the cache; solo:
// (cluster kernel) CTA 0 finishes the context alone.
struct SplitPlan {
  bool valid, solo;
  int n_eff, j0, n;
};

// Split c of the workspace kernel's n_split: a context of at most
// kAttnSoloMax positions is one split, longer ones take
// min(n_split, ceil(len / kAttnMinChunk)) equal shares.
BW_PLAN_FN SplitPlan ws_plan(int p, int S, int n_split, int c) {
  SplitPlan r{p >= 0 && p < S, false, 0, 0, 0};
  if (r.valid) {
    const int len = p + 1;
    const int want = (len + kAttnMinChunk - 1) / kAttnMinChunk;
    r.n_eff = len <= kAttnSoloMax ? 1 : (want < n_split ? want : n_split);
    if (c < r.n_eff) {
      r.j0 = int(int64_t(c) * len / r.n_eff);
      r.n = int(int64_t(c + 1) * len / r.n_eff) - r.j0;
    }
  }
  return r;
}

// ---- cluster kernel: one thread-block cluster per KV head ----
// A context of at most kClSoloMax positions (and an invalid position) is
// finished by CTA 0 alone, straight from its shared memory, with no cluster
// barrier: the other CTAs leave at once.  Every CTA reads the same position,
// so the choice is the same in the whole cluster, and otherwise every CTA
// executes every cluster barrier on every path: a barrier never waits for a
// CTA that has left.
// The kernel comes in two sizes of a CTA's staging, kClChunk positions
// (caches of up to kClMaxS) and kClChunkSmall (a launch that serves short
// contexts only: less shared memory, so its CTAs fit beside other kernels'
// on an SM); a launch of cl CTAs per KV head serves contexts of at most
// cl * chunk positions.
constexpr int kClMaxCtas = 16;                  // CTAs per KV head
constexpr int kClChunk = 256;                   // positions per CTA, at most
constexpr int kClChunkSmall = 128;
constexpr int kClMinChunk = 32;                 // positions per used CTA
constexpr int kClSoloMax = 128;                 // contexts CTA 0 finishes alone
constexpr int kClMaxS = kClMaxCtas * kClChunk;  // 4096
static_assert(kClSoloMax <= kClChunkSmall, "CTA 0 stages a solo context");

// CTAs per KV head for a cache of S <= kClMaxS positions.
inline int cl_ctas(int S) {
  const int n = (S + kClMinChunk - 1) / kClMinChunk;
  return n < 1 ? 1 : (n > kClMaxCtas ? kClMaxCtas : n);
}

// CTAs per KV head of the smaller staging for contexts of at most max_len
// positions; the launch takes it where max_len is below the cache size and
// at most kClMaxCtas * kClChunkSmall.
inline int cl_ctas_small(int max_len) {
  return (max_len + kClChunkSmall - 1) / kClChunkSmall;
}

// CTA c of a cluster of cl: a context of at most kClSoloMax positions, and
// an invalid position, are CTA 0's alone (solo); longer contexts take
// min(cl, ceil(len / kClMinChunk)) equal shares.  A position is invalid
// outside the cache and past the launch's cap = cl * chunk contexts (which
// keeps every share within a CTA's staging).  Every CTA of the cluster
// reads the same position, so solo is the same in all of them.
BW_PLAN_FN SplitPlan cl_plan(int p, int S, int cl, int c, int cap) {
  SplitPlan r{p >= 0 && p < S && p < cap, false, 0, 0, 0};
  r.solo = !r.valid || p < kClSoloMax;
  if (r.solo) {
    r.n_eff = 1;
    r.n = (r.valid && c == 0) ? p + 1 : 0;
    return r;
  }
  const int len = p + 1;
  const int want = (len + kClMinChunk - 1) / kClMinChunk;
  r.n_eff = want < cl ? want : cl;
  if (c < r.n_eff) {
    r.j0 = int(int64_t(c) * len / r.n_eff);
    r.n = int(int64_t(c + 1) * len / r.n_eff) - r.j0;
  }
  return r;
}

}  // namespace bw

#undef BW_PLAN_FN
