// Host check of the decode-attention split plans (bw_attn_plan.cuh), built
// with the host compiler by tests/test_attn_plan_host.py.  For each position
// p of caches of several sizes and for each launch shape the kernels use:
//  * every CTA of the launch agrees on valid, solo and the splits in use;
//  * a valid position's shares partition positions 0..p in CTA order, none
//    in use is empty and none is larger than a CTA's staging;
//  * CTAs past the splits in use, and every CTA of an invalid position,
//    get no positions;
//  * a position is valid exactly when it lies in the cache (and, for the
//    cluster kernel, below the launch's cap of CTAs x staging);
//  * the launch shapes serve every context they are chosen for.
// Prints "ok <checks>" and exits 0, or prints the first failures and exits 1.
#include <cstdio>
#include <vector>

#include "bw_attn_plan.cuh"

using namespace bw;

static long g_failures = 0;
static long g_checks = 0;

#define CHECK(cond, ...)                          \
  do {                                            \
    ++g_checks;                                   \
    if (!(cond) && g_failures++ < 20) {           \
      std::printf(__VA_ARGS__);                   \
      std::printf("\n");                          \
    }                                             \
  } while (0)

// The shares of CTAs 0..n_ctas-1 for one position p (plan(c) gives CTA c's).
template <class Plan>
static void check_position(const char *what, int S, int p, int n_ctas,
                           int max_share, bool expect_valid, Plan plan) {
  const SplitPlan first = plan(0);
  CHECK(first.valid == expect_valid, "%s S=%d p=%d: valid %d, expected %d",
        what, S, p, int(first.valid), int(expect_valid));
  if (first.valid)
    CHECK(first.n_eff >= 1 && first.n_eff <= n_ctas,
          "%s S=%d p=%d: %d splits in use of %d", what, S, p, first.n_eff,
          n_ctas);
  int next = 0;
  for (int c = 0; c < n_ctas; ++c) {
    const SplitPlan r = plan(c);
    CHECK(r.valid == first.valid && r.solo == first.solo &&
              r.n_eff == first.n_eff,
          "%s S=%d p=%d: CTA %d disagrees with CTA 0", what, S, p, c);
    if (!r.valid || c >= r.n_eff) {
      CHECK(r.n == 0, "%s S=%d p=%d: CTA %d takes %d positions, none expected",
            what, S, p, c, r.n);
      continue;
    }
    CHECK(r.j0 == next, "%s S=%d p=%d: CTA %d starts at %d, not %d", what, S,
          p, c, r.j0, next);
    CHECK(r.n >= 1 && r.n <= max_share,
          "%s S=%d p=%d: CTA %d takes %d positions (1..%d)", what, S, p, c,
          r.n, max_share);
    next = r.j0 + r.n;
  }
  if (first.valid)
    CHECK(next == p + 1, "%s S=%d p=%d: shares cover %d positions", what, S,
          p, next);
}

// Positions to try for a cache of S: all of them up to 5000, else the first
// 2048, every 97th and the last 300; and the invalid ones around the ends.
static std::vector<int> positions(int S) {
  std::vector<int> ps = {-2, -1, S, S + 1};
  if (S <= 5000) {
    for (int p = 0; p < S; ++p) ps.push_back(p);
  } else {
    for (int p = 0; p < 2048; ++p) ps.push_back(p);
    for (int p = 2048; p < S - 300; p += 97) ps.push_back(p);
    for (int p = S - 300; p < S; ++p) ps.push_back(p);
  }
  return ps;
}

// Workspace kernel: n_split from attn_splits, shares at most kAttnChunk.
static void check_workspace() {
  const int sizes[] = {1,   2,   63,   64,   65,   127,  128,   129,  159,
                       160, 161, 300,  1000, 4096, 4097, 10000, 65536};
  const int kv_heads[] = {1, 5, 8, 32};
  const int sm_counts[] = {1, 16, 152};
  for (int S : sizes)
    for (int Hkv : kv_heads)
      for (int sms : sm_counts) {
        const int n_split = attn_splits(S, Hkv, sms);
        CHECK(n_split >= 1 && n_split <= max_splits(S),
              "workspace S=%d: %d splits, the workspace holds %d", S, n_split,
              max_splits(S));
        CHECK(int64_t(n_split) * kAttnChunk >= S,
              "workspace S=%d: %d splits of %d positions are too few", S,
              n_split, kAttnChunk);
        for (int p : positions(S))
          check_position("workspace", S, p, n_split, kAttnChunk,
                         p >= 0 && p < S,
                         [&](int c) { return ws_plan(p, S, n_split, c); });
      }
}

// Cluster kernel: a launch of cl CTAs with a staging of `chunk` positions
// serves positions below cap = cl * chunk.
static void check_cluster_shape(const char *what, int S, int cl, int chunk,
                                int served) {
  const int cap = cl * chunk;
  CHECK(cl >= 1 && cl <= kClMaxCtas, "%s S=%d: %d CTAs per head", what, S,
        cl);
  CHECK(cap >= served, "%s S=%d: %d x %d positions serve %d", what, S, cl,
        chunk, served);
  for (int p : positions(S)) {
    const bool valid = p >= 0 && p < S && p < cap;
    check_position(what, S, p, cl, chunk, valid,
                   [&](int c) { return cl_plan(p, S, cl, c, cap); });
    const SplitPlan r = cl_plan(p, S, cl, 0, cap);
    CHECK(r.solo == (!valid || p < kClSoloMax), "%s S=%d p=%d: solo %d", what,
          S, p, int(r.solo));
  }
}

// The shapes the launch picks for contexts of at most max_len positions of
// a cache of S: the small staging where max_len < S and it fits, and the
// full staging (which the launch falls back to).  Caches longer than
// kClMaxS take the cluster kernel for short contexts too (a launch that
// serves at most max_len positions); positions past its cap are invalid.
static void check_cluster() {
  const int lens[] = {1,   2,    31,   32,   33,   127,  128,  129,
                      200, 255,  256,  257,  511,  512,  513,  1000,
                      1024, 1025, 2047, 2048, 2049, 3000, 4095, 4096};
  for (int max_len : lens) {
    const int caches[] = {max_len, max_len + 1, kClMaxS, 65536};
    for (int S : caches) {
      if (S < max_len) continue;
      if (max_len <= kClMaxCtas * kClChunkSmall && max_len < S)
        check_cluster_shape("cluster/small", S, cl_ctas_small(max_len),
                            kClChunkSmall, max_len);
      check_cluster_shape("cluster", S, cl_ctas(max_len), kClChunk, max_len);
    }
  }
  // every cluster size with either staging, on caches of several sizes
  for (int cl = 1; cl <= kClMaxCtas; ++cl)
    for (int chunk : {kClChunkSmall, kClChunk}) {
      const int caches[] = {cl * chunk, cl * chunk + 7, kClMaxS, 65536};
      for (int S : caches) check_cluster_shape("cluster/any", S, cl, chunk, 0);
    }
}

int main() {
  check_workspace();
  check_cluster();
  if (g_failures) {
    std::printf("FAILED %ld of %ld checks\n", g_failures, g_checks);
    return 1;
  }
  std::printf("ok %ld\n", g_checks);
  return 0;
}
