// kvq_key_splits.h -- how many CTAs share the key tiles of one (row tile,
// KV head) pair of the prompt-chunk attention.
//
// A chunk with at least as many (row tile, KV head) pairs as SMs fills the
// GPU by itself: one CTA per pair.  A short chunk over a long context would
// leave most SMs idle, each CTA streaming every key tile; its key tiles are
// then split over a cluster of up to kMaxKeySplits CTAs.  The count is the
// one that minimises (waves of clusters) x (key tiles per split) + 2 (the
// merge of a split costs about two tiles), with the waves counted in the
// clusters that can be resident at once; each split keeps at least four
// tiles, and a cluster size that cannot be resident is skipped.  Plain C++
// (no CUDA headers), so the choice is testable on a host without a GPU.
#pragma once

namespace kvq {

constexpr int kMaxKeySplits = 8;  // CTAs of a key-split cluster (the portable maximum)

// base: (row tile, KV head) pairs; n_all: key tiles of the longest row
// tile; sms: multiprocessors; max_clusters(ns): clusters of ns CTAs that can
// be resident at once (0: none).  Returns a count in [1, kMaxKeySplits].
template <class MaxClusters>
int choose_key_splits(long long base, int n_all, int sms, MaxClusters max_clusters) {
  if (sms <= 0 || base >= sms) return 1;
  double best_t = (double)((base + sms - 1) / sms) * n_all;
  int best = 1;
  for (int ns = 2; ns <= kMaxKeySplits && n_all >= 4 * ns; ++ns) {
    const int maxc = max_clusters(ns);
    if (maxc <= 0) continue;
    const double t = (double)((base + maxc - 1) / maxc) * ((n_all + ns - 1) / ns) + 2.0;
    if (t < best_t) {
      best_t = t;
      best = ns;
    }
  }
  return best;
}

}  // namespace kvq
