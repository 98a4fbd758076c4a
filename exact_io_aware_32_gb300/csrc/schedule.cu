// Host-side choice of the CTA order for the attention kernels.
//
// Each kernel's grid is (heads x blocks); CTAs start roughly in increasing
// linear index and each SM takes the next one when its current CTA ends. The
// kernels map the linear index to (head, block) in head groups (see
// block_order.cuh): small groups keep the CTAs that share a head's K/V (or
// Q/dO) tiles resident together, so the tiles are read from DRAM about once,
// but under the causal mask the CTAs of a group differ in cost (block b of n
// sees n - b tiles), and a group that starts late can leave a heavy CTA
// running alone at the end. pick_head_group simulates that greedy dispatch
// for every group size and returns the smallest one whose makespan is within
// 1% of the best. Results are cached per shape.
#include <algorithm>
#include <cstdint>
#include <functional>
#include <map>
#include <mutex>
#include <queue>
#include <tuple>
#include <vector>

#include "fa_internal.h"

namespace fa {
namespace {

// Makespan, in units of one block's work, of dispatching the grid in
// head-group order to num_sms SMs, each CTA costing (its tile count +
// overhead) units.
double simulate(int BH, int nblk, int group, bool causal, int num_sms, double overhead) {
  std::priority_queue<double, std::vector<double>, std::greater<double>> free_at;
  for (int i = 0; i < num_sms; ++i) free_at.push(0.0);
  double makespan = 0.0;
  const long long per_group = (long long)group * nblk;
  const long long total = (long long)BH * nblk;
  for (long long lin = 0; lin < total; ++lin) {
    const long long g = lin / per_group;
    const long long idx = lin - g * per_group;
    const long long gsize = std::min<long long>(group, BH - g * group);
    const int blk = (int)(idx / gsize);  // heaviest block first under the causal mask
    const double cost = (causal ? nblk - blk : nblk) + overhead;
    const double t = free_at.top() + cost;
    free_at.pop();
    free_at.push(t);
    makespan = std::max(makespan, t);
  }
  return makespan;
}

std::mutex g_mu;
std::map<std::tuple<int, int, bool, int, int>, int> g_cache;

}  // namespace

int pick_head_group(int BH, int nblk, bool causal, int num_sms, double overhead) {
  if (BH < 1 || nblk < 1 || num_sms < 1) return 1;
  const int fallback = std::max(1, std::min(BH, num_sms / nblk));
  if (!causal) return 1;  // equal CTAs: any order balances; one head at a time keeps its tiles in L2
  if ((long long)BH * nblk > 262144) return fallback;  // keep the one-off simulation cheap
  const auto key = std::make_tuple(BH, nblk, causal, num_sms, (int)(overhead * 16.0));
  {
    std::lock_guard<std::mutex> lock(g_mu);
    auto it = g_cache.find(key);
    if (it != g_cache.end()) return it->second;
  }
  // Every group size up to 32 heads, then steps of about 1/8, and all heads;
  // each scored by its worst makespan relative to the best over three per-CTA
  // overheads, since the dispatch is sensitive to the exact costs.
  std::vector<int> cand;
  for (int g = 1; g <= BH; g = g < 32 ? g + 1 : g + g / 8) cand.push_back(g);
  if (cand.back() != BH) cand.push_back(BH);
  const double ovh[3] = {0.5 * overhead, overhead, 1.5 * overhead};
  std::vector<double> score(cand.size(), 0.0);
  for (double o : ovh) {
    std::vector<double> span(cand.size());
    double best = 0.0;
    for (size_t i = 0; i < cand.size(); ++i) {
      span[i] = simulate(BH, nblk, cand[i], causal, num_sms, o);
      best = i == 0 ? span[i] : std::min(best, span[i]);
    }
    for (size_t i = 0; i < cand.size(); ++i) score[i] = std::max(score[i], span[i] / best);
  }
  // the smallest group (best L2 reuse) within 1% of the best balance
  int chosen = cand[std::min_element(score.begin(), score.end()) - score.begin()];
  for (size_t i = 0; i < cand.size(); ++i)
    if (score[i] <= 1.01) {
      chosen = cand[i];
      break;
    }
  std::lock_guard<std::mutex> lock(g_mu);
  g_cache[key] = chosen;
  return chosen;
}

int pick_key_splits(int BH, int Nq, int Nk, int num_sms, int rows_per_cta) {
  const long long ctas = (long long)BH * ((Nq + rows_per_cta - 1) / rows_per_cta);  // CTAs without a split
  const int nkv = (Nk + 127) / 128;
  if (num_sms <= 0 || ctas >= num_sms || nkv < 4) return 1;
  // The fewest ranges whose CTAs fill their waves of num_sms CTA slots to 90%
  // (a short last wave would double the time of a bandwidth-bound call), else
  // the best filling; each range at least two key blocks.
  const int cap = (int)std::min<long long>(kMaxKeySplits, nkv / 2);
  int best = 1;
  double best_fill = 0.0;
  for (int n = 1; n <= cap; ++n) {
    const long long total = ctas * n;
    const long long waves = (total + num_sms - 1) / num_sms;
    const double fill = (double)total / (double)(waves * num_sms);
    if (fill >= 0.9) return n;
    if (fill > best_fill) {
      best_fill = fill;
      best = n;
    }
  }
  return best;
}

}  // namespace fa
