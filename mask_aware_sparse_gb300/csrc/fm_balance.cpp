// fm_balance.cpp — sparsity-aware chunk balancing for context parallelism (host code).
//
// What it computes: FlashMask-3 project page, §3.3 ("Balance the work, not the
// length"). The query axis is cut into n = P * kappa chunks, each rank takes
// exactly kappa of them, and the load of a chunk comes from the tile cost model
// {0, alpha_p, alpha_u} (skipped, partial, unmasked tile). Stage 1 of HCC-IPO
// minimises the makespan Phi = max_j L_j with LPT, then exact pairwise (P2)
// and exact three-rank (P3) repartition, and certifies the result optimal when
// Phi reaches LB = max(ceil(sum w / P), max w) (§3.3 and the "IPO phase
// ablation" table of §4).
//
// A second lower bound uses the cardinality constraint the first one ignores
// (pigeonhole; not on the pages): with the chunks sorted ascending, the m
// lightest are held by at most m ranks, so at least P - m ranks hold none of
// them and carry at least the (P - m) * kappa lightest of the rest, hence
//   Phi >= ceil(sum of sorted w[m .. m + (P - m) * kappa) / (P - m)),  0 <= m < P,
// and the rank holding the heaviest chunk also holds kappa - 1 others:
//   Phi >= max w + sum of the kappa - 1 lightest.
// Their maximum, LB_kappa >= LB (m = 0 is ceil(sum w / P)), is the certificate
// and the stopping point of every phase; it proves optimal, for example, a
// sliding-window mask's split, where equal chunks leave LB unreachable.
//
// The pages give the phases, not their details; the rules fixed here:
//   * LPT: chunks by load descending (ties: lower index first), each to the
//     least-loaded rank holding fewer than kappa chunks (ties: lower rank).
//   * A repartition pools the k * kappa chunks of k ranks (k = 2 or 3) and
//     deals them out again, kappa each, minimising the group's largest load;
//     it is applied only when that is strictly below the group's current
//     largest load. Among the best deals the first is taken in this order:
//     pool by chunk index, the first rank's set over the kappa-combinations of
//     the pool in lexicographic order, the second rank's over those of the
//     rest, the last rank takes what is left.
//   * Only groups holding a rank at the current makespan are visited (no other
//     group can lower it), in lexicographic order of rank indices; a sweep
//     visits each such group once and applies improvements as found. P2 sweeps
//     until a sweep moves nothing; P3 alternates a triple sweep with P2 run to
//     its end until a triple sweep moves nothing. Every phase stops at
//     Phi == LB_kappa.
//
// The exact repartition is a depth-first branch and bound that walks the deals
// in the order above. It prunes only subtrees that hold no deal below the
// current best (a set already too heavy, or too light to leave the other
// ranks below it), so the first deal it records at the optimal value is the
// first optimal deal in that order, and it stops once the group's own lower
// bound max(ceil(T / k), max w) is reached. A node budget bounds the work per
// group; a group whose search runs out of budget is left as it was and the
// report says so.
#include <algorithm>
#include <climits>
#include <cstdint>
#include <vector>

#include "fm.h"

namespace {

constexpr int64_t kDefaultNodeBudget = 4000000;

// Branch and bound over the deals of one group.
class DealSearch {
 public:
  DealSearch(const std::vector<int64_t>& wp, int k, int kappa, int64_t bar, int64_t budget)
      : wp_(wp), m_(static_cast<int>(wp.size())), k_(k), kappa_(kappa), best_(bar), budget_(budget) {
    int64_t total = 0, wmax = 0;
    for (int64_t x : wp_) {
      total += x;
      wmax = std::max(wmax, x);
    }
    total_ = total;
    floor_ = std::max((total + k - 1) / k, wmax);
    cur_.assign(k, std::vector<int>());
    best_sets_.assign(k, std::vector<int>());
  }

  // True when a deal strictly below the bar was found (then set(s) holds the
  // pool positions of rank s of the group, ascending).
  bool run() {
    if (floor_ >= best_) return false;  // nothing can beat the bar
    level(0, 0ull, total_, 0);
    return found_ && !aborted_;
  }
  bool aborted() const { return aborted_; }
  const std::vector<int>& set(int s) const { return best_sets_[s]; }

 private:
  // One rank of the group: choose its kappa positions among the unused ones.
  struct Level {
    std::vector<int> avail;               // unused pool positions, ascending
    std::vector<int64_t> lo_sum, hi_sum;  // [t * (kappa + 1) + j]: sum of the j lightest / heaviest of avail[t..]
  };

  void level(int s, uint64_t used, int64_t rest, int64_t prev_max) {
    if (s == k_ - 1) {  // the last rank takes what is left
      std::vector<int>& last = cur_[s];
      last.clear();
      for (int p = 0; p < m_; ++p)
        if (!((used >> p) & 1ull)) last.push_back(p);
      record(std::max(prev_max, rest));
      return;
    }
    Level L;
    for (int p = 0; p < m_; ++p)
      if (!((used >> p) & 1ull)) L.avail.push_back(p);
    const int r = static_cast<int>(L.avail.size());
    const int K1 = kappa_ + 1;
    L.lo_sum.assign(static_cast<size_t>(r + 1) * K1, 0);
    L.hi_sum.assign(static_cast<size_t>(r + 1) * K1, 0);
    std::vector<int64_t> suffix;  // weights of avail[t..], ascending
    for (int t = r - 1; t >= 0; --t) {
      const int64_t x = wp_[L.avail[t]];
      suffix.insert(std::upper_bound(suffix.begin(), suffix.end(), x), x);
      const int n = static_cast<int>(suffix.size());
      for (int j = 1; j <= kappa_; ++j) {
        L.lo_sum[t * K1 + j] = (j <= n) ? L.lo_sum[t * K1 + j - 1] + suffix[j - 1] : LLONG_MAX / 4;
        L.hi_sum[t * K1 + j] = (j <= n) ? L.hi_sum[t * K1 + j - 1] + suffix[n - j] : LLONG_MAX / 4;
      }
    }
    cur_[s].clear();
    dfs(L, s, 0, 0, used, rest, prev_max);
  }

  // positions avail[t..] still open for rank s; cnt chosen so far with sum x
  void dfs(const Level& L, int s, int t, int64_t x, uint64_t used, int64_t rest, int64_t prev_max) {
    if (done_ || aborted_) return;
    if (++nodes_ > budget_) {
      aborted_ = true;
      return;
    }
    const int cnt = static_cast<int>(cur_[s].size());
    const int q = k_ - s - 1;  // ranks after this one
    if (cnt == kappa_) {
      if (x >= best_) return;
      const int64_t rem = rest - x;
      if (rem > static_cast<int64_t>(q) * (best_ - 1)) return;  // some later rank would reach best
      uint64_t u = used;
      for (int p : cur_[s]) u |= 1ull << p;
      level(s + 1, u, rem, std::max(prev_max, x));
      return;
    }
    const int need = kappa_ - cnt;
    const int r = static_cast<int>(L.avail.size());
    if (r - t < need) return;
    const int K1 = kappa_ + 1;
    if (x + L.lo_sum[t * K1 + need] >= best_) return;                                   // too heavy
    if (x + L.hi_sum[t * K1 + need] < rest - static_cast<int64_t>(q) * (best_ - 1)) return;  // too light
    // take avail[t] first: the deals that hold it come first in the order
    cur_[s].push_back(L.avail[t]);
    dfs(L, s, t + 1, x + wp_[L.avail[t]], used, rest, prev_max);
    cur_[s].pop_back();
    if (done_ || aborted_) return;
    dfs(L, s, t + 1, x, used, rest, prev_max);
  }

  void record(int64_t value) {
    if (value >= best_) return;
    best_ = value;
    found_ = true;
    best_sets_ = cur_;
    if (best_ <= floor_) done_ = true;
  }

  const std::vector<int64_t>& wp_;
  int m_, k_, kappa_;
  int64_t total_ = 0, floor_ = 0, best_;
  int64_t nodes_ = 0, budget_;
  bool found_ = false, done_ = false, aborted_ = false;
  std::vector<std::vector<int>> cur_, best_sets_;
};

class Balancer {
 public:
  Balancer(const int64_t* w, int n, int P, int kappa, int64_t budget)
      : w_(w), n_(n), P_(P), kappa_(kappa), budget_(budget), owner_(n, -1), load_(P, 0), chunks_(P) {
    int64_t total = 0, wmax = 0;
    for (int i = 0; i < n; ++i) {
      total += w[i];
      wmax = std::max(wmax, w[i]);
    }
    lb_page_ = std::max((total + P - 1) / P, wmax);
    std::vector<int64_t> sorted(w, w + n);
    std::sort(sorted.begin(), sorted.end());
    std::vector<int64_t> prefix(n + 1, 0);
    for (int i = 0; i < n; ++i) prefix[i + 1] = prefix[i] + sorted[i];
    lb_ = wmax + prefix[kappa - 1];
    for (int m = 0; m < P; ++m) {
      const int64_t s = prefix[m + static_cast<int64_t>(P - m) * kappa] - prefix[m];
      lb_ = std::max(lb_, (s + (P - m) - 1) / (P - m));
    }
  }

  void lpt() {
    std::vector<int> order(n_);
    for (int i = 0; i < n_; ++i) order[i] = i;
    std::stable_sort(order.begin(), order.end(), [&](int a, int b) { return w_[a] > w_[b]; });
    std::vector<int> count(P_, 0);
    for (int i : order) {
      int best = -1;
      for (int r = 0; r < P_; ++r)
        if (count[r] < kappa_ && (best < 0 || load_[r] < load_[best])) best = r;
      owner_[i] = best;
      load_[best] += w_[i];
      ++count[best];
    }
    for (int i = 0; i < n_; ++i) chunks_[owner_[i]].push_back(i);  // ascending chunk index
  }

  int64_t makespan() const { return *std::max_element(load_.begin(), load_.end()); }
  int64_t lower_bound_page() const { return lb_page_; }
  int64_t lower_bound() const { return lb_; }
  bool budget_exhausted() const { return budget_hit_; }
  const std::vector<int>& owner() const { return owner_; }

  // P2 run to its end; returns the number of moves
  int pair_phase() {
    int moves = 0;
    while (makespan() > lb_) {
      const int m = sweep(2);
      moves += m;
      if (m == 0) break;
    }
    return moves;
  }

  // P3: triple sweeps, each followed by P2 to its end; returns (triple moves, pair moves)
  void triple_phase(int* triple_moves, int* pair_moves) {
    while (makespan() > lb_) {
      const int m = sweep(3);
      *triple_moves += m;
      if (m == 0) break;
      *pair_moves += pair_phase();
    }
  }

 private:
  int sweep(int k) {
    int moves = 0;
    int g[3] = {0, 1, 2};
    // groups of k ranks in lexicographic order
    auto next = [&]() -> bool {
      for (int i = k - 1; i >= 0; --i) {
        if (g[i] < P_ - k + i) {
          ++g[i];
          for (int j = i + 1; j < k; ++j) g[j] = g[j - 1] + 1;
          return true;
        }
      }
      return false;
    };
    if (P_ < k) return 0;
    do {
      const int64_t phi = makespan();
      if (phi == lb_) break;
      bool holds_max = false;
      int64_t bar = 0;
      for (int i = 0; i < k; ++i) {
        holds_max |= load_[g[i]] == phi;
        bar = std::max(bar, load_[g[i]]);
      }
      if (!holds_max) continue;
      if (repartition(g, k, bar)) ++moves;
    } while (next());
    return moves;
  }

  bool repartition(const int* g, int k, int64_t bar) {
    std::vector<int> pool;
    for (int i = 0; i < k; ++i) pool.insert(pool.end(), chunks_[g[i]].begin(), chunks_[g[i]].end());
    std::sort(pool.begin(), pool.end());
    std::vector<int64_t> wp(pool.size());
    for (size_t i = 0; i < pool.size(); ++i) wp[i] = w_[pool[i]];
    DealSearch search(wp, k, kappa_, bar, budget_);
    const bool found = search.run();
    if (search.aborted()) budget_hit_ = true;
    if (!found) return false;
    for (int i = 0; i < k; ++i) {
      const int r = g[i];
      chunks_[r].clear();
      load_[r] = 0;
      for (int p : search.set(i)) {
        const int c = pool[p];
        chunks_[r].push_back(c);
        owner_[c] = r;
        load_[r] += w_[c];
      }
    }
    return true;
  }

  const int64_t* w_;
  int n_, P_, kappa_;
  int64_t budget_;
  int64_t lb_page_ = 0, lb_ = 0;  // LB as printed, LB_kappa
  bool budget_hit_ = false;
  std::vector<int> owner_;
  std::vector<int64_t> load_;
  std::vector<std::vector<int>> chunks_;  // per rank, ascending chunk index
};

}  // namespace

extern "C" fm_status fm_chunk_loads(const uint8_t* tile_class, int32_t B, int32_t nQ, int32_t nK,
                                    int32_t blocks_per_chunk, int64_t cost_partial, int64_t cost_unmasked,
                                    int64_t* w) {
  if (!tile_class || !w || B < 1 || nQ < 1 || nK < 1 || blocks_per_chunk < 1 || cost_partial < 0 ||
      cost_unmasked < 0)
    return FM_ERR_INVALID_ARG;
  // every sum stays far from overflow: at most B * nQ * nK tiles of the larger cost
  const int64_t tiles = static_cast<int64_t>(B) * nQ * nK;
  const int64_t cmax = std::max(cost_partial, cost_unmasked);
  if (cmax > 0 && tiles > (LLONG_MAX / 4) / cmax) return FM_ERR_INVALID_ARG;
  const int n = (nQ + blocks_per_chunk - 1) / blocks_per_chunk;
  for (int c = 0; c < n; ++c) w[c] = 0;
  for (int b = 0; b < B; ++b)
    for (int qb = 0; qb < nQ; ++qb) {
      const uint8_t* row = tile_class + (static_cast<int64_t>(b) * nQ + qb) * nK;
      int64_t np = 0, nu = 0;
      for (int kb = 0; kb < nK; ++kb) {
        np += row[kb] == 1;
        nu += row[kb] == 2;
      }
      w[qb / blocks_per_chunk] += np * cost_partial + nu * cost_unmasked;
    }
  return FM_OK;
}

// Mask-aware pruning of the K / V exchange (FlashMask-3 project page, §3.4:
// a chunk the mask fully hides is never sent): need[r * n_chunks + c] = 1 iff
// some tile between the query blocks of rank r's chunks and the key blocks of
// chunk c is not skipped, in any batch entry.
extern "C" fm_status fm_needed_chunks(const uint8_t* tile_class, int32_t B, int32_t nQ, int32_t nK,
                                      const int32_t* owner, int32_t n_chunks, int32_t P, int32_t blocks_per_chunk,
                                      uint8_t* need) {
  if (!tile_class || !owner || !need || B < 1 || nQ < 1 || nK < 1 || P < 1 || blocks_per_chunk < 1)
    return FM_ERR_INVALID_ARG;
  if ((int64_t)n_chunks * blocks_per_chunk < nQ || (int64_t)n_chunks * blocks_per_chunk < nK) return FM_ERR_INVALID_ARG;
  for (int c = 0; c < n_chunks; ++c)
    if (owner[c] < 0 || owner[c] >= P) return FM_ERR_INVALID_ARG;
  for (int64_t i = 0; i < (int64_t)P * n_chunks; ++i) need[i] = 0;
  for (int b = 0; b < B; ++b)
    for (int qb = 0; qb < nQ; ++qb) {
      uint8_t* row_need = need + (int64_t)owner[qb / blocks_per_chunk] * n_chunks;
      const uint8_t* row = tile_class + ((int64_t)b * nQ + qb) * nK;
      for (int kb = 0; kb < nK; ++kb)
        if (row[kb] != 0) row_need[kb / blocks_per_chunk] = 1;
    }
  return FM_OK;
}

extern "C" fm_status fm_balance_chunks(const int64_t* w, int32_t n_chunks, int32_t P, int32_t kappa,
                                       int32_t phases, int64_t node_budget, int32_t* owner,
                                       fm_balance_report* report) {
  if (!w || !owner || P < 1 || kappa < 1 || phases < 1 || phases > 3) return FM_ERR_INVALID_ARG;
  if (static_cast<int64_t>(P) * kappa != n_chunks) return FM_ERR_INVALID_ARG;
  // loads >= 0 and small enough that no sum of them can overflow
  for (int i = 0; i < n_chunks; ++i)
    if (w[i] < 0 || w[i] > LLONG_MAX / 4 / n_chunks) return FM_ERR_INVALID_ARG;
  // a repartition tracks its pool in one 64-bit mask
  if ((phases >= 2 && P >= 2 && 2 * kappa > 64) || (phases >= 3 && P >= 3 && 3 * kappa > 64))
    return FM_ERR_UNSUPPORTED;
  Balancer bal(w, n_chunks, P, kappa, node_budget > 0 ? node_budget : kDefaultNodeBudget);
  bal.lpt();
  fm_balance_report rep = {};
  rep.lower_bound = bal.lower_bound_page();
  rep.lower_bound_kappa = bal.lower_bound();
  rep.makespan_lpt = bal.makespan();
  if (phases >= 2 && P >= 2) rep.pair_moves += bal.pair_phase();
  rep.makespan_pair = bal.makespan();
  if (phases >= 3 && P >= 3) bal.triple_phase(&rep.triple_moves, &rep.pair_moves);
  rep.makespan = bal.makespan();
  rep.certified = rep.makespan == rep.lower_bound_kappa;
  rep.budget_exhausted = bal.budget_exhausted();
  for (int i = 0; i < n_chunks; ++i) owner[i] = bal.owner()[i];
  if (report) *report = rep;
  return FM_OK;
}
