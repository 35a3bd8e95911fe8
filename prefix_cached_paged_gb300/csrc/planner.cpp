// Host planners of the stacked passes (host C++, no device work):
//   rc_plan_extend_stacking  which consecutive extend requests share a cached prefix long enough
//                            to attend to it together (the shared-prefix query stacking of the
//                            paper digest's related work, Sec. 7), level by level of the radix
//                            tree, which groups are estimated to pay, and which innermost groups
//                            take their members' remainders in the same pass (fold);
//   rc_plan_decode_groups    which decode requests read a context prefix together.
// Both work on the host slot rows the batch was planned with (a shared prefix is a run of equal
// slot indices) and feed rc_extend_args / rc_decode_args. Decisions use a cost model of the
// extend kernel calibrated on GB300 (kernel replays of the few-shot, two-level and fork
// workloads).
#include <algorithm>
#include <cstdint>
#include <map>
#include <utility>
#include <vector>

#include "host_common.h"

namespace rc {
namespace {

// Cost model of one extend CTA (a pair of 128-row query tiles): per 128-key tile about 2.15 us
// in a batch without stacking groups and 3.3 us in one with them (every pass of such a batch
// runs the kernel's stacking build, whose larger code misses the instruction cache more, and a
// folded pass's query tiles are less balanced) -- half that for a lone tile, whose key tiles
// split across the two softmax groups --, 10 us of fixed cost per CTA, 1 us to merge with a
// partial result. Fitted to kernel replays of the few-shot, two-level and fork batches.
constexpr double kTileUs = 2.15, kStackTileUs = 3.3, kCtaUs = 10.0, kMergeUs = 1.0;

int64_t cdiv(int64_t x, int64_t y) { return (x + y - 1) / y; }

// CTA-time of one request's own pass over keys [key0, P) and its S new tokens.
double request_cost(int64_t P, int64_t S, int64_t key0, int64_t ppt, bool merge, double tile) {
  if (S <= 0) return 0.0;
  const int64_t tiles = cdiv(P - key0, 128) + cdiv(S, 128);
  const int64_t pairs = cdiv(S, 2 * ppt);
  const double per = (double)tiles * (S > ppt ? tile : tile / 2);
  return (double)pairs * (per + kCtaUs + (merge ? kMergeUs : 0.0));
}

// Remainder key tiles member r of a folded group needs in a CTA whose rows end at stacked
// position `end` (the kernel's walk): its cached keys past the shared prefix, then its new
// tokens up to its last row before `end`.
int64_t fold_tiles(const std::vector<int64_t>& qo, const int32_t* P, int r, int64_t shared,
                   int64_t end) {
  const int64_t last = std::min(qo[r + 1], end) - 1 - qo[r];
  return last < 0 ? 0 : cdiv(P[r] - shared + last + 1, 128);
}

// A folded pass over members [0, n): CTA-time, or (limits) whether every CTA's remainder tiles
// and members fit the kernel's table (kFoldTiles / kFoldMembers in the kernel).
constexpr int64_t kFoldTiles = 512, kFoldMembers = 256;
double folded_cost(const int32_t* P, const int32_t* S, int n, int64_t shared, int64_t start,
                   int64_t ppt, bool limits, bool* fits) {
  std::vector<int64_t> qo(n + 1, 0);
  for (int i = 0; i < n; ++i) qo[i + 1] = qo[i] + S[i];
  const int64_t U = qo[n], n_pre = cdiv(shared - start, 128);
  double total = 0.0;
  int r0 = 0;
  if (fits) *fits = true;
  for (int64_t iA = 0; iA < U; iA += 2 * ppt) {
    const int64_t endA = std::min(iA + ppt, U), endC = std::min(iA + 2 * ppt, U);
    while (qo[r0 + 1] <= iA) ++r0;
    int64_t n_rem = 0, n_rem_a = 0;
    int r = r0;
    while (r < n && qo[r] < endC) {
      const int64_t nt = fold_tiles(qo, P, r, shared, endC);
      n_rem += nt;
      if (qo[r + 1] < endA) n_rem_a += nt;
      else if (qo[r] < endA) n_rem_a += fold_tiles(qo, P, r, shared, endA);
      ++r;
    }
    if (limits && (n_rem > kFoldTiles || r - r0 > kFoldMembers)) {
      if (fits) *fits = false;
      return 0.0;
    }
    const int64_t nA = n_pre + n_rem_a;
    const double per = endC > endA ? (double)std::max(nA, n_pre + n_rem) * kStackTileUs
                                    : (double)nA * kStackTileUs / 2;
    total += per + kCtaUs + (start > 0 ? kMergeUs : 0.0);
  }
  return total;
}

struct Costs {
  double alone, unfolded, folded;
};
// Members [0, n) over keys from `start`: their own passes alone; a stacked pass over
// [start, shared) plus their own passes over the rest; one folded pass.
Costs stacking_costs(const int32_t* P, const int32_t* S, int n, int64_t shared, int group,
                     int64_t start) {
  const int64_t ppt = std::max(128 / group, 1);
  Costs c{0.0, 0.0, 0.0};
  int64_t U = 0;
  for (int i = 0; i < n; ++i) {
    c.alone += request_cost(P[i], S[i], start, ppt, start > 0, kTileUs);
    U += S[i];
  }
  const int64_t stacked_tiles = cdiv(shared - start, 128);
  const double first =
      (double)cdiv(U, 2 * ppt) *
      ((double)stacked_tiles * (U > ppt ? kStackTileUs : kStackTileUs / 2) + kCtaUs +
       (start > 0 ? kMergeUs : 0.0));
  double second = 0.0;
  for (int i = 0; i < n; ++i)
    second += request_cost(P[i], S[i], shared, ppt, true, kStackTileUs);
  c.unfolded = first + second;
  c.folded = folded_cost(P, S, n, shared, start, ppt, false, nullptr);
  return c;
}

// Stacking members [0, n) over [start, shared) saves at least 10% (stacked + own passes, or
// folded).
bool stacking_pays(const int32_t* P, const int32_t* S, int n, int64_t shared, int group,
                   int64_t start) {
  int64_t U = 0;
  for (int i = 0; i < n; ++i) U += S[i];
  if (U <= 0) return false;
  const Costs c = stacking_costs(P, S, n, shared, group, start);
  return std::min(c.unfolded, c.folded) < 0.9 * c.alone;
}

// Runs of consecutive requests among [p0, p1) whose slot rows agree over at least min_shared
// leading positions: a run grows while the next request agrees with the run's first over
// min_shared or more of the positions both matched; its shared length is the smallest such
// agreement. Runs of one request, or below min_shared, or with no new token, are not groups.
struct Run {
  int b0, b1;
  int64_t shared;
};
std::vector<Run> runs(const int32_t* rows, int64_t stride, const int32_t* P, const int32_t* S,
                      int p0, int p1, int64_t min_shared) {
  std::vector<Run> out;
  int b = p0;
  while (b < p1) {
    int e = b + 1;
    int64_t sh = P[b];
    while (e < p1) {
      const int64_t n = std::min<int64_t>(sh, P[e]);
      const int32_t* x = rows + (int64_t)b * stride;
      const int32_t* y = rows + (int64_t)e * stride;
      int64_t agree = 0;
      while (agree < n && x[agree] == y[agree]) ++agree;
      if (agree < min_shared) break;
      sh = agree;
      ++e;
    }
    int64_t U = 0;
    for (int i = b; i < e; ++i) U += S[i];
    if (e - b >= 2 && sh >= min_shared && U > 0) out.push_back({b, e, sh});
    b = e;
  }
  return out;
}

}  // namespace
}  // namespace rc

extern "C" int rc_plan_extend_stacking(const rc_stack_plan_args* a, rc_stack_plan* out) {
  RC_CHECK_ARG(a != nullptr && out != nullptr, "rc_plan_extend_stacking: NULL argument");
  RC_CHECK_ARG(a->num_reqs >= 0 && a->row_stride >= 0 && a->min_shared >= 1 &&
                   a->group_size >= 1 && a->max_levels >= 1 &&
                   a->max_levels <= RC_MAX_STACK_LEVELS,
               "rc_plan_extend_stacking: bad sizes");
  RC_CHECK_ARG(a->policy == RC_STACK_COST || a->policy == RC_STACK_ALL,
               "rc_plan_extend_stacking: policy %d", a->policy);
  RC_CHECK_ARG(a->fold == RC_FOLD_NONE || a->fold == RC_FOLD_COST || a->fold == RC_FOLD_ALL,
               "rc_plan_extend_stacking: fold %d", a->fold);
  const int B = a->num_reqs;
  RC_CHECK_ARG(B == 0 || (a->rows && a->prefix_len && a->new_len),
               "rc_plan_extend_stacking: NULL array");
  for (int b = 0; b < B; ++b)
    RC_CHECK_ARG(a->prefix_len[b] >= 0 && a->prefix_len[b] <= a->row_stride && a->new_len[b] >= 0,
                 "rc_plan_extend_stacking: request %d: prefix %d / new %d / row stride %lld", b,
                 a->prefix_len[b], a->new_len[b], (long long)a->row_stride);
  RC_CHECK_ARG(out->capacity >= 0 && (out->capacity == 0 ||
                                      (out->group_range && out->group_shared &&
                                       out->group_start && out->group_fold)),
               "rc_plan_extend_stacking: output arrays");
  const int32_t* P = a->prefix_len;
  const int32_t* S = a->new_len;
  // levels: inside each kept group of level l (shared s), runs agreeing over s + min_shared
  // positions form level l + 1 with key start s; a group not kept is not searched further
  struct G {
    int b0, b1;
    int64_t shared, start;
  };
  std::vector<G> groups;
  std::vector<int32_t> level_indptr{0};
  std::vector<G> parents{{0, B, 0, 0}};
  for (int l = 0; l < a->max_levels; ++l) {
    std::vector<G> found;
    for (const G& par : parents) {
      for (const auto& r : rc::runs(a->rows, a->row_stride, P, S, par.b0, par.b1,
                                    par.shared + a->min_shared)) {
        if (a->policy == RC_STACK_ALL ||
            rc::stacking_pays(P + r.b0, S + r.b0, r.b1 - r.b0, r.shared, a->group_size,
                              par.shared))
          found.push_back({r.b0, r.b1, r.shared, par.shared});
      }
    }
    if (found.empty()) break;
    groups.insert(groups.end(), found.begin(), found.end());
    level_indptr.push_back((int32_t)groups.size());
    parents = found;
  }
  const int NG = (int)groups.size();
  RC_CHECK(NG <= out->capacity, RC_ERR_INVALID,
           "rc_plan_extend_stacking: %d groups, capacity %d", NG, out->capacity);
  // fold: an innermost group whose every CTA fits the kernel's table, where the folded pass is
  // estimated at no more than the stacked pass plus the members' own passes (or always)
  std::vector<int> level(NG);
  for (int l = 0; l + 1 < (int)level_indptr.size(); ++l)
    for (int g = level_indptr[l]; g < level_indptr[l + 1]; ++g) level[g] = l;
  std::vector<char> covered(B, 0);
  int max_rows = 0;
  const int64_t ppt = std::max(128 / a->group_size, 1);
  for (int g = 0; g < NG; ++g) {
    const G& gr = groups[g];
    int64_t U = 0;
    for (int b = gr.b0; b < gr.b1; ++b) U += S[b];
    max_rows = std::max<int64_t>(max_rows, U);
    out->group_range[2 * g] = gr.b0;
    out->group_range[2 * g + 1] = gr.b1;
    out->group_shared[g] = (int32_t)gr.shared;
    out->group_start[g] = (int32_t)gr.start;
    int fold = 0;
    if (a->fold != RC_FOLD_NONE) {
      bool inner = false;
      for (int h = 0; h < NG && !inner; ++h)
        inner = level[h] > level[g] && gr.b0 <= groups[h].b0 && groups[h].b1 <= gr.b1;
      bool fits = false;
      if (!inner)
        rc::folded_cost(P + gr.b0, S + gr.b0, gr.b1 - gr.b0, gr.shared, gr.start, ppt, true,
                        &fits);
      if (!inner && fits) {
        if (a->fold == RC_FOLD_ALL) {
          fold = 1;
        } else {
          const rc::Costs c = rc::stacking_costs(P + gr.b0, S + gr.b0, gr.b1 - gr.b0,
                                                 gr.shared, a->group_size, gr.start);
          fold = c.folded <= c.unfolded;
        }
      }
    }
    out->group_fold[g] = fold;
    if (fold)
      for (int b = gr.b0; b < gr.b1; ++b) covered[b] = 1;
  }
  out->num_groups = NG;
  out->num_levels = (int32_t)level_indptr.size() - 1;
  for (int l = 0; l <= RC_MAX_STACK_LEVELS; ++l)
    out->level_indptr[l] = l < (int)level_indptr.size() ? level_indptr[l] : NG;
  out->max_group_rows = max_rows;
  bool all = true;
  for (int b = 0; b < B; ++b) all = all && covered[b];
  out->all_folded = (NG > 0 && all) ? 1 : 0;
  return RC_OK;
}

extern "C" int rc_plan_decode_groups(const int32_t* rows, int64_t row_stride,
                                     const int64_t* lengths, int32_t num_reqs,
                                     int32_t group_size, int64_t min_shared,
                                     int32_t* out_indptr, int32_t* out_members,
                                     int32_t* out_shared, int32_t* out_num_groups) {
  RC_CHECK_ARG(out_indptr && out_members && out_shared && out_num_groups,
               "rc_plan_decode_groups: NULL output");
  RC_CHECK_ARG(num_reqs >= 0 && row_stride >= 0 && (num_reqs == 0 || (rows && lengths)),
               "rc_plan_decode_groups: bad arguments");
  for (int b = 0; b < num_reqs; ++b)
    RC_CHECK_ARG(lengths[b] >= 0 && lengths[b] <= row_stride,
                 "rc_plan_decode_groups: request %d length %lld", b, (long long)lengths[b]);
  out_indptr[0] = 0;
  *out_num_groups = 0;
  const int B = num_reqs;
  if (group_size < 2 || B < 2) return RC_OK;
  auto lcp = [&](int x, int y) -> int64_t {
    const int64_t n = std::min(lengths[x], lengths[y]);
    const int32_t* rx = rows + (int64_t)x * row_stride;
    const int32_t* ry = rows + (int64_t)y * row_stride;
    int64_t i = 0;
    while (i < n && rx[i] == ry[i]) ++i;
    return i;
  };
  // requests long enough, bucketed by their first slot in order of first appearance
  std::vector<std::vector<int>> buckets;
  std::map<int32_t, int> bucket_of;
  for (int b = 0; b < B; ++b) {
    if (lengths[b] < std::max<int64_t>(min_shared, 1)) continue;
    const int32_t key = rows[(int64_t)b * row_stride];
    auto it = bucket_of.find(key);
    if (it == bucket_of.end()) {
      bucket_of.emplace(key, (int)buckets.size());
      buckets.push_back({b});
    } else {
      buckets[it->second].push_back(b);
    }
  }
  // greedy: the first request of a bucket leads; the others with the longest common slot prefix
  // join (ties: the later request first), up to group_size members, while that prefix is at
  // least min_shared; the group's shared length is its members' smallest common prefix
  int nm = 0, ng = 0;
  for (auto& rest : buckets) {
    while (rest.size() >= 2) {
      const int lead = rest[0];
      std::vector<std::pair<int64_t, int>> cand;
      for (size_t i = 1; i < rest.size(); ++i) cand.push_back({lcp(lead, rest[i]), rest[i]});
      std::sort(cand.begin(), cand.end(), [](const auto& x, const auto& y) { return x > y; });
      std::vector<std::pair<int64_t, int>> take;
      for (size_t i = 0; i < cand.size() && (int)i < group_size - 1; ++i)
        if (cand[i].first >= min_shared) take.push_back(cand[i]);
      if (take.empty()) {
        rest.erase(rest.begin());
        continue;
      }
      out_members[nm++] = lead;
      int64_t sh = take[0].first;
      std::vector<char> used(B, 0);
      used[lead] = 1;
      for (const auto& t : take) {
        out_members[nm++] = t.second;
        sh = std::min(sh, t.first);
        used[t.second] = 1;
      }
      out_shared[ng] = (int32_t)sh;
      out_indptr[++ng] = nm;
      std::vector<int> keep;
      for (int m : rest)
        if (!used[m]) keep.push_back(m);
      rest.swap(keep);
    }
  }
  *out_num_groups = ng;
  return RC_OK;
}
