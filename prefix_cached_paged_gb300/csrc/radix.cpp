// Radix tree over token sequences with per-node reference counts and LRU leaf eviction
// (paper digest Sec. 3 and Fig. 3; SGLang blog Sec. 2.3: traverse, reuse, compute, insert, and
// leaf-first LRU eviction; RadixAttention explainer: insert, match, split, evict).
//
// Host-side structure, built for a scheduler thread that runs it every step:
//   * nodes live in an arena (vector) and are recycled through a free list; a handle packs the
//     arena index with a generation so stale handles are detected;
//   * child lookup is one hash map keyed by (parent index, first token of the edge);
//   * evictable leaves (not the root, reference count 0, no children) sit in an ordered set keyed
//     by (stamp, node id), so eviction pops the least recently used leaf in O(log n) and a parent
//     that becomes such a leaf is inserted as soon as its last child goes.
//
// Semantics (kept identical to the readings stated in the header rc.h):
//   * a match that ends inside an edge splits it; the new upper node takes the next node id,
//     copies the reference count and the stamp; the lower node keeps its id and handle;
//   * match and insert stamp the nodes of their path from the root down with a logical clock;
//   * eviction frees whole nodes, smallest (stamp, id) first, slots in token order.
#include <algorithm>
#include <new>
#include <set>
#include <tuple>
#include <unordered_map>
#include <vector>

#include "host_common.h"
#include "pool_impl.h"

using rc::fail;

namespace {

struct Node {
  int32_t parent = -1;
  uint32_t gen = 0;
  bool live = false;
  bool in_lru = false;
  int32_t nchildren = 0;
  int64_t id = 0;
  int64_t stamp = 0;
  int64_t ref = 0;
  std::vector<int32_t> key;
  std::vector<int32_t> slots;
};

inline uint64_t child_key(int32_t parent, int32_t tok) {
  return ((uint64_t)(uint32_t)parent << 32) | (uint32_t)tok;
}

}  // namespace

struct rc_radix {
  rc_pool* pool = nullptr;
  std::vector<Node> nodes;
  std::vector<int32_t> free_idx;
  std::unordered_map<uint64_t, int32_t> child;
  std::set<std::tuple<int64_t, int64_t, int32_t>> lru;  // (stamp, id, index)
  std::vector<int32_t> path_buf;
  int64_t clock = 0;
  int64_t next_id = 1;
  int64_t cached_tokens = 0;
  int64_t evictable_tokens = 0;  // tokens in nodes with reference count 0 (root excluded)
  int64_t splits = 0, evicted_nodes = 0, evicted_tokens = 0;
  int64_t matched_tokens = 0, match_queries = 0;

  rc_node handle(int32_t idx) const {
    return ((uint64_t)nodes[(size_t)idx].gen << 32) | (uint32_t)idx;
  }
  // index of a live node, or -1
  int32_t resolve(rc_node h) const {
    const uint32_t idx = (uint32_t)(h & 0xFFFFFFFFu);
    const uint32_t gen = (uint32_t)(h >> 32);
    if (idx >= nodes.size()) return -1;
    const Node& n = nodes[idx];
    if (!n.live || n.gen != gen) return -1;
    return (int32_t)idx;
  }
  bool evictable(int32_t i) const {
    const Node& n = nodes[(size_t)i];
    return i != 0 && n.live && n.ref == 0 && n.nchildren == 0;
  }
  void lru_out(int32_t i) {
    Node& n = nodes[(size_t)i];
    if (n.in_lru) {
      lru.erase(std::make_tuple(n.stamp, n.id, i));
      n.in_lru = false;
    }
  }
  void lru_refresh(int32_t i) {
    Node& n = nodes[(size_t)i];
    const bool want = evictable(i);
    if (want && !n.in_lru) {
      lru.emplace(n.stamp, n.id, i);
      n.in_lru = true;
    } else if (!want && n.in_lru) {
      lru_out(i);
    }
  }
  int32_t new_node() {
    int32_t i;
    if (!free_idx.empty()) {
      i = free_idx.back();
      free_idx.pop_back();
    } else {
      i = (int32_t)nodes.size();
      nodes.emplace_back();
    }
    Node& n = nodes[(size_t)i];
    n.gen += 1;
    n.live = true;
    n.in_lru = false;
    n.nchildren = 0;
    n.ref = 0;
    n.stamp = 0;
    n.parent = -1;
    n.id = next_id++;
    n.key.clear();
    n.slots.clear();
    return i;
  }
  int32_t find_child(int32_t parent, int32_t tok) const {
    auto it = child.find(child_key(parent, tok));
    return it == child.end() ? -1 : it->second;
  }
  // Split node c after its first k tokens; returns the new upper node.
  int32_t split(int32_t c, size_t k) {
    const int32_t u = new_node();  // may reallocate `nodes`: take references afterwards
    Node& up = nodes[(size_t)u];
    Node& lo = nodes[(size_t)c];
    up.parent = lo.parent;
    up.key.assign(lo.key.begin(), lo.key.begin() + (std::ptrdiff_t)k);
    up.slots.assign(lo.slots.begin(), lo.slots.begin() + (std::ptrdiff_t)k);
    up.ref = lo.ref;
    up.stamp = lo.stamp;
    up.nchildren = 1;
    lo.key.erase(lo.key.begin(), lo.key.begin() + (std::ptrdiff_t)k);
    lo.slots.erase(lo.slots.begin(), lo.slots.begin() + (std::ptrdiff_t)k);
    lo.parent = u;
    child[child_key(up.parent, up.key[0])] = u;
    child[child_key(u, lo.key[0])] = c;
    splits++;
    return u;
  }
  void touch_path(int32_t end) {
    path_buf.clear();
    for (int32_t x = end; x != 0; x = nodes[(size_t)x].parent) path_buf.push_back(x);
    for (auto it = path_buf.rbegin(); it != path_buf.rend(); ++it) {
      const int32_t x = *it;
      const bool was = nodes[(size_t)x].in_lru;
      if (was) lru_out(x);
      nodes[(size_t)x].stamp = ++clock;
      if (was) lru_refresh(x);
    }
  }
  // common prefix of node edge and tokens[pos:n]
  size_t common(int32_t c, const int32_t* tok, int64_t pos, int64_t n) const {
    const Node& nd = nodes[(size_t)c];
    const size_t lim = std::min<size_t>(nd.key.size(), (size_t)(n - pos));
    size_t k = 0;
    while (k < lim && nd.key[k] == tok[pos + (int64_t)k]) ++k;
    return k;
  }
  int64_t match(const int32_t* tok, int64_t n, int32_t* out_slots, int32_t* out_end) {
    int32_t cur = 0;
    int64_t pos = 0;
    while (pos < n) {
      int32_t c = find_child(cur, tok[pos]);
      if (c < 0) break;
      const size_t k = common(c, tok, pos, n);
      const bool inside = k < nodes[(size_t)c].key.size();
      if (inside) c = split(c, k);
      std::copy(nodes[(size_t)c].slots.begin(), nodes[(size_t)c].slots.begin() + (std::ptrdiff_t)k,
                out_slots + pos);
      pos += (int64_t)k;
      cur = c;
      if (inside) break;
    }
    touch_path(cur);
    matched_tokens += pos;
    match_queries += n;
    *out_end = cur;
    return pos;
  }
  // Longest cached prefix of tokens[0:n] without changing the tree (no split, no stamp).
  // When `visit` is given it is called with (node index, matched tokens of its edge) for every
  // node on the matched path, root excluded, from the root down.
  template <class Visit>
  int64_t peek(const int32_t* tok, int64_t n, Visit&& visit) const {
    int32_t cur = 0;
    int64_t pos = 0;
    while (pos < n) {
      const int32_t c = find_child(cur, tok[pos]);
      if (c < 0) break;
      const size_t k = common(c, tok, pos, n);
      visit(c, (int64_t)k);
      pos += (int64_t)k;
      if (k < nodes[(size_t)c].key.size()) break;
      cur = c;
    }
    return pos;
  }
  int64_t insert(const int32_t* tok, const int32_t* slots, int64_t n, int32_t* out_end) {
    int32_t cur = 0;
    int64_t pos = 0;
    while (pos < n) {
      int32_t c = find_child(cur, tok[pos]);
      if (c < 0) {
        const int32_t leaf = new_node();
        Node& lf = nodes[(size_t)leaf];
        lf.parent = cur;
        lf.key.assign(tok + pos, tok + n);
        lf.slots.assign(slots + pos, slots + n);
        child[child_key(cur, tok[pos])] = leaf;
        nodes[(size_t)cur].nchildren += 1;
        if (cur != 0) lru_refresh(cur);
        cached_tokens += n - pos;
        evictable_tokens += n - pos;
        cur = leaf;
        break;
      }
      const size_t k = common(c, tok, pos, n);
      if (k < nodes[(size_t)c].key.size()) c = split(c, k);
      pos += (int64_t)k;
      cur = c;
    }
    touch_path(cur);
    if (cur != 0) lru_refresh(cur);
    *out_end = cur;
    return pos;
  }
  int lock(int32_t i) {
    for (int32_t x = i; x != 0; x = nodes[(size_t)x].parent) {
      Node& n = nodes[(size_t)x];
      if (++n.ref == 1) {
        lru_out(x);
        evictable_tokens -= (int64_t)n.key.size();
      }
    }
    return RC_OK;
  }
  int unlock(int32_t i) {
    for (int32_t x = i; x != 0; x = nodes[(size_t)x].parent)
      if (nodes[(size_t)x].ref <= 0)
        return fail(RC_ERR_INVALID, "radix_unlock: reference count of node %lld is already 0",
                    (long long)nodes[(size_t)x].id);
    for (int32_t x = i; x != 0; x = nodes[(size_t)x].parent) {
      Node& n = nodes[(size_t)x];
      if (--n.ref == 0) {
        evictable_tokens += (int64_t)n.key.size();
        lru_refresh(x);
      }
    }
    return RC_OK;
  }
  int evict(int64_t want, int64_t* freed_out) {
    int64_t freed = 0;
    while (freed < want && !lru.empty()) {
      const int32_t i = std::get<2>(*lru.begin());
      Node& n = nodes[(size_t)i];
      const int rc = rc::pool_give(pool, n.slots.data(), (int64_t)n.slots.size());
      if (rc != RC_OK) {
        *freed_out = freed;
        return fail(RC_ERR_INVALID, "radix_evict_lru: node %lld holds slots the pool rejects",
                    (long long)n.id);
      }
      lru_out(i);
      freed += (int64_t)n.slots.size();
      cached_tokens -= (int64_t)n.slots.size();
      evictable_tokens -= (int64_t)n.slots.size();
      evicted_tokens += (int64_t)n.slots.size();
      evicted_nodes++;
      const int32_t par = n.parent;
      child.erase(child_key(par, n.key[0]));
      n.live = false;
      n.key.clear();
      n.key.shrink_to_fit();
      n.slots.clear();
      n.slots.shrink_to_fit();
      free_idx.push_back(i);
      nodes[(size_t)par].nchildren -= 1;
      if (par != 0) lru_refresh(par);
    }
    *freed_out = freed;
    if (freed < want)
      return fail(RC_ERR_INSUFFICIENT, "radix_evict_lru: freed %lld of %lld tokens",
                  (long long)freed, (long long)want);
    return RC_OK;
  }
};

extern "C" {

int rc_radix_create(rc_pool* pool, rc_radix** out) {
  RC_CHECK_ARG(pool != nullptr && out != nullptr, "rc_radix_create: NULL argument");
  rc_radix* t = new (std::nothrow) rc_radix();
  if (!t) return fail(RC_ERR_OOM, "rc_radix_create: host allocation failed");
  t->pool = pool;
  t->nodes.emplace_back();  // root: index 0, generation 0, id 0
  t->nodes[0].live = true;
  *out = t;
  return RC_OK;
}

void rc_radix_destroy(rc_radix* tree) { delete tree; }

int rc_radix_match_prefix(rc_radix* t, const int32_t* tokens, int64_t n, int32_t* out_slots,
                          int64_t* out_len, rc_node* out_node) {
  RC_CHECK_ARG(t && out_len && out_node && n >= 0, "rc_radix_match_prefix: bad argument");
  RC_CHECK_ARG(n == 0 || (tokens && out_slots), "rc_radix_match_prefix: NULL tokens/out_slots");
  int32_t end;
  *out_len = t->match(tokens, n, out_slots, &end);
  *out_node = t->handle(end);
  return RC_OK;
}

int rc_radix_insert(rc_radix* t, const int32_t* tokens, const int32_t* slots, int64_t n,
                    int64_t* out_existing, rc_node* out_node) {
  RC_CHECK_ARG(t && out_existing && out_node && n >= 0, "rc_radix_insert: bad argument");
  RC_CHECK_ARG(n == 0 || (tokens && slots), "rc_radix_insert: NULL tokens/slots");
  int32_t end;
  *out_existing = t->insert(tokens, slots, n, &end);
  *out_node = t->handle(end);
  return RC_OK;
}

int rc_radix_lock(rc_radix* t, rc_node node) {
  RC_CHECK_ARG(t != nullptr, "rc_radix_lock: tree is NULL");
  const int32_t i = t->resolve(node);
  RC_CHECK_ARG(i >= 0, "rc_radix_lock: stale or invalid node handle");
  return t->lock(i);
}

int rc_radix_unlock(rc_radix* t, rc_node node) {
  RC_CHECK_ARG(t != nullptr, "rc_radix_unlock: tree is NULL");
  const int32_t i = t->resolve(node);
  RC_CHECK_ARG(i >= 0, "rc_radix_unlock: stale or invalid node handle");
  return t->unlock(i);
}

int rc_radix_evict_lru(rc_radix* t, int64_t n_tokens, int64_t* out_freed) {
  RC_CHECK_ARG(t && out_freed && n_tokens >= 0, "rc_radix_evict_lru: bad argument");
  return t->evict(n_tokens, out_freed);
}

int rc_radix_stats(const rc_radix* t, rc_stats* s) {
  RC_CHECK_ARG(t && s, "rc_radix_stats: NULL argument");
  *s = rc_stats{};
  for (size_t i = 1; i < t->nodes.size(); ++i) {
    const Node& n = t->nodes[i];
    if (!n.live) continue;
    s->nodes++;
    if (n.ref > 0)
      s->protected_tokens += (int64_t)n.key.size();
    else
      s->evictable_tokens += (int64_t)n.key.size();
  }
  s->cached_tokens = t->cached_tokens;
  s->splits = t->splits;
  s->evicted_nodes = t->evicted_nodes;
  s->evicted_tokens = t->evicted_tokens;
  s->matched_tokens = t->matched_tokens;
  s->match_queries = t->match_queries;
  return RC_OK;
}

int64_t rc_radix_dump(const rc_radix* t, int64_t* buf, int64_t cap) {
  if (!t) return 0;
  // children of every live node, ordered by first token
  std::vector<std::vector<std::pair<int32_t, int32_t>>> kids(t->nodes.size());
  int64_t need = 0;
  for (size_t i = 1; i < t->nodes.size(); ++i) {
    const Node& n = t->nodes[i];
    if (!n.live) continue;
    kids[(size_t)n.parent].emplace_back(n.key[0], (int32_t)i);
    need += 5 + 2 * (int64_t)n.key.size();
  }
  if (need > cap || !buf) return -need;
  for (auto& k : kids) std::sort(k.begin(), k.end());
  int64_t w = 0;
  std::vector<int32_t> stack;
  for (auto it = kids[0].rbegin(); it != kids[0].rend(); ++it) stack.push_back(it->second);
  while (!stack.empty()) {
    const int32_t i = stack.back();
    stack.pop_back();
    const Node& n = t->nodes[(size_t)i];
    buf[w++] = n.id;
    buf[w++] = t->nodes[(size_t)n.parent].id;
    buf[w++] = n.ref;
    buf[w++] = n.stamp;
    buf[w++] = (int64_t)n.key.size();
    for (int32_t v : n.key) buf[w++] = v;
    for (int32_t v : n.slots) buf[w++] = v;
    for (auto it = kids[(size_t)i].rbegin(); it != kids[(size_t)i].rend(); ++it)
      stack.push_back(it->second);
  }
  return w;
}

int rc_radix_match_batch(rc_radix* t, const int32_t* tokens, const int64_t* indptr, int32_t B,
                         const int32_t* match_len, int32_t* rows, int64_t row_stride,
                         int32_t* prefix_len, rc_node* nodes) {
  RC_CHECK_ARG(t && B >= 0 && (B == 0 || (tokens && indptr && rows && prefix_len && nodes)),
               "rc_radix_match_batch: bad argument");
  for (int32_t b = 0; b < B; ++b) {
    const int64_t len = indptr[b + 1] - indptr[b];
    const int64_t n = match_len ? (int64_t)match_len[b] : len;
    RC_CHECK_ARG(len >= 0 && n >= 0 && n <= len && len <= row_stride,
                 "rc_radix_match_batch: request %d: length %lld, match %lld, row %lld", b,
                 (long long)len, (long long)n, (long long)row_stride);
  }
  for (int32_t b = 0; b < B; ++b) {
    const int64_t len = indptr[b + 1] - indptr[b];
    const int64_t n = match_len ? (int64_t)match_len[b] : len;
    int32_t end;
    const int64_t p = t->match(tokens + indptr[b], n, rows + (int64_t)b * row_stride, &end);
    t->lock(end);
    prefix_len[b] = (int32_t)p;
    nodes[b] = t->handle(end);
  }
  return RC_OK;
}

int rc_radix_insert_batch(rc_radix* t, const int32_t* tokens, const int64_t* indptr, int32_t B,
                          const int32_t* rows, int64_t row_stride, const int32_t* prefix_len,
                          const rc_node* unlock_nodes, int32_t keep_locked, rc_node* end_nodes,
                          int64_t* out_freed) {
  RC_CHECK_ARG(t && B >= 0 && (B == 0 || (tokens && indptr && rows && prefix_len)),
               "rc_radix_insert_batch: bad argument");
  for (int32_t b = 0; b < B; ++b) {
    const int64_t len = indptr[b + 1] - indptr[b];
    RC_CHECK_ARG(len >= 0 && len <= row_stride && prefix_len[b] >= 0 && prefix_len[b] <= len,
                 "rc_radix_insert_batch: request %d: bad length", b);
    if (unlock_nodes)
      RC_CHECK_ARG(t->resolve(unlock_nodes[b]) >= 0, "rc_radix_insert_batch: request %d: stale node",
                   b);
  }
  int64_t freed = 0;
  for (int32_t b = 0; b < B; ++b) {
    const int64_t len = indptr[b + 1] - indptr[b];
    const int32_t* row = rows + (int64_t)b * row_stride;
    int32_t end;
    const int64_t ex = t->insert(tokens + indptr[b], row, len, &end);
    if (ex > prefix_len[b]) {
      const int rc = rc::pool_give(t->pool, row + prefix_len[b], ex - prefix_len[b]);
      if (rc != RC_OK) return rc;
      freed += ex - prefix_len[b];
    }
    if (keep_locked) t->lock(end);
    if (end_nodes) end_nodes[b] = t->handle(end);
    if (unlock_nodes) {
      const int32_t u = t->resolve(unlock_nodes[b]);
      if (u < 0) return fail(RC_ERR_INVALID, "rc_radix_insert_batch: request %d: stale node", b);
      const int rc = t->unlock(u);
      if (rc != RC_OK) return rc;
    }
  }
  if (out_freed) *out_freed = freed;
  return RC_OK;
}

int rc_schedule_batch(const rc_radix* t, const int32_t* tokens, const int64_t* indptr, int32_t B,
                      const int32_t* match_len, int32_t policy, int32_t max_batch,
                      int64_t max_new_tokens, int64_t reserve_slots, int32_t* out_order,
                      int32_t* out_match, int32_t* out_admitted) {
  RC_CHECK_ARG(t && out_admitted && B >= 0 && max_batch >= 0 && reserve_slots >= 0 &&
                   (policy == RC_SCHED_LSPF || policy == RC_SCHED_FCFS) &&
                   (B == 0 || (tokens && indptr && out_order && out_match)),
               "rc_schedule_batch: bad argument");
  for (int32_t w = 0; w < B; ++w) {
    const int64_t len = indptr[w + 1] - indptr[w];
    const int64_t n = match_len ? (int64_t)match_len[w] : len;
    RC_CHECK_ARG(indptr[w] >= 0 && len >= 0 && n >= 0 && n <= len,
                 "rc_schedule_batch: sequence %d: length %lld, match %lld", w, (long long)len,
                 (long long)n);
  }
  auto seq = [&](int32_t w) { return tokens + indptr[w]; };
  auto lim = [&](int32_t w) {
    return match_len ? (int64_t)match_len[w] : indptr[w + 1] - indptr[w];
  };
  for (int32_t w = 0; w < B; ++w)
    out_match[w] = (int32_t)t->peek(seq(w), lim(w), [](int32_t, int64_t) {});
  for (int32_t w = 0; w < B; ++w) out_order[w] = w;
  if (policy == RC_SCHED_LSPF)
    std::stable_sort(out_order, out_order + B,
                     [&](int32_t a, int32_t b) { return out_match[a] > out_match[b]; });
  // Room: free slots plus every cached token in an unreferenced node (all of them can be
  // evicted, leaves first), minus the reserve. An admitted sequence takes its computed tokens
  // and locks its match, which takes the unreferenced cached tokens on that path out of the
  // evictable room (each counted once across the batch).
  int64_t free_slots = 0;
  rc_kv_pool_available(t->pool, &free_slots);
  const int64_t room = free_slots + t->evictable_tokens - reserve_slots;
  std::unordered_map<int32_t, int64_t> held;  // node index -> protected prefix of its edge
  std::vector<std::pair<int32_t, int64_t>> ups;
  int64_t used = 0, computed = 0;
  int32_t admitted = 0;
  for (int32_t i = 0; i < B && admitted < max_batch; ++i) {
    const int32_t w = out_order[i];
    const int64_t fresh = indptr[w + 1] - indptr[w] - out_match[w];
    if (max_new_tokens >= 0 && computed + fresh > max_new_tokens) break;
    int64_t locked = 0;
    ups.clear();
    t->peek(seq(w), lim(w), [&](int32_t c, int64_t k) {
      if (t->nodes[(size_t)c].ref != 0) return;
      auto it = held.find(c);
      const int64_t have = it == held.end() ? 0 : it->second;
      if (k > have) {
        locked += k - have;
        ups.emplace_back(c, k);
      }
    });
    if (used + fresh + locked > room) break;
    used += fresh + locked;
    computed += fresh;
    for (const auto& u : ups) held[u.first] = u.second;
    ++admitted;
  }
  *out_admitted = admitted;
  return RC_OK;
}

}  // extern "C"
