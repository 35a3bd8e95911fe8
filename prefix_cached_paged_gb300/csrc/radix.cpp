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
  bool in_lru = false;    // in the device eviction set
  bool in_hlru = false;   // in the host eviction set
  bool host = false;      // KV held in host-tier slots (a tree with a host tier only)
  int32_t nchildren = 0;
  int32_t ndev = 0;       // device-resident children
  int64_t pending = -1;   // first pending spill copy of this node (-1: none)
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
  rc_pool* host_pool = nullptr;  // host tier (NULL: evicted leaves are freed)
  std::vector<Node> nodes;
  std::vector<int32_t> free_idx;
  std::unordered_map<uint64_t, int32_t> child;
  std::set<std::tuple<int64_t, int64_t, int32_t>> lru;   // device leaves: (stamp, id, index)
  std::set<std::tuple<int64_t, int64_t, int32_t>> hlru;  // host leaves
  // copies the caller owes the pool contents: spills (device slot -> host slot, dst -1 =
  // cancelled) before loads (host slot -> device slot), drained by rc_radix_drain_copies
  std::vector<int32_t> spill_src, spill_dst, load_src, load_dst;
  std::vector<int32_t> spill_node;  // node index of each spill copy
  std::vector<int32_t> path_buf;
  int64_t clock = 0;
  int64_t next_id = 1;
  int64_t cached_tokens = 0;
  int64_t evictable_tokens = 0;  // tokens in nodes with reference count 0 (root excluded)
  int64_t splits = 0, evicted_nodes = 0, evicted_tokens = 0;
  int64_t matched_tokens = 0, match_queries = 0;
  int64_t host_tokens = 0, spilled_tokens = 0, loaded_tokens = 0, dropped_tokens = 0;

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
  // device leaf: device-resident, unreferenced, no device-resident child
  bool evictable(int32_t i) const {
    const Node& n = nodes[(size_t)i];
    return i != 0 && n.live && !n.host && n.ref == 0 && n.ndev == 0;
  }
  // host leaf: host-resident, unreferenced, no child at all
  bool host_evictable(int32_t i) const {
    const Node& n = nodes[(size_t)i];
    return i != 0 && n.live && n.host && n.ref == 0 && n.nchildren == 0;
  }
  void lru_out(int32_t i) {
    Node& n = nodes[(size_t)i];
    if (n.in_lru) {
      lru.erase(std::make_tuple(n.stamp, n.id, i));
      n.in_lru = false;
    }
    if (n.in_hlru) {
      hlru.erase(std::make_tuple(n.stamp, n.id, i));
      n.in_hlru = false;
    }
  }
  void lru_refresh(int32_t i) {
    Node& n = nodes[(size_t)i];
    const bool want = evictable(i), hwant = host_evictable(i);
    if (want != n.in_lru) {
      if (want)
        lru.emplace(n.stamp, n.id, i);
      else
        lru.erase(std::make_tuple(n.stamp, n.id, i));
      n.in_lru = want;
    }
    if (hwant != n.in_hlru) {
      if (hwant)
        hlru.emplace(n.stamp, n.id, i);
      else
        hlru.erase(std::make_tuple(n.stamp, n.id, i));
      n.in_hlru = hwant;
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
    n.in_hlru = false;
    n.host = false;
    n.nchildren = 0;
    n.ndev = 0;
    n.pending = -1;
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
    up.host = lo.host;
    up.nchildren = 1;
    up.ndev = lo.host ? 0 : 1;
    lo.key.erase(lo.key.begin(), lo.key.begin() + (std::ptrdiff_t)k);
    lo.slots.erase(lo.slots.begin(), lo.slots.begin() + (std::ptrdiff_t)k);
    lo.parent = u;
    if (lo.pending >= 0) {  // its pending spill copies are in token order: the first k go up
      up.pending = lo.pending;
      for (size_t j = 0; j < k; ++j) spill_node[(size_t)up.pending + j] = u;
      lo.pending += (int64_t)k;
    }
    child[child_key(up.parent, up.key[0])] = u;
    child[child_key(u, lo.key[0])] = c;
    splits++;
    return u;
  }
  // ---------------------------------------------------------------- host tier
  void cancel_pending(int32_t i) {
    Node& n = nodes[(size_t)i];
    if (n.pending < 0) return;
    for (size_t j = 0; j < n.key.size(); ++j) spill_dst[(size_t)n.pending + j] = -1;
    n.pending = -1;
  }
  // Unlink a childless node (either tier) and recycle its arena entry; slots are the caller's.
  void unlink(int32_t i) {
    Node& n = nodes[(size_t)i];
    lru_out(i);
    const int32_t par = n.parent;
    child.erase(child_key(par, n.key[0]));
    Node& p = nodes[(size_t)par];
    p.nchildren -= 1;
    if (!n.host) p.ndev -= 1;
    n.live = false;
    n.key.clear();
    n.key.shrink_to_fit();
    n.slots.clear();
    n.slots.shrink_to_fit();
    free_idx.push_back(i);
    if (par != 0) lru_refresh(par);
  }
  // Drop the least recently used host leaf.
  void drop_host_leaf() {
    const int32_t i = std::get<2>(*hlru.begin());
    Node& n = nodes[(size_t)i];
    const int64_t len = (int64_t)n.slots.size();
    cancel_pending(i);
    rc::pool_give(host_pool, n.slots.data(), len);
    host_tokens -= len;
    dropped_tokens += len;
    unlink(i);
  }
  // Host-resident node i becomes device-resident with device slots dev[0:len]; its host slots
  // are released now (release_now) or after the pending copies are drained (a load reads them).
  void to_device(int32_t i, const int32_t* dev, bool release_now) {
    Node& n = nodes[(size_t)i];
    const size_t len = n.key.size();
    if (release_now) {
      cancel_pending(i);
      rc::pool_give(host_pool, n.slots.data(), (int64_t)len);
    }
    n.slots.assign(dev, dev + len);
    n.host = false;
    host_tokens -= (int64_t)len;
    cached_tokens += (int64_t)len;
    if (n.ref == 0) evictable_tokens += (int64_t)len;
    nodes[(size_t)n.parent].ndev += 1;
    lru_refresh(i);
    if (n.parent != 0) lru_refresh(n.parent);
  }
  void touch_path(int32_t end) {
    path_buf.clear();
    for (int32_t x = end; x != 0; x = nodes[(size_t)x].parent) path_buf.push_back(x);
    for (auto it = path_buf.rbegin(); it != path_buf.rend(); ++it) {
      const int32_t x = *it;
      const bool was = nodes[(size_t)x].in_lru || nodes[(size_t)x].in_hlru;
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
  // Longest device-resident cached prefix (with host_len: continue through host-resident nodes,
  // whose tokens are counted in *host_len and whose slots are not written).
  int64_t match(const int32_t* tok, int64_t n, int32_t* out_slots, int32_t* out_end,
                int64_t* host_len = nullptr) {
    int32_t cur = 0;
    int64_t pos = 0, hpos = 0;
    while (pos + hpos < n) {
      int32_t c = find_child(cur, tok[pos + hpos]);
      if (c < 0) break;
      if (nodes[(size_t)c].host) {
        if (!host_len) break;
        const size_t k = common(c, tok, pos + hpos, n);
        const bool inside = k < nodes[(size_t)c].key.size();
        if (inside) c = split(c, k);
        hpos += (int64_t)k;
        cur = c;
        if (inside) break;
        continue;
      }
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
    if (host_len) *host_len = hpos;
    matched_tokens += pos + hpos;
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
      if (c < 0 || nodes[(size_t)c].host) break;
      const size_t k = common(c, tok, pos, n);
      visit(c, (int64_t)k);
      pos += (int64_t)k;
      if (k < nodes[(size_t)c].key.size()) break;
      cur = c;
    }
    return pos;
  }
  // Insert tokens[0:n] with slots[0:n]. Device-resident tokens already present keep their
  // slots; tokens held by host-resident nodes take the caller's slots (the node returns to the
  // device, its host slots are freed). Returns the length of the leading device-resident part
  // that was already present.
  int64_t insert(const int32_t* tok, const int32_t* slots, int64_t n, int32_t* out_end) {
    int32_t cur = 0;
    int64_t pos = 0, existing = -1;
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
        nodes[(size_t)cur].ndev += 1;
        if (cur != 0) lru_refresh(cur);
        cached_tokens += n - pos;
        evictable_tokens += n - pos;
        if (existing < 0) existing = pos;
        cur = leaf;
        pos = n;
        break;
      }
      const size_t k = common(c, tok, pos, n);
      if (k < nodes[(size_t)c].key.size()) c = split(c, k);
      if (nodes[(size_t)c].host) {
        if (existing < 0) existing = pos;
        to_device(c, slots + pos, true);
      }
      pos += (int64_t)k;
      cur = c;
    }
    touch_path(cur);
    if (cur != 0) lru_refresh(cur);
    *out_end = cur;
    return existing < 0 ? pos : existing;
  }
  int lock(int32_t i) {
    for (int32_t x = i; x != 0; x = nodes[(size_t)x].parent) {
      Node& n = nodes[(size_t)x];
      if (++n.ref == 1) {
        lru_out(x);
        if (!n.host) evictable_tokens -= (int64_t)n.key.size();
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
        if (!n.host) evictable_tokens += (int64_t)n.key.size();
        lru_refresh(x);
      }
    }
    return RC_OK;
  }
  int evict(int64_t want, int64_t* freed_out) {
    int64_t freed = 0;
    if (host_pool && !load_src.empty()) {
      *freed_out = 0;
      return fail(RC_ERR_INVALID,
                  "radix_evict_lru: host-tier loads are pending; drain the copies first");
    }
    while (freed < want && !lru.empty()) {
      const int32_t i = std::get<2>(*lru.begin());
      const int64_t len = (int64_t)nodes[(size_t)i].slots.size();
      const int rc = rc::pool_give(pool, nodes[(size_t)i].slots.data(), len);
      if (rc != RC_OK) {
        *freed_out = freed;
        return fail(RC_ERR_INVALID, "radix_evict_lru: node %lld holds slots the pool rejects",
                    (long long)nodes[(size_t)i].id);
      }
      freed += len;
      cached_tokens -= len;
      evictable_tokens -= len;
      evicted_tokens += len;
      if (host_pool) {
        // make room in the host tier, least recently used host leaves first
        while (rc::pool_free_count(host_pool) < len && !hlru.empty()) drop_host_leaf();
        if (rc::pool_free_count(host_pool) >= len) {
          // spill: the node keeps its place in the tree, its KV moves to host slots
          Node& n = nodes[(size_t)i];
          lru_out(i);
          const size_t at = spill_src.size();
          spill_src.insert(spill_src.end(), n.slots.begin(), n.slots.end());
          spill_dst.resize(at + (size_t)len);
          rc::pool_take(host_pool, len, spill_dst.data() + at);
          spill_node.insert(spill_node.end(), (size_t)len, i);
          n.slots.assign(spill_dst.begin() + (std::ptrdiff_t)at, spill_dst.end());
          n.pending = (int64_t)at;
          n.host = true;
          host_tokens += len;
          spilled_tokens += len;
          evicted_nodes++;
          nodes[(size_t)n.parent].ndev -= 1;
          lru_refresh(i);
          if (n.parent != 0) lru_refresh(n.parent);
          continue;
        }
        dropped_tokens += len;  // the host tier cannot take it: freed (it has no child left)
      }
      evicted_nodes++;
      unlink(i);
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
    if (n.host)
      continue;
    else if (n.ref > 0)
      s->protected_tokens += (int64_t)n.key.size();
    else
      s->evictable_tokens += (int64_t)n.key.size();
  }
  s->host_tokens = t->host_tokens;
  s->spilled_tokens = t->spilled_tokens;
  s->loaded_tokens = t->loaded_tokens;
  s->dropped_tokens = t->dropped_tokens;
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

static int match_batch_impl(rc_radix* t, const int32_t* tokens, const int64_t* indptr, int32_t B,
                            const int32_t* match_len, int32_t* rows, int64_t row_stride,
                            int32_t* prefix_len, rc_node* nodes, int32_t* host_len,
                            const char* name) {
  RC_CHECK_ARG(t && B >= 0 && (B == 0 || (tokens && indptr && rows && prefix_len && nodes)),
               "%s: bad argument", name);
  for (int32_t b = 0; b < B; ++b) {
    const int64_t len = indptr[b + 1] - indptr[b];
    const int64_t n = match_len ? (int64_t)match_len[b] : len;
    RC_CHECK_ARG(len >= 0 && n >= 0 && n <= len && len <= row_stride,
                 "%s: request %d: length %lld, match %lld, row %lld", name, b, (long long)len,
                 (long long)n, (long long)row_stride);
  }
  for (int32_t b = 0; b < B; ++b) {
    const int64_t len = indptr[b + 1] - indptr[b];
    const int64_t n = match_len ? (int64_t)match_len[b] : len;
    int32_t end;
    int64_t h = 0;
    const int64_t p = t->match(tokens + indptr[b], n, rows + (int64_t)b * row_stride, &end,
                               host_len ? &h : nullptr);
    t->lock(end);
    prefix_len[b] = (int32_t)p;
    nodes[b] = t->handle(end);
    if (host_len) host_len[b] = (int32_t)h;
  }
  return RC_OK;
}

int rc_radix_match_batch(rc_radix* t, const int32_t* tokens, const int64_t* indptr, int32_t B,
                         const int32_t* match_len, int32_t* rows, int64_t row_stride,
                         int32_t* prefix_len, rc_node* nodes) {
  return match_batch_impl(t, tokens, indptr, B, match_len, rows, row_stride, prefix_len, nodes,
                          nullptr, "rc_radix_match_batch");
}

int rc_radix_match_batch_tiered(rc_radix* t, const int32_t* tokens, const int64_t* indptr,
                                int32_t B, const int32_t* match_len, int32_t* rows,
                                int64_t row_stride, int32_t* prefix_len, rc_node* nodes,
                                int32_t* host_len) {
  RC_CHECK_ARG(host_len != nullptr, "rc_radix_match_batch_tiered: host_len is NULL");
  return match_batch_impl(t, tokens, indptr, B, match_len, rows, row_stride, prefix_len, nodes,
                          host_len, "rc_radix_match_batch_tiered");
}

int rc_radix_attach_host_tier(rc_radix* t, rc_pool* host_pool) {
  RC_CHECK_ARG(t && host_pool && host_pool != t->pool, "rc_radix_attach_host_tier: bad argument");
  RC_CHECK_ARG(t->host_pool == nullptr, "rc_radix_attach_host_tier: a host tier is attached");
  t->host_pool = host_pool;
  return RC_OK;
}

int rc_radix_load_batch(rc_radix* t, const int32_t* tokens, const int64_t* indptr, int32_t B,
                        int32_t* rows, int64_t row_stride, int32_t* prefix_len,
                        const int32_t* host_len) {
  RC_CHECK_ARG(t && t->host_pool && B >= 0 &&
                   (B == 0 || (tokens && indptr && rows && prefix_len && host_len)),
               "rc_radix_load_batch: bad argument (or no host tier)");
  int64_t need = 0;
  for (int32_t b = 0; b < B; ++b) {
    const int64_t len = indptr[b + 1] - indptr[b];
    RC_CHECK_ARG(prefix_len[b] >= 0 && host_len[b] >= 0 &&
                     (int64_t)prefix_len[b] + host_len[b] <= len && len <= row_stride,
                 "rc_radix_load_batch: request %d: bad lengths", b);
    need += host_len[b];
  }
  int64_t avail = rc::pool_free_count(t->pool);
  RC_CHECK(avail >= need, RC_ERR_OOM,
           "rc_radix_load_batch: %lld device slots free, up to %lld needed", (long long)avail,
           (long long)need);
  std::vector<int32_t> dev;
  for (int32_t b = 0; b < B; ++b) {
    const int32_t* tok = tokens + indptr[b];
    int32_t* row = rows + (int64_t)b * row_stride;
    const int64_t end = (int64_t)prefix_len[b] + host_len[b];
    int32_t cur = 0;
    int64_t pos = 0;
    while (pos < end) {
      const int32_t c = t->find_child(cur, tok[pos]);
      RC_CHECK(c >= 0, RC_ERR_INVALID, "rc_radix_load_batch: request %d: path gone at %lld", b,
               (long long)pos);
      Node& n = t->nodes[(size_t)c];
      const int64_t len = (int64_t)n.key.size();
      RC_CHECK(pos + len <= end && t->common(c, tok, pos, end) == (size_t)len, RC_ERR_INVALID,
               "rc_radix_load_batch: request %d: the matched path changed", b);
      if (n.host) {
        RC_CHECK(n.ref > 0, RC_ERR_INVALID,
                 "rc_radix_load_batch: request %d: host node not locked by its match", b);
        dev.resize((size_t)len);
        rc::pool_take(t->pool, len, dev.data());
        t->load_src.insert(t->load_src.end(), n.slots.begin(), n.slots.end());
        t->load_dst.insert(t->load_dst.end(), dev.begin(), dev.end());
        t->loaded_tokens += len;
        n.pending = -1;  // pending spill copies stay valid: they run before the loads
        t->to_device(c, dev.data(), false);
      }
      if (pos >= prefix_len[b])
        std::copy(t->nodes[(size_t)c].slots.begin(), t->nodes[(size_t)c].slots.end(), row + pos);
      pos += len;
      cur = c;
    }
    prefix_len[b] = (int32_t)end;
  }
  return RC_OK;
}

int rc_radix_pending_copies(const rc_radix* t, int64_t* n_spill, int64_t* n_load) {
  RC_CHECK_ARG(t && n_spill && n_load, "rc_radix_pending_copies: NULL argument");
  int64_t ns = 0;
  for (int32_t d : t->spill_dst) ns += d >= 0;
  *n_spill = ns;
  *n_load = (int64_t)t->load_src.size();
  return RC_OK;
}

int rc_radix_drain_copies(rc_radix* t, int32_t* spill_dev, int32_t* spill_host, int32_t* load_host,
                          int32_t* load_dev) {
  RC_CHECK_ARG(t, "rc_radix_drain_copies: tree is NULL");
  int64_t ns = 0;
  for (size_t j = 0; j < t->spill_src.size(); ++j) {
    if (t->spill_dst[j] < 0) continue;
    RC_CHECK_ARG(spill_dev && spill_host, "rc_radix_drain_copies: NULL spill buffers");
    spill_dev[ns] = t->spill_src[j];
    spill_host[ns] = t->spill_dst[j];
    ++ns;
  }
  if (!t->load_src.empty()) {
    RC_CHECK_ARG(load_host && load_dev, "rc_radix_drain_copies: NULL load buffers");
    std::copy(t->load_src.begin(), t->load_src.end(), load_host);
    std::copy(t->load_dst.begin(), t->load_dst.end(), load_dev);
    // the loads' host slots were held until their copies were handed out
    const int rc = rc::pool_give(t->host_pool, t->load_src.data(), (int64_t)t->load_src.size());
    if (rc != RC_OK) return rc;
  }
  for (auto& n : t->nodes) n.pending = -1;
  t->spill_src.clear();
  t->spill_dst.clear();
  t->spill_node.clear();
  t->load_src.clear();
  t->load_dst.clear();
  return RC_OK;
}

int64_t rc_radix_tiers(const rc_radix* t, int64_t* buf, int64_t cap) {
  if (!t) return 0;
  std::vector<std::vector<std::pair<int32_t, int32_t>>> kids(t->nodes.size());
  int64_t need = 0;
  for (size_t i = 1; i < t->nodes.size(); ++i) {
    const Node& n = t->nodes[i];
    if (!n.live) continue;
    kids[(size_t)n.parent].emplace_back(n.key[0], (int32_t)i);
    need += 2;
  }
  if (need > cap || !buf) return -need;
  for (auto& k : kids) std::sort(k.begin(), k.end());
  int64_t w = 0;
  std::vector<int32_t> stack;
  for (auto it = kids[0].rbegin(); it != kids[0].rend(); ++it) stack.push_back(it->second);
  while (!stack.empty()) {
    const int32_t i = stack.back();
    stack.pop_back();
    buf[w++] = t->nodes[(size_t)i].id;
    buf[w++] = t->nodes[(size_t)i].host ? 1 : 0;
    for (auto it = kids[(size_t)i].rbegin(); it != kids[(size_t)i].rend(); ++it)
      stack.push_back(it->second);
  }
  return w;
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

}  // extern "C"

namespace {
// Batch formation over W waiting sequences; sequence w is tokens[start(w), start(w) + len(w)).
// Shared by rc_schedule_batch (contiguous sequences) and rc_schedule_batch_ranges.
template <typename Start, typename Len>
int schedule_impl(const rc_radix* t, const int32_t* tokens, Start start, Len len_of, int32_t B,
                  const int32_t* match_len, int32_t policy, int32_t max_batch,
                  int64_t max_new_tokens, int64_t reserve_slots, int32_t* out_order,
                  int32_t* out_match, int32_t* out_admitted, const char* what) {
  for (int32_t w = 0; w < B; ++w) {
    const int64_t len = len_of(w);
    const int64_t n = match_len ? (int64_t)match_len[w] : len;
    RC_CHECK_ARG(start(w) >= 0 && len >= 0 && n >= 0 && n <= len,
                 "%s: sequence %d: length %lld, match %lld", what, w, (long long)len,
                 (long long)n);
  }
  auto seq = [&](int32_t w) { return tokens + start(w); };
  auto lim = [&](int32_t w) { return match_len ? (int64_t)match_len[w] : len_of(w); };
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
    const int64_t fresh = len_of(w) - out_match[w];
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
}  // namespace

extern "C" {

int rc_schedule_batch(const rc_radix* t, const int32_t* tokens, const int64_t* indptr, int32_t B,
                      const int32_t* match_len, int32_t policy, int32_t max_batch,
                      int64_t max_new_tokens, int64_t reserve_slots, int32_t* out_order,
                      int32_t* out_match, int32_t* out_admitted) {
  RC_CHECK_ARG(t && out_admitted && B >= 0 && max_batch >= 0 && reserve_slots >= 0 &&
                   (policy == RC_SCHED_LSPF || policy == RC_SCHED_FCFS) &&
                   (B == 0 || (tokens && indptr && out_order && out_match)),
               "rc_schedule_batch: bad argument");
  return schedule_impl(
      t, tokens, [&](int32_t w) { return indptr[w]; },
      [&](int32_t w) { return indptr[w + 1] - indptr[w]; }, B, match_len, policy, max_batch,
      max_new_tokens, reserve_slots, out_order, out_match, out_admitted, "rc_schedule_batch");
}

int rc_schedule_batch_ranges(const rc_radix* t, const int32_t* tokens, const int64_t* starts,
                             const int64_t* lengths, int32_t W, const int32_t* match_len,
                             int32_t policy, int32_t max_batch, int64_t max_new_tokens,
                             int64_t reserve_slots, int32_t* out_order, int32_t* out_match,
                             int32_t* out_admitted) {
  RC_CHECK_ARG(t && out_admitted && W >= 0 && max_batch >= 0 && reserve_slots >= 0 &&
                   (policy == RC_SCHED_LSPF || policy == RC_SCHED_FCFS) &&
                   (W == 0 || (tokens && starts && lengths && out_order && out_match)),
               "rc_schedule_batch_ranges: bad argument");
  return schedule_impl(
      t, tokens, [&](int32_t w) { return starts[w]; }, [&](int32_t w) { return lengths[w]; }, W,
      match_len, policy, max_batch, max_new_tokens, reserve_slots, out_order, out_match,
      out_admitted, "rc_schedule_batch_ranges");
}

}  // extern "C"
