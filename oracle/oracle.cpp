// Oracle for prefix-cached paged attention -- TEST INFRASTRUCTURE ONLY.
//
// A plain, slow, obviously correct CPU restatement of what the hot path computes. Only the test
// suite, the smoke check and the benchmark's CPU-baseline leg may load it; the product library
// never does, and the two share no code.
//
// What it restates (SGLang, "Efficient Execution of Structured Language Model Programs",
// arXiv 2312.07104, as summarised on the pages):
//   * a token-granular KV pool: one page per token, one free list shared by cached and running
//     requests (paper digest, Sec. 3 "RadixAttention": paged storage, one token per page, shared
//     memory pool);
//   * a radix tree whose edges are token sequences and whose nodes carry the pool slots of their
//     edge; longest-prefix match, insert with node split, per-node reference counts, and LRU
//     eviction of unreferenced leaves (paper digest Sec. 3 and Fig. 3; SGLang blog Sec. 2.3
//     "traverse / reuse / compute / insert" and "leaf first"; RadixAttention explainer
//     "insert, match, split, evict");
//   * attention of each query over all keys at positions <= its own, as the textbook softmax
//     definition in fp64 (paper digest App. A.1: KV of a token depends only on the tokens before
//     it, so reused KV equals recomputed KV).
//
// Readings where the pages are silent (each also listed in the design notes):
//   * match splits the edge where the match ends inside it; the new node is the matched (upper)
//     part, gets a fresh id and the lower part keeps the old id; both keep the old stamp and the
//     upper part copies the reference count;
//   * every match and insert stamps the nodes on its path root-to-leaf with a logical clock
//     (+1 per node), so deeper nodes are newer; eviction takes the unreferenced leaf with the
//     smallest (stamp, id) and repeats until enough tokens are freed; whole nodes only;
//   * alloc takes slots from the head of the free list, free appends at the tail in the order
//     given, eviction frees a node's slots in token order;
//   * insert keeps the slots already in the tree and reports how many leading tokens were
//     already present.
//
// Parity pins: brute-force per-token trie, LRU scenario, worked few-shot count, attention closed
// forms and the reuse invariant (see tests/test_oracle_*.py).

#include <cmath>
#include <cstdint>
#include <cstring>
#include <deque>
#include <map>
#include <thread>
#include <vector>
#include <algorithm>

namespace {

struct Pool {
  int64_t num_slots = 0;
  std::deque<int32_t> free_list;
};

struct Node {
  int64_t id = 0;
  Node* parent = nullptr;
  std::vector<int32_t> key;
  std::vector<int32_t> slots;
  std::map<int32_t, Node*> children;  // keyed by the first token of the child's edge
  int64_t ref = 0;
  int64_t stamp = 0;
  bool host = false;  // KV held in host-tier slots
};

struct Copy {
  int32_t src, dst;
};

struct Tree {
  Pool* pool = nullptr;
  Node* root = nullptr;
  int64_t clock = 0;
  int64_t next_id = 1;  // the root has id 0
  std::map<int64_t, Node*> by_id;
  int64_t splits = 0, evicted_nodes = 0, evicted_tokens = 0;
  Pool* host = nullptr;                     // host tier, or none
  std::vector<Copy> spills, loads;          // owed copies; a spill with dst -1 is cancelled
  int64_t host_tokens = 0, spilled = 0, loaded = 0, dropped = 0;
};

Node* new_node(Tree* t) {
  Node* n = new Node();
  n->id = t->next_id++;
  t->by_id[n->id] = n;
  return n;
}

// Split `child` after its first `k` tokens. Returns the new upper node.
Node* split(Tree* t, Node* child, size_t k) {
  Node* up = new_node(t);
  Node* par = child->parent;
  up->parent = par;
  up->key.assign(child->key.begin(), child->key.begin() + k);
  up->slots.assign(child->slots.begin(), child->slots.begin() + k);
  up->ref = child->ref;
  up->stamp = child->stamp;
  up->host = child->host;
  child->key.erase(child->key.begin(), child->key.begin() + k);
  child->slots.erase(child->slots.begin(), child->slots.begin() + k);
  child->parent = up;
  up->children[child->key[0]] = child;
  par->children[up->key[0]] = up;
  t->splits++;
  return up;
}

void touch_path(Tree* t, Node* last) {
  std::vector<Node*> path;
  for (Node* n = last; n != t->root; n = n->parent) path.push_back(n);
  for (auto it = path.rbegin(); it != path.rend(); ++it) (*it)->stamp = ++t->clock;
}

// Cancel the owed spill copies that write into any of these host slots.
void cancel_spills_into(Tree* t, const std::vector<int32_t>& host_slots) {
  for (Copy& c : t->spills)
    for (int32_t h : host_slots)
      if (c.dst == h) c.dst = -1;
}

bool has_device_child(const Node* x) {
  for (auto& kv : x->children)
    if (!kv.second->host) return true;
  return false;
}

void remove_leaf(Tree* t, Node* x) {
  x->parent->children.erase(x->key[0]);
  t->by_id.erase(x->id);
  delete x;
}

void free_node(Tree* t, Node* n) {
  for (auto& kv : n->children) free_node(t, kv.second);
  t->by_id.erase(n->id);
  delete n;
}

}  // namespace

extern "C" {

// ----- pool -----
void* or_pool_create(int64_t num_slots, const int32_t* order) {
  Pool* p = new Pool();
  p->num_slots = num_slots;
  for (int64_t i = 0; i < num_slots; ++i) p->free_list.push_back(order ? order[i] : (int32_t)i);
  return p;
}
void or_pool_destroy(void* p) { delete (Pool*)p; }
int64_t or_pool_available(void* p) { return (int64_t)((Pool*)p)->free_list.size(); }
// all or nothing: returns 0 on success, -1 when fewer than n slots are free
int or_pool_alloc(void* pv, int64_t n, int32_t* out) {
  Pool* p = (Pool*)pv;
  if ((int64_t)p->free_list.size() < n) return -1;
  for (int64_t i = 0; i < n; ++i) {
    out[i] = p->free_list.front();
    p->free_list.pop_front();
  }
  return 0;
}
void or_pool_free(void* pv, const int32_t* slots, int64_t n) {
  Pool* p = (Pool*)pv;
  for (int64_t i = 0; i < n; ++i) p->free_list.push_back(slots[i]);
}

// ----- tree -----
void* or_tree_create(void* pool) {
  Tree* t = new Tree();
  t->pool = (Pool*)pool;
  t->root = new Node();
  t->root->id = 0;
  t->by_id[0] = t->root;
  return t;
}
void or_tree_destroy(void* tv) {
  Tree* t = (Tree*)tv;
  free_node(t, t->root);
  delete t;
}

// Longest cached prefix of tok[0:n]. Writes its slots, its length and the id of the node where it
// ends (0 = root). Splits the edge when the match ends inside it. Stamps the path.
void or_match(void* tv, const int32_t* tok, int64_t n, int32_t* out_slots, int64_t* out_len,
              int64_t* out_node) {
  Tree* t = (Tree*)tv;
  Node* cur = t->root;
  int64_t pos = 0;
  while (pos < n) {
    auto it = cur->children.find(tok[pos]);
    if (it == cur->children.end() || it->second->host) break;
    Node* child = it->second;
    size_t k = 0;
    while (k < child->key.size() && pos + (int64_t)k < n && child->key[k] == tok[pos + k]) ++k;
    const bool ends_inside = k < child->key.size();
    if (ends_inside) child = split(t, child, k);
    for (size_t i = 0; i < k; ++i) out_slots[pos + i] = child->slots[i];
    pos += (int64_t)k;
    cur = child;
    if (ends_inside) break;
  }
  touch_path(t, cur);
  *out_len = pos;
  *out_node = cur->id;
}

// Insert tok[0:n] with slots[0:n]. Existing tokens keep their slots; *out_existing = how many
// leading tokens were already present. *out_node = id of the node where the sequence ends.
void or_insert(void* tv, const int32_t* tok, const int32_t* slots, int64_t n, int64_t* out_existing,
               int64_t* out_node) {
  Tree* t = (Tree*)tv;
  Node* cur = t->root;
  int64_t pos = 0, existing = -1;
  while (pos < n) {
    auto it = cur->children.find(tok[pos]);
    if (it == cur->children.end()) {
      Node* leaf = new_node(t);
      leaf->parent = cur;
      leaf->key.assign(tok + pos, tok + n);
      leaf->slots.assign(slots + pos, slots + n);
      cur->children[tok[pos]] = leaf;
      cur = leaf;
      if (existing < 0) existing = pos;
      pos = n;
      break;
    }
    Node* child = it->second;
    size_t k = 0;
    while (k < child->key.size() && pos + (int64_t)k < n && child->key[k] == tok[pos + k]) ++k;
    if (k < child->key.size()) child = split(t, child, k);
    if (child->host) {
      // tokens held in the host tier take the caller's slots; the host copy is released
      if (existing < 0) existing = pos;
      or_pool_free(t->host, child->slots.data(), (int64_t)child->slots.size());
      cancel_spills_into(t, child->slots);
      child->slots.assign(slots + pos, slots + pos + k);
      child->host = false;
      t->host_tokens -= (int64_t)k;
    }
    pos += (int64_t)k;
    cur = child;
  }
  touch_path(t, cur);
  *out_node = cur->id;
  // present = the leading device-resident tokens: the walk stopped at n (all present), at the
  // first host-resident node, or where the new leaf starts
  *out_existing = existing >= 0 ? existing : pos;
}

int or_lock(void* tv, int64_t node_id) {
  Tree* t = (Tree*)tv;
  auto it = t->by_id.find(node_id);
  if (it == t->by_id.end()) return -1;
  for (Node* x = it->second; x != t->root; x = x->parent) x->ref += 1;
  return 0;
}
int or_unlock(void* tv, int64_t node_id) {
  Tree* t = (Tree*)tv;
  auto it = t->by_id.find(node_id);
  if (it == t->by_id.end()) return -1;
  for (Node* x = it->second; x != t->root; x = x->parent)
    if (x->ref <= 0) return -2;
  for (Node* x = it->second; x != t->root; x = x->parent) x->ref -= 1;
  return 0;
}

// Evict unreferenced leaves in LRU order until at least n tokens are freed. Returns 0 if enough
// were freed, -1 otherwise; *out_freed = tokens freed. Evicted node ids go to out_ids (cap ids).
int or_evict(void* tv, int64_t n, int64_t* out_freed, int64_t* out_ids, int64_t cap,
             int64_t* out_nids) {
  Tree* t = (Tree*)tv;
  int64_t freed = 0, nids = 0;
  if (t->host && !t->loads.empty()) return -2;   // loads owed: drain first
  while (freed < n) {
    // the least recently used device leaf: device-resident, unreferenced, no device child
    Node* best = nullptr;
    for (auto& kv : t->by_id) {
      Node* x = kv.second;
      if (x == t->root || x->host || x->ref != 0 || has_device_child(x)) continue;
      if (!best || x->stamp < best->stamp || (x->stamp == best->stamp && x->id < best->id))
        best = x;
    }
    if (!best) break;
    const int64_t len = (int64_t)best->slots.size();
    or_pool_free(t->pool, best->slots.data(), len);
    freed += len;
    if (out_ids && nids < cap) out_ids[nids] = best->id;
    nids++;
    t->evicted_nodes++;
    t->evicted_tokens += len;
    if (t->host) {
      // drop the least recently used host leaves until the host tier can take it
      while ((int64_t)t->host->free_list.size() < len) {
        Node* h = nullptr;
        for (auto& kv : t->by_id) {
          Node* x = kv.second;
          if (x == t->root || !x->host || x->ref != 0 || !x->children.empty()) continue;
          if (!h || x->stamp < h->stamp || (x->stamp == h->stamp && x->id < h->id)) h = x;
        }
        if (!h) break;
        or_pool_free(t->host, h->slots.data(), (int64_t)h->slots.size());
        cancel_spills_into(t, h->slots);
        t->host_tokens -= (int64_t)h->slots.size();
        t->dropped += (int64_t)h->slots.size();
        remove_leaf(t, h);
      }
      if ((int64_t)t->host->free_list.size() >= len) {
        std::vector<int32_t> hs((size_t)len);
        or_pool_alloc(t->host, len, hs.data());
        for (int64_t k = 0; k < len; ++k) t->spills.push_back({best->slots[k], hs[k]});
        best->slots = hs;
        best->host = true;
        t->host_tokens += len;
        t->spilled += len;
        continue;
      }
      t->dropped += len;   // not even an emptied host tier takes it; it has no child left
    }
    remove_leaf(t, best);
  }
  *out_freed = freed;
  if (out_nids) *out_nids = nids;
  return freed >= n ? 0 : -1;
}

// ----- host tier -----
void or_attach_host(void* tv, void* host_pool) { ((Tree*)tv)->host = (Pool*)host_pool; }

// Match through both tiers: *out_dev = device-resident tokens matched (their slots written),
// *out_host = host-resident tokens matched after them; splits where the match ends, stamps the
// path. *out_node = the node where it ends.
void or_match_tiered(void* tv, const int32_t* tok, int64_t n, int32_t* out_slots,
                     int64_t* out_dev, int64_t* out_host, int64_t* out_node) {
  Tree* t = (Tree*)tv;
  Node* cur = t->root;
  int64_t pos = 0, dev = 0;
  while (pos < n) {
    auto it = cur->children.find(tok[pos]);
    if (it == cur->children.end()) break;
    Node* child = it->second;
    size_t k = 0;
    while (k < child->key.size() && pos + (int64_t)k < n && child->key[k] == tok[pos + k]) ++k;
    const bool ends_inside = k < child->key.size();
    if (ends_inside) child = split(t, child, k);
    if (!child->host) {
      for (size_t i = 0; i < k; ++i) out_slots[pos + i] = child->slots[i];
      dev = pos + (int64_t)k;
    }
    pos += (int64_t)k;
    cur = child;
    if (ends_inside) break;
  }
  touch_path(t, cur);
  *out_dev = dev;
  *out_host = pos - dev;
  *out_node = cur->id;
}

// Move the host-resident nodes on the path of tok[0:n] back to the device: fresh device slots
// per node (token order), a load copy per token; the host slots are released at the drain.
// Writes the path's slots to row[0:n]. Returns 0, or -1 if the device pool is short.
int or_load(void* tv, const int32_t* tok, int64_t n, int32_t* row) {
  Tree* t = (Tree*)tv;
  Node* cur = t->root;
  int64_t pos = 0;
  while (pos < n) {
    Node* child = cur->children.at(tok[pos]);
    const int64_t len = (int64_t)child->key.size();
    if (child->host) {
      std::vector<int32_t> ds((size_t)len);
      if (or_pool_alloc(t->pool, len, ds.data()) != 0) return -1;
      for (int64_t k = 0; k < len; ++k) t->loads.push_back({child->slots[k], ds[k]});
      child->slots = ds;
      child->host = false;
      t->host_tokens -= len;
      t->loaded += len;
    }
    for (int64_t k = 0; k < len; ++k) row[pos + k] = child->slots[k];
    pos += len;
    cur = child;
  }
  return 0;
}

void or_pending(void* tv, int64_t* n_spill, int64_t* n_load) {
  Tree* t = (Tree*)tv;
  int64_t ns = 0;
  for (const Copy& c : t->spills) ns += c.dst >= 0;
  *n_spill = ns;
  *n_load = (int64_t)t->loads.size();
}

void or_drain(void* tv, int32_t* sd, int32_t* sh, int32_t* lh, int32_t* ld) {
  Tree* t = (Tree*)tv;
  int64_t w = 0;
  for (const Copy& c : t->spills)
    if (c.dst >= 0) {
      sd[w] = c.src;
      sh[w] = c.dst;
      ++w;
    }
  for (size_t i = 0; i < t->loads.size(); ++i) {
    lh[i] = t->loads[i].src;
    ld[i] = t->loads[i].dst;
    or_pool_free(t->host, &t->loads[i].src, 1);
  }
  t->spills.clear();
  t->loads.clear();
}

// (id, 1 if host-resident) per node, in the dump's order.
int64_t or_tiers(void* tv, int64_t* buf, int64_t cap) {
  Tree* t = (Tree*)tv;
  std::vector<int64_t> out;
  std::vector<Node*> stack;
  for (auto it = t->root->children.rbegin(); it != t->root->children.rend(); ++it)
    stack.push_back(it->second);
  while (!stack.empty()) {
    Node* x = stack.back();
    stack.pop_back();
    out.push_back(x->id);
    out.push_back(x->host ? 1 : 0);
    for (auto it = x->children.rbegin(); it != x->children.rend(); ++it) stack.push_back(it->second);
  }
  if ((int64_t)out.size() > cap) return -(int64_t)out.size();
  std::memcpy(buf, out.data(), out.size() * sizeof(int64_t));
  return (int64_t)out.size();
}

// Canonical dump: depth-first, children in ascending first-token order. Per node (root excluded):
// id, parent id, ref, stamp, len, len tokens, len slots. Returns the number of int64 written, or
// the number needed (negated) if cap is too small.
int64_t or_dump(void* tv, int64_t* buf, int64_t cap) {
  Tree* t = (Tree*)tv;
  std::vector<int64_t> out;
  std::vector<Node*> stack;
  for (auto it = t->root->children.rbegin(); it != t->root->children.rend(); ++it)
    stack.push_back(it->second);
  while (!stack.empty()) {
    Node* x = stack.back();
    stack.pop_back();
    out.push_back(x->id);
    out.push_back(x->parent->id);
    out.push_back(x->ref);
    out.push_back(x->stamp);
    out.push_back((int64_t)x->key.size());
    for (int32_t v : x->key) out.push_back(v);
    for (int32_t v : x->slots) out.push_back(v);
    for (auto it = x->children.rbegin(); it != x->children.rend(); ++it) stack.push_back(it->second);
  }
  if ((int64_t)out.size() > cap) return -(int64_t)out.size();
  std::memcpy(buf, out.data(), out.size() * sizeof(int64_t));
  return (int64_t)out.size();
}

// counters: [splits, evicted_nodes, evicted_tokens, node_count (excl. root), cached_tokens,
//            protected_tokens (ref > 0), host_tokens, spilled, loaded, dropped]; cached and
//            protected count device-resident nodes only
void or_stats(void* tv, int64_t* out) {
  Tree* t = (Tree*)tv;
  int64_t nodes = 0, cached = 0, prot = 0;
  for (auto& kv : t->by_id) {
    if (kv.second == t->root) continue;
    nodes++;
    if (kv.second->host) continue;
    cached += (int64_t)kv.second->key.size();
    if (kv.second->ref > 0) prot += (int64_t)kv.second->key.size();
  }
  out[0] = t->splits;
  out[1] = t->evicted_nodes;
  out[2] = t->evicted_tokens;
  out[3] = nodes;
  out[4] = cached;
  out[5] = prot;
  out[6] = t->host_tokens;
  out[7] = t->spilled;
  out[8] = t->loaded;
  out[9] = t->dropped;
}

// ----- attention -----
// One request: queries at absolute positions P .. P+S-1 over keys 0 .. P+S-1.
// q [S, Hq, d], k and v [P+S, Hkv, d], all fp64. Query head h reads kv head h / (Hq / Hkv).
// out [S, Hq, d]; lse [S, Hq] (natural log of the softmax denominator of the scaled scores).
// O[i,h] = sum_{j <= P+i} softmax_j(scale * <q_i,h , k_j,h'>) v_j,h'
void or_attention(const double* q, const double* k, const double* v, int64_t P, int64_t S,
                  int64_t Hq, int64_t Hkv, int64_t d, double scale, double* out, double* lse) {
  const int64_t g = Hq / Hkv;
  std::vector<double> s(P + S);
  for (int64_t i = 0; i < S; ++i) {
    const int64_t nkeys = P + i + 1;
    for (int64_t h = 0; h < Hq; ++h) {
      const int64_t hk = h / g;
      const double* qi = q + (i * Hq + h) * d;
      double m = -INFINITY;
      for (int64_t j = 0; j < nkeys; ++j) {
        const double* kj = k + (j * Hkv + hk) * d;
        double dot = 0.0;
        for (int64_t c = 0; c < d; ++c) dot += qi[c] * kj[c];
        s[j] = scale * dot;
        if (s[j] > m) m = s[j];
      }
      double den = 0.0;
      for (int64_t j = 0; j < nkeys; ++j) den += std::exp(s[j] - m);
      double* oi = out + (i * Hq + h) * d;
      for (int64_t c = 0; c < d; ++c) oi[c] = 0.0;
      for (int64_t j = 0; j < nkeys; ++j) {
        const double w = std::exp(s[j] - m) / den;
        const double* vj = v + (j * Hkv + hk) * d;
        for (int64_t c = 0; c < d; ++c) oi[c] += w * vj[c];
      }
      if (lse) lse[i * Hq + h] = m + std::log(den);
    }
  }
}

// Many independent requests (units) on `threads` host threads; unit u has its own pointers.
// Used only to time the oracle as a CPU baseline.
void or_attention_units(int64_t nunits, const double* const* q, const double* const* k,
                        const double* const* v, const int64_t* P, const int64_t* S, int64_t Hq,
                        int64_t Hkv, int64_t d, double scale, double* const* out, int64_t threads) {
  if (threads < 1) threads = 1;
  std::vector<std::thread> pool;
  for (int64_t w = 0; w < threads; ++w) {
    pool.emplace_back([=]() {
      for (int64_t u = w; u < nunits; u += threads)
        or_attention(q[u], k[u], v[u], P[u], S[u], Hq, Hkv, d, scale, out[u], nullptr);
    });
  }
  for (auto& th : pool) th.join();
}

// Combine partial attention states: n parts with (o_i [d], lse_i) over disjoint key sets.
// O = sum_i exp(lse_i - M) o_i / sum_i exp(lse_i - M), M = max_i lse_i; lse = M + log(sum).
void or_merge(const double* o_parts, const double* lse_parts, int64_t n, int64_t d, double* out,
              double* out_lse) {
  double M = -INFINITY;
  for (int64_t i = 0; i < n; ++i) M = std::max(M, lse_parts[i]);
  double den = 0.0;
  for (int64_t c = 0; c < d; ++c) out[c] = 0.0;
  for (int64_t i = 0; i < n; ++i) {
    const double w = std::exp(lse_parts[i] - M);
    den += w;
    for (int64_t c = 0; c < d; ++c) out[c] += w * o_parts[i * d + c];
  }
  for (int64_t c = 0; c < d; ++c) out[c] /= den;
  if (out_lse) *out_lse = M + std::log(den);
}

}  // extern "C"
