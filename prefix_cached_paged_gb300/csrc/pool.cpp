// Token pool: the free list of KV pages, one page per token (paper digest Sec. 3: paged KV with
// one token per page, one pool shared by cached and running requests).
//
// The free list is a ring buffer over a fixed array of num_slots entries: alloc pops from the
// head, free pushes at the tail, both O(n) in the slots moved and allocation-free. A bitmap of
// free slots rejects double frees before anything changes.
#include <cstring>
#include <new>
#include <vector>

#include "host_common.h"
#include "pool_impl.h"

using rc::fail;

extern "C" {

int rc_pool_create(int64_t num_slots, const int32_t* initial_order, rc_pool** out) {
  RC_CHECK_ARG(out != nullptr, "rc_pool_create: out is NULL");
  RC_CHECK_ARG(num_slots > 0 && num_slots <= INT32_MAX, "rc_pool_create: num_slots %lld",
               (long long)num_slots);
  rc_pool* p = new (std::nothrow) rc_pool();
  if (!p) return fail(RC_ERR_OOM, "rc_pool_create: host allocation failed");
  p->ring.resize((size_t)num_slots);
  p->is_free.assign((size_t)num_slots, 1);
  p->head = 0;
  p->count = num_slots;
  if (initial_order) {
    std::vector<uint8_t> seen((size_t)num_slots, 0);
    for (int64_t i = 0; i < num_slots; ++i) {
      const int32_t s = initial_order[i];
      if (s < 0 || s >= num_slots || seen[(size_t)s]) {
        delete p;
        return fail(RC_ERR_INVALID, "rc_pool_create: initial_order is not a permutation (at %lld)",
                    (long long)i);
      }
      seen[(size_t)s] = 1;
      p->ring[(size_t)i] = s;
    }
  } else {
    for (int64_t i = 0; i < num_slots; ++i) p->ring[(size_t)i] = (int32_t)i;
  }
  *out = p;
  return RC_OK;
}

void rc_pool_destroy(rc_pool* pool) { delete pool; }

int rc_kv_pool_alloc(rc_pool* p, int64_t n, int32_t* out_slots) {
  RC_CHECK_ARG(p != nullptr, "rc_kv_pool_alloc: pool is NULL");
  RC_CHECK_ARG(n >= 0, "rc_kv_pool_alloc: n = %lld", (long long)n);
  RC_CHECK_ARG(n == 0 || out_slots != nullptr, "rc_kv_pool_alloc: out_slots is NULL");
  if (p->fail_after == 0) {   // the injected failure (rc_pool_inject_alloc_failure)
    p->fail_after = -1;
    return fail(RC_ERR_OOM, "kv_pool_alloc: injected failure (%lld requested, %lld free)",
                (long long)n, (long long)p->count);
  }
  const int rc_take = rc::pool_take(p, n, out_slots);
  if (rc_take == RC_OK && p->fail_after > 0) --p->fail_after;
  return rc_take;
}

int rc_kv_pool_free(rc_pool* p, const int32_t* slots, int64_t n) {
  RC_CHECK_ARG(p != nullptr, "rc_kv_pool_free: pool is NULL");
  RC_CHECK_ARG(n >= 0 && (n == 0 || slots != nullptr), "rc_kv_pool_free: bad slots/n");
  return rc::pool_give(p, slots, n);
}

int rc_kv_pool_available(const rc_pool* p, int64_t* out) {
  RC_CHECK_ARG(p != nullptr && out != nullptr, "rc_kv_pool_available: NULL argument");
  *out = p->count;
  return RC_OK;
}

int rc_pool_inject_alloc_failure(rc_pool* p, int64_t after_calls) {
  RC_CHECK_ARG(p != nullptr, "rc_pool_inject_alloc_failure: pool is NULL");
  RC_CHECK_ARG(after_calls >= -1, "rc_pool_inject_alloc_failure: after_calls = %lld",
               (long long)after_calls);
  p->fail_after = after_calls;
  return RC_OK;
}

}  // extern "C"

namespace rc {

int pool_take(rc_pool* p, int64_t n, int32_t* out) {
  if (n > p->count)
    return fail(RC_ERR_OOM, "kv_pool_alloc: %lld requested, %lld free", (long long)n,
                (long long)p->count);
  const int64_t cap = (int64_t)p->ring.size();
  const int64_t first = std::min<int64_t>(n, cap - p->head);
  std::memcpy(out, p->ring.data() + p->head, (size_t)first * sizeof(int32_t));
  std::memcpy(out + first, p->ring.data(), (size_t)(n - first) * sizeof(int32_t));
  for (int64_t i = 0; i < n; ++i) p->is_free[(size_t)out[i]] = 0;
  p->head = (p->head + n) % cap;
  p->count -= n;
  return RC_OK;
}

int pool_give(rc_pool* p, const int32_t* slots, int64_t n) {
  const int64_t cap = (int64_t)p->ring.size();
  // validate everything first: range, not already free, no repeats within the call
  for (int64_t i = 0; i < n; ++i) {
    const int32_t s = slots[i];
    if (s < 0 || s >= cap || p->is_free[(size_t)s]) {
      for (int64_t j = 0; j < i; ++j) p->is_free[(size_t)slots[j]] = 0;  // undo marks
      return fail(RC_ERR_INVALID, "kv_pool_free: slot %d at %lld is out of range or already free",
                  (int)s, (long long)i);
    }
    p->is_free[(size_t)s] = 1;
  }
  int64_t tail = (p->head + p->count) % cap;
  for (int64_t i = 0; i < n; ++i) {
    p->ring[(size_t)tail] = slots[i];
    tail = tail + 1 == cap ? 0 : tail + 1;
  }
  p->count += n;
  return RC_OK;
}

}  // namespace rc
