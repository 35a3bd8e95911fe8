// Internal layout of rc_pool, shared by the pool and the radix tree (which frees into it).
#pragma once
#include <algorithm>
#include <cstdint>
#include <vector>

#include "rc.h"

struct rc_pool {
  std::vector<int32_t> ring;     // free list, num_slots entries, valid from head for count
  std::vector<uint8_t> is_free;  // 1 if the slot is on the free list
  int64_t head = 0;
  int64_t count = 0;
  int64_t fail_after = -1;       // injected failure: takes left before one fails (-1: none)
};

namespace rc {
int pool_take(rc_pool* p, int64_t n, int32_t* out);
int pool_give(rc_pool* p, const int32_t* slots, int64_t n);
inline int64_t pool_free_count(const rc_pool* p) { return p->count; }
}  // namespace rc
