// Shared host-side helpers of librc: thread-local error messages and the launch counter.
#pragma once
#include <atomic>
#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <string>

#include "rc.h"

namespace rc {

// Record a failure message for rc_last_error() and return `code`.
int fail(int code, const char* fmt, ...);
void clear_error();
void count_launches(uint64_t n);

}  // namespace rc

#define RC_CHECK_ARG(cond, ...)                     \
  do {                                              \
    if (!(cond)) return ::rc::fail(RC_ERR_INVALID, __VA_ARGS__); \
  } while (0)

#define RC_CHECK(cond, code, ...)                     \
  do {                                                \
    if (!(cond)) return ::rc::fail((code), __VA_ARGS__); \
  } while (0)
