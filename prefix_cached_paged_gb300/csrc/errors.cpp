// rc_last_error / rc_launch_count.
#include "host_common.h"

namespace rc {
namespace {
thread_local std::string g_last_error;
std::atomic<uint64_t> g_launches{0};
}  // namespace

int fail(int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return code;
}
void clear_error() { g_last_error.clear(); }
void count_launches(uint64_t n) { g_launches.fetch_add(n, std::memory_order_relaxed); }
}  // namespace rc

extern "C" const char* rc_last_error(void) { return rc::g_last_error.c_str(); }
extern "C" uint64_t rc_launch_count(void) { return rc::g_launches.load(); }
