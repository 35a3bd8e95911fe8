// The device status word: kernels that meet bad data (an out-of-range slot or position, an
// expired wait) record a code here instead of trapping, and the host reads it back.
#include <atomic>
#include <mutex>

#include "device_common.cuh"
#include "host_common.h"

namespace {
__device__ int g_status_word;
int* g_status_ptr[rc::kMaxDevices] = {};
std::mutex g_status_mu;
}  // namespace

namespace rc {

int* device_status_ptr() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lk(g_status_mu);
  if (!g_status_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) return nullptr;
    g_status_ptr[dev] = (int*)p;
  }
  return g_status_ptr[dev];
}

namespace {
std::atomic<uint64_t> g_wait_limit_ns{0};
}  // namespace

uint64_t wait_limit_ns() {
  const uint64_t v = g_wait_limit_ns.load();
  return v ? v : 2000000000ull;
}

int check_launch(const char* what) {
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fail(RC_ERR_CUDA, "%s: launch failed: %s", what, cudaGetErrorString(e));
  return RC_OK;
}

}  // namespace rc

extern "C" int rc_device_status(int32_t* out_code, void* stream) {
  RC_CHECK_ARG(out_code != nullptr, "rc_device_status: out_code is NULL");
  int* p = rc::device_status_ptr();
  if (!p) return rc::fail(RC_ERR_CUDA, "rc_device_status: no device status word");
  cudaStream_t s = (cudaStream_t)stream;
  int v = 0;
  cudaError_t e = cudaMemcpyAsync(&v, p, sizeof(int), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e == cudaSuccess && v != 0) e = cudaMemsetAsync(p, 0, sizeof(int), s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return rc::fail(RC_ERR_CUDA, "rc_device_status: %s", cudaGetErrorString(e));
  *out_code = v;
  return RC_OK;
}

extern "C" int rc_debug_set_wait_limit_ns(uint64_t ns) {
  rc::g_wait_limit_ns.store(ns);
  return RC_OK;
}
