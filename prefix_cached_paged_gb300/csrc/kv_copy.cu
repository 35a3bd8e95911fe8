// Slot-to-slot KV row copies between two pools: device planes and the host tier's pinned host
// planes (SGLang blog Sec. 6.1 HiCache: GPU memory holds the hottest KV, host memory the next
// tier). On a Grace-Blackwell node the GPU reads and writes pinned host memory directly over the
// chip-to-chip link, so a spill (device -> host) or a load (host -> device) is one kernel that
// gathers rows by slot index on one side and scatters them on the other: no staging buffer and
// no separate memcpy per node.
//
// Work split: one warp per (copy, layer, K or V) row, 16-byte chunks, each lane keeping four
// chunks in flight; a grid-stride loop over rows. Slot indices outside their pool set the
// device status word and the row is skipped.
#include <algorithm>

#include "device_common.cuh"
#include "host_common.h"

namespace rc {
namespace {

constexpr int kThreads = 256;
constexpr int kUnroll = 4;

__global__ void __launch_bounds__(kThreads) kv_copy_kernel(rc_kv_copy_args a, int* status) {
  const int lane = threadIdx.x & 31;
  const int64_t warps = (int64_t)gridDim.x * (kThreads / 32);
  const int64_t cpr = a.row_bytes >> 4;                  // 16-byte chunks per row
  const int64_t rows = a.n * a.layers * 2;
  for (int64_t r = (int64_t)blockIdx.x * (kThreads / 32) + (threadIdx.x >> 5); r < rows;
       r += warps) {
    const int t = (int)(r & 1);                          // 0: K, 1: V
    const int64_t il = r >> 1;
    const int64_t i = il / a.layers;
    const int64_t layer = il - i * a.layers;
    const int32_t s = a.src_slots[i];
    const int32_t d = a.dst_slots[i];
    if (s < 0 || s >= a.src_num_slots || d < 0 || d >= a.dst_num_slots) {
      if (lane == 0) set_status(status, kStatusSlotRange);
      continue;
    }
    const char* src = (const char*)(t ? a.src_v : a.src_k) +
                      ((layer * a.src_num_slots + s) * a.row_bytes);
    char* dst = (char*)(t ? a.dst_v : a.dst_k) + ((layer * a.dst_num_slots + d) * a.row_bytes);
    const uint4* s4 = (const uint4*)src;
    uint4* d4 = (uint4*)dst;
    for (int64_t c0 = lane; c0 < cpr; c0 += 32 * kUnroll) {
      uint4 v[kUnroll];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int64_t c = c0 + 32 * u;
        if (c < cpr) v[u] = s4[c];
      }
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int64_t c = c0 + 32 * u;
        if (c < cpr) d4[c] = v[u];
      }
    }
  }
}

}  // namespace
}  // namespace rc

extern "C" int rc_kv_copy(const rc_kv_copy_args* a, void* stream) {
  RC_CHECK_ARG(a != nullptr, "rc_kv_copy: args is NULL");
  RC_CHECK_ARG(a->n >= 0 && a->layers > 0 && a->row_bytes > 0 && a->row_bytes % 16 == 0 &&
                   a->src_num_slots > 0 && a->dst_num_slots > 0,
               "rc_kv_copy: bad sizes (row_bytes must be a positive multiple of 16)");
  if (a->n == 0) return RC_OK;
  RC_CHECK_ARG(a->src_slots && a->dst_slots && a->src_k && a->src_v && a->dst_k && a->dst_v,
               "rc_kv_copy: NULL pointer");
  RC_CHECK_ARG((((uintptr_t)a->src_k | (uintptr_t)a->src_v | (uintptr_t)a->dst_k |
                 (uintptr_t)a->dst_v) & 15) == 0,
               "rc_kv_copy: planes must be 16-byte aligned");
  int* st = rc::device_status_ptr();
  if (!st) return rc::fail(RC_ERR_CUDA, "rc_kv_copy: no device status word");
  int sms = 0, dev = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int64_t rows = a->n * a->layers * 2;
  const int64_t want = (rows + rc::kThreads / 32 - 1) / (rc::kThreads / 32);
  const int blocks = (int)std::min<int64_t>(want, (int64_t)std::max(sms, 1) * 8);
  rc::kv_copy_kernel<<<blocks, rc::kThreads, 0, (cudaStream_t)stream>>>(*a, st);
  rc::count_launches(1);
  return rc::check_launch("rc_kv_copy");
}
