// Slot-table write: req_to_token[row, col + j] = values[indptr + j] for a batch of segments.
// One CTA per segment, threads stride over the segment; bounds are checked per segment.
#include "device_common.cuh"
#include "host_common.h"

namespace rc {
namespace {

__global__ void slot_table_write_kernel(rc_slot_write_args a, int* status) {
  const int i = blockIdx.x;
  const int row = a.seg_row[i];
  const int col = a.seg_col[i];
  const int beg = a.seg_indptr[i];
  const int len = a.seg_indptr[i + 1] - beg;
  if (row < 0 || row >= a.max_reqs || col < 0 || len < 0 || (int64_t)col + len > a.max_ctx ||
      beg < 0 || (int64_t)beg + len > a.total_values) {
    if (threadIdx.x == 0) set_status(status, kStatusPosRange);
    return;
  }
  int32_t* dst = a.req_to_token + (int64_t)row * a.max_ctx + col;
  const int32_t* src = a.values + beg;
  for (int j = threadIdx.x; j < len; j += blockDim.x) dst[j] = src[j];
}

}  // namespace
}  // namespace rc

extern "C" int rc_slot_table_write(const rc_slot_write_args* a, void* stream) {
  RC_CHECK_ARG(a != nullptr, "rc_slot_table_write: args is NULL");
  RC_CHECK_ARG(a->num_segments >= 0 && a->max_reqs > 0 && a->max_ctx > 0 && a->total_values >= 0,
               "rc_slot_table_write: bad sizes");
  if (a->num_segments == 0) return RC_OK;
  RC_CHECK_ARG(a->seg_row && a->seg_col && a->seg_indptr && a->req_to_token &&
                   (a->total_values == 0 || a->values),
               "rc_slot_table_write: NULL pointer");
  int* st = rc::device_status_ptr();
  if (!st) return rc::fail(RC_ERR_CUDA, "rc_slot_table_write: no device status word");
  rc::slot_table_write_kernel<<<a->num_segments, 256, 0, (cudaStream_t)stream>>>(*a, st);
  rc::count_launches(1);
  return rc::check_launch("rc_slot_table_write");
}
