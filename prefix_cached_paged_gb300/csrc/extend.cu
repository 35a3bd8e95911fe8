// rc_extend_attention: argument checks and the dtype -> kernel mapping.
//   bf16, head_dim 128 -> the tcgen05 tensor-core kernel (extend_tc.cu)
//   fp32               -> the CUDA-core kernel (extend_simt.cu)
#include "device_common.cuh"
#include "extend_common.h"
#include "host_common.h"

extern "C" int rc_extend_workspace_bytes(const rc_extend_args* a, size_t* out_bytes) {
  RC_CHECK_ARG(a != nullptr && out_bytes != nullptr, "rc_extend_workspace_bytes: NULL argument");
  RC_CHECK_ARG(a->num_tokens >= 0 && a->num_q_heads > 0,
               "rc_extend_workspace_bytes: bad sizes");
  // one fp32 log-sum-exp per (token, query head) for the stacked pass's partial results
  *out_bytes = ((size_t)a->num_tokens * (size_t)a->num_q_heads * sizeof(float) + 255) &
               ~(size_t)255;
  return RC_OK;
}

extern "C" int rc_extend_attention(const rc_extend_args* a, void* stream) {
  RC_CHECK_ARG(a != nullptr, "rc_extend_attention: args is NULL");
  RC_CHECK_ARG(a->dtype == RC_DTYPE_BF16 || a->dtype == RC_DTYPE_F32,
               "rc_extend_attention: dtype %d", a->dtype);
  RC_CHECK_ARG(a->num_reqs >= 0 && a->num_q_heads > 0 && a->num_kv_heads > 0 &&
                   a->num_q_heads % a->num_kv_heads == 0,
               "rc_extend_attention: bad head counts");
  RC_CHECK_ARG(a->head_dim == 128 || (a->dtype == RC_DTYPE_F32 && a->head_dim == 64),
               "rc_extend_attention: head_dim %d unsupported for this dtype", a->head_dim);
  RC_CHECK_ARG(a->max_ctx > 0 && a->max_ctx % 4 == 0 && a->max_reqs > 0,
               "rc_extend_attention: max_ctx %d / max_reqs %d", a->max_ctx, a->max_reqs);
  RC_CHECK_ARG(a->max_q_len >= 0 && a->max_prefix_len >= 0 && a->num_tokens >= 0 &&
                   a->num_slots > 0,
               "rc_extend_attention: bad sizes");
  if (a->num_reqs == 0 || a->num_tokens == 0 || a->max_q_len == 0) return RC_OK;
  RC_CHECK_ARG(a->q && a->k_new && a->v_new && a->out_loc && a->qo_indptr && a->prefix_len &&
                   a->req_idx && a->req_to_token && a->k_pool && a->v_pool && a->o,
               "rc_extend_attention: NULL pointer");
  const uintptr_t al = (uintptr_t)a->q | (uintptr_t)a->k_new | (uintptr_t)a->v_new |
                       (uintptr_t)a->k_pool | (uintptr_t)a->v_pool | (uintptr_t)a->o |
                       (uintptr_t)a->req_to_token;
  RC_CHECK_ARG((al & 15) == 0, "rc_extend_attention: tensors must be 16-byte aligned");
  RC_CHECK_ARG(a->num_groups >= 0, "rc_extend_attention: num_groups %d", a->num_groups);
  if (a->num_groups > 0 && a->dtype == RC_DTYPE_BF16) {
    RC_CHECK_ARG(a->group_range && a->group_shared && a->max_group_rows > 0,
                 "rc_extend_attention: stacking groups need group_range, group_shared and "
                 "max_group_rows");
    size_t need = 0;
    rc_extend_workspace_bytes(a, &need);
    RC_CHECK_ARG(a->workspace && ((uintptr_t)a->workspace & 15) == 0 && a->workspace_bytes >= need,
                 "rc_extend_attention: stacking needs a 16-byte aligned workspace of %zu bytes",
                 need);
    RC_CHECK_ARG(a->num_levels >= 0 && a->num_levels <= RC_MAX_STACK_LEVELS,
                 "rc_extend_attention: num_levels %d (at most %d)", a->num_levels,
                 RC_MAX_STACK_LEVELS);
    if (a->num_levels > 1) {
      RC_CHECK_ARG(a->level_indptr && a->level_indptr[0] == 0 &&
                       a->level_indptr[a->num_levels] == a->num_groups,
                   "rc_extend_attention: level_indptr must run from 0 to num_groups");
      for (int l = 0; l < a->num_levels; ++l)
        RC_CHECK_ARG(a->level_indptr[l + 1] > a->level_indptr[l],
                     "rc_extend_attention: level %d holds no group", l);
    }
  }
  int* st = rc::device_status_ptr();
  if (!st) return rc::fail(RC_ERR_CUDA, "rc_extend_attention: no device status word");
  cudaStream_t s = (cudaStream_t)stream;
  if (a->dtype == RC_DTYPE_BF16) return rc::launch_extend_tc(a, st, s);
  return rc::launch_extend_simt(a, st, s);
}
