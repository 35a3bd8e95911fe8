// Extend attention on CUDA cores: the fp32 path (tcgen05 has no fp32-input kind, and tf32
// would round the inputs). Same contract as the tensor-core bf16 kernel: new tokens' queries
// attend to their request's cached prefix (gathered through the slot table) and causally to the
// new tokens; the new K/V rows are scattered to their pool slots.
//
// One CTA per (16 query rows, query head, request); keys stream through shared memory in tiles
// of 32; each warp owns 4 query rows, one key per lane for the scores, head_dim/32 output
// columns per lane for P.V, online softmax in base 2.
#include "device_common.cuh"
#include "host_common.h"
#include "extend_common.h"

namespace rc {
namespace {

constexpr int kRows = 16;
constexpr int kKeys = 32;

template <typename T, int D>
__global__ void __launch_bounds__(128) extend_simt_kernel(rc_extend_args a, int* status) {
  __shared__ float q_s[kRows][D];
  __shared__ float k_s[kKeys][D + 1];
  __shared__ float v_s[kKeys][D];
  const int b = blockIdx.z;
  const int hq = blockIdx.y;
  const int i0 = blockIdx.x * kRows;
  const int qo = a.qo_indptr[b];
  const int S = a.qo_indptr[b + 1] - qo;
  const int P = a.prefix_len[b];
  if (i0 >= S) return;
  const int Hq = a.num_q_heads, Hkv = a.num_kv_heads, G = Hq / Hkv;
  const int hk = hq / G;
  const int row = a.req_idx[b];
  if (P < 0 || (int64_t)P + S > a.max_ctx || row < 0 || row >= a.max_reqs || qo < 0 ||
      (int64_t)qo + S > a.num_tokens) {
    if (threadIdx.x == 0) set_status(status, kStatusPosRange);
    return;
  }
  const int32_t* rt = a.req_to_token + (int64_t)row * a.max_ctx;
  const T* q = (const T*)a.q;
  const T* kn = (const T*)a.k_new;
  const T* vn = (const T*)a.v_new;
  const T* kp = (const T*)a.k_pool;
  const T* vp = (const T*)a.v_pool;
  const float qscale = a.sm_scale * kLog2e;
  const int nrows = min(kRows, S - i0);

  for (int e = threadIdx.x; e < kRows * D; e += blockDim.x) {
    const int r = e / D, d = e - r * D;
    q_s[r][d] = r < nrows ? Elem<T>::to_f(q[((int64_t)(qo + i0 + r) * Hq + hq) * D + d]) * qscale : 0.f;
  }
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  constexpr int DPL = D / 32;
  float m[4], l[4], acc[4][DPL];
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    m[r] = -INFINITY;
    l[r] = 0.f;
#pragma unroll
    for (int k = 0; k < DPL; ++k) acc[r][k] = 0.f;
  }
  const int kend = P + i0 + nrows;  // keys [0, kend) are visible to some row of this tile
  for (int j0 = 0; j0 < kend; j0 += kKeys) {
    __syncthreads();
    for (int e = threadIdx.x; e < kKeys * D; e += blockDim.x) {
      const int r = e / D, d = e - r * D;
      const int j = j0 + r;
      float kv = 0.f, vv = 0.f;
      if (j < P) {
        const int sl = rt[j];
        if (sl >= 0 && (int64_t)sl < a.num_slots) {
          kv = Elem<T>::to_f(kp[((int64_t)sl * Hkv + hk) * D + d]);
          vv = Elem<T>::to_f(vp[((int64_t)sl * Hkv + hk) * D + d]);
        } else if (d == 0) {
          set_status(status, kStatusSlotRange);
        }
      } else if (j < kend) {
        const int64_t t = qo + (j - P);
        kv = Elem<T>::to_f(kn[(t * Hkv + hk) * D + d]);
        vv = Elem<T>::to_f(vn[(t * Hkv + hk) * D + d]);
      }
      k_s[r][d] = kv;
      v_s[r][d] = vv;
    }
    __syncthreads();
#pragma unroll
    for (int rr = 0; rr < 4; ++rr) {
      const int r = wid * 4 + rr;
      if (r >= nrows) break;
      const int qpos = P + i0 + r;  // absolute position of this query
      const int j = j0 + lane;
      float s = 0.f;
#pragma unroll 8
      for (int d = 0; d < D; ++d) s = fmaf(q_s[r][d], k_s[lane][d], s);
      if (j > qpos) s = -INFINITY;
      float mx = s;
#pragma unroll
      for (int o = 16; o; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
      const float mn = fmaxf(m[rr], mx);
      const float alpha = mn == -INFINITY ? 1.f : exp2f(m[rr] - mn);
      const float pr = s == -INFINITY ? 0.f : exp2f(s - mn);
      float ps = pr;
#pragma unroll
      for (int o = 16; o; o >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, o);
      l[rr] = l[rr] * alpha + ps;
      m[rr] = mn;
#pragma unroll
      for (int k = 0; k < DPL; ++k) acc[rr][k] *= alpha;
      for (int jj = 0; jj < kKeys; ++jj) {
        const float pj = __shfl_sync(0xffffffffu, pr, jj);
#pragma unroll
        for (int k = 0; k < DPL; ++k) acc[rr][k] = fmaf(pj, v_s[jj][lane + 32 * k], acc[rr][k]);
      }
    }
  }
  T* o = (T*)a.o;
#pragma unroll
  for (int rr = 0; rr < 4; ++rr) {
    const int r = wid * 4 + rr;
    if (r >= nrows) break;
    const int64_t t = qo + i0 + r;
    const float inv = 1.f / l[rr];
#pragma unroll
    for (int k = 0; k < DPL; ++k) o[(t * Hq + hq) * D + lane + 32 * k] = Elem<T>::from_f(acc[rr][k] * inv);
    if (a.lse && lane == 0) a.lse[t * Hq + hq] = (m[rr] + log2f(l[rr])) * kLn2;
  }
  // the first query head of each KV group scatters the new K/V rows of its query rows
  if (hq % G == 0) {
    for (int e = threadIdx.x; e < nrows * D; e += blockDim.x) {
      const int r = e / D, d = e - r * D;
      const int64_t t = qo + i0 + r;
      const int sl = a.out_loc[t];
      if (sl < 0 || (int64_t)sl >= a.num_slots) {
        if (d == 0) set_status(status, kStatusSlotRange);
        continue;
      }
      ((T*)a.k_pool)[((int64_t)sl * Hkv + hk) * D + d] = kn[(t * Hkv + hk) * D + d];
      ((T*)a.v_pool)[((int64_t)sl * Hkv + hk) * D + d] = vn[(t * Hkv + hk) * D + d];
    }
  }
}

}  // namespace

int launch_extend_simt(const rc_extend_args* a, int* status, cudaStream_t s) {
  dim3 grid((a->max_q_len + kRows - 1) / kRows, a->num_q_heads, a->num_reqs);
  if (a->dtype == RC_DTYPE_F32) {
    if (a->head_dim == 128)
      extend_simt_kernel<float, 128><<<grid, 128, 0, s>>>(*a, status);
    else
      extend_simt_kernel<float, 64><<<grid, 128, 0, s>>>(*a, status);
  } else {
    if (a->head_dim == 128)
      extend_simt_kernel<__nv_bfloat16, 128><<<grid, 128, 0, s>>>(*a, status);
    else
      extend_simt_kernel<__nv_bfloat16, 64><<<grid, 128, 0, s>>>(*a, status);
  }
  count_launches(1);
  return check_launch("rc_extend_attention (simt)");
}

}  // namespace rc
