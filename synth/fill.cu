// Device-side copy of the synthetic value generator (see synth/__init__.py for the definition):
// writes the values of token rows keyed by prefix hashes, either densely [n, H, D] or into the
// rows of a KV pool plane [num_slots, H, D] given a slot per row. Input generation only.
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

namespace {

__device__ __forceinline__ uint64_t mix64(uint64_t x) {
  uint64_t z = x + 0x9E3779B97F4A7C15ull;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

__device__ __forceinline__ float value_of(uint64_t base, int e, float scale) {
  const uint64_t u = mix64(base + (uint64_t)e);
  const int64_t s = (int64_t)(u & 0xFFFF) + (int64_t)((u >> 16) & 0xFFFF) +
                    (int64_t)((u >> 32) & 0xFFFF) + (int64_t)(u >> 48) - 131070;
  return __fmul_rn((float)s, scale);
}

// one thread = 8 consecutive elements of one (row, head)
template <bool BF16>
__global__ void fill_kernel(const uint64_t* __restrict__ hashes, const int32_t* __restrict__ slots,
                            int64_t n, int tensor, int layer, int head0, int H, int D, float scale,
                            void* dst) {
  const int per_row = H * (D / 8);
  const int64_t nthreads = n * per_row;
  for (int64_t t = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; t < nthreads;
       t += (int64_t)gridDim.x * blockDim.x) {
    const int64_t i = t / per_row;
    const int rem = (int)(t - i * per_row);
    const int h = rem / (D / 8);
    const int e0 = (rem - h * (D / 8)) * 8;
    const uint64_t key = mix64(((uint64_t)tensor << 48) | ((uint64_t)layer << 24) |
                               (uint64_t)(head0 + h));
    const uint64_t base = mix64(hashes[i] ^ key);
    const int64_t row = slots ? (int64_t)slots[i] : i;
    const int64_t off = (row * H + h) * D + e0;
    if (BF16) {
      __nv_bfloat16* o = (__nv_bfloat16*)dst + off;
      __align__(16) __nv_bfloat16 v[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) v[k] = __float2bfloat16_rn(value_of(base, e0 + k, scale));
      *(uint4*)o = *(const uint4*)v;
    } else {
      float* o = (float*)dst + off;
#pragma unroll
      for (int k = 0; k < 8; ++k) o[k] = value_of(base, e0 + k, scale);
    }
  }
}

}  // namespace

extern "C" int synth_fill_rows(const uint64_t* hashes, const int32_t* slots, int64_t n, int tensor,
                               int layer, int head0, int H, int D, int bf16, float scale,
                               void* dst, void* stream) {
  if (n <= 0) return 0;
  if (D % 8) return -1;
  const int threads = 256;
  const int64_t work = n * H * (D / 8);
  const int64_t blocks64 = (work + threads - 1) / threads;
  const int blocks = (int)(blocks64 < 152 * 64 ? blocks64 : 152 * 64);
  if (bf16)
    fill_kernel<true><<<blocks, threads, 0, (cudaStream_t)stream>>>(hashes, slots, n, tensor, layer,
                                                                     head0, H, D, scale, dst);
  else
    fill_kernel<false><<<blocks, threads, 0, (cudaStream_t)stream>>>(hashes, slots, n, tensor, layer,
                                                                      head0, H, D, scale, dst);
  return cudaGetLastError() == cudaSuccess ? 0 : -2;
}
