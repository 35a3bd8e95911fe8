// Decode attention over the paged KV pool with split-K (RadixAttention explainer: every new
// token attends to the KV of all previous tokens; paper digest App. A.1 decoding).
//
// Design (HBM-bound: every context token's K and V row is read once per KV head):
//   * plan kernel (1 CTA): cuts each request's context into chunks of kv_chunk tokens, gives
//     every (request, chunk) a partial-state slot and writes the job list; the chunks of a
//     shared-context group that lie wholly inside its shared prefix are listed once, as the
//     leader's stacked jobs (see rc_decode_args);
//   * main kernel (persistent, #SMs x occupancy CTAs of 4 warps): every warp is an independent
//     worker that takes (job, KV head) items from an atomic counter. For an item it streams the
//     chunk's K and V rows (one contiguous row of head_dim elements per token) from the pool into
//     a private 2-stage shared-memory ring of 16-token stages, the slot indices prefetched one
//     stage ahead. bf16 (decode_mma_kernel): 16-byte cp.async from all lanes, mma.sync m16n8k16
//     with the tokens as M and the query columns (G heads, or G heads of each stacked group
//     member) as N. fp32 (decode_main_kernel): cp.async.bulk rows, scores by lanes (token, half
//     of head_dim) with a one-step shuffle, P.V with each lane owning head_dim/32 output
//     columns of every query head. Online softmax in base 2 (scale * log2 e folded in). The new
//     token's K/V come from k_new/v_new (and are scattered to the pool by the last chunk's
//     item), so no read races the scatter;
//   * a request with one chunk writes its output directly; otherwise each chunk writes
//     (O normalised, log2-sum-exp) to its slot in the workspace and the merge kernel combines
//     them.
#include <algorithm>
#include <mutex>
#include <type_traits>

#include "device_common.cuh"
#include "host_common.h"

namespace rc {
namespace {

constexpr int kTok = 16;     // tokens per stage
constexpr int kStages = 2;   // ring depth per warp (two: 3 CTAs of 4 warps fit an SM)
constexpr int kWarps = 4;    // warps per CTA
constexpr int kDefaultChunk = 512;

struct Workspace {
  int* njobs;     // [0]: jobs written, [1]: item counter, [2]: warps finished (bf16 kernel)
  int* pbase;     // [B+1]: request b's partial states are slots pbase[b] + chunk
  int* group_of;  // [B]: shared-context group of each request, -1 for none
  int4* jobs;     // [max_jobs] (request, chunk, group of a stacked chunk or -1, 0)
  float* plse;    // [max_jobs * Hkv * G]
  float* po;      // [max_jobs * Hkv * G * D]
  int64_t max_jobs;
};

inline size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

Workspace carve(void* base, int B, int G, int D, int64_t max_jobs, int Hkv, size_t* total) {
  Workspace w{};
  char* p = (char*)base;
  size_t off = 0;
  w.njobs = (int*)(p + off);
  off += align256(3 * sizeof(int));
  w.pbase = (int*)(p + off);
  off += align256((size_t)(B + 1) * sizeof(int));
  w.group_of = (int*)(p + off);
  off += align256((size_t)B * sizeof(int));
  w.jobs = (int4*)(p + off);
  off += align256((size_t)max_jobs * sizeof(int4));
  const int64_t max_items = max_jobs * Hkv;
  w.plse = (float*)(p + off);
  off += align256((size_t)max_items * G * sizeof(float));
  w.po = (float*)(p + off);
  off += align256((size_t)max_items * G * D * sizeof(float));
  w.max_jobs = max_jobs;
  if (total) *total = off;
  return w;
}

struct Params {
  rc_decode_args a;
  Workspace w;
  int chunk;
  int use_groups;    // stack the shared chunks of the argument's groups (bf16)
  int max_members;   // 8 / G: query columns of one MMA tile
  int* status;
};

// ---------------------------------------------------------------- plan
// Exclusive scan of one int per thread over the block; returns this thread's prefix and adds the
// block total to *running (all threads see the same value afterwards).
__device__ int block_excl_scan(int x, int* warp_sums, int* running) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
  int v = x;
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += y;
  }
  if (lane == 31) warp_sums[wid] = v;
  __syncthreads();
  if (wid == 0) {
    int t = lane < nw ? warp_sums[lane] : 0;
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, t, o);
      if (lane >= o) t += y;
    }
    warp_sums[lane] = t;  // inclusive
  }
  __syncthreads();
  const int excl = *running + (wid ? warp_sums[wid - 1] : 0) + v - x;
  __syncthreads();
  if (threadIdx.x == 0) *running += warp_sums[nw - 1];
  __syncthreads();
  return excl;
}

// One CTA. Every request gets ceil(L / chunk) partial-state slots (pbase); the job list holds
// its chunks, except that a group's chunks wholly inside the shared context appear once, as the
// leader's stacked jobs.
__global__ void decode_plan_kernel(Params p) {
  __shared__ int warp_sums[32];
  __shared__ int run_p, run_j;
  const int tid = threadIdx.x;
  const int B = p.a.num_reqs;
  if (tid == 0) run_p = run_j = 0;
  for (int b = tid; b < B; b += blockDim.x) p.w.group_of[b] = -1;
  __syncthreads();
  if (p.use_groups) {
    for (int g = tid; g < p.a.num_groups; g += blockDim.x) {
      const int m0 = p.a.group_indptr[g], m1 = p.a.group_indptr[g + 1];
      if (m0 < 0 || m1 < m0 || m1 - m0 > p.max_members) {
        set_status(p.status, kStatusPosRange);
        continue;
      }
      for (int i = m0; i < m1; ++i) {
        const int b = p.a.group_members[i];
        if (b < 0 || b >= B || atomicCAS(&p.w.group_of[b], -1, g) != -1)
          set_status(p.status, kStatusPosRange);   // out of range, or in two groups
      }
    }
  }
  __syncthreads();
  for (int base = 0; base < B; base += blockDim.x) {
    const int b = base + tid;
    int n = 0, first = 0, nj = 0, g = -1, sc = 0;
    if (b < B) {
      const int L = p.a.seq_len[b];
      const int row = p.a.req_idx[b];
      if (L < 1 || L > p.a.max_ctx || row < 0 || row >= p.a.max_reqs) {
        set_status(p.status, kStatusPosRange);
      } else {
        n = (L + p.chunk - 1) / p.chunk;
        g = p.w.group_of[b];
        if (g >= 0) {
          const int sh = p.a.group_shared[g];
          if (sh < 0 || sh > L - 1) set_status(p.status, kStatusPosRange);
          sc = min(max(sh, 0), L - 1) / p.chunk;   // stacked chunks: wholly inside [0, sh)
          // the leader runs the stacked chunks for the whole group, the others skip them
          if (p.a.group_members[p.a.group_indptr[g]] != b) first = sc;
        }
        nj = n - first;
      }
    }
    const int pb = block_excl_scan(n, warp_sums, &run_p);
    const int jb = block_excl_scan(nj, warp_sums, &run_j);
    if (b < B) {
      p.w.pbase[b] = pb;
      for (int k = 0; k < nj; ++k) {
        const int c = first + k;
        if (jb + k < p.w.max_jobs && pb + n <= p.w.max_jobs)
          p.w.jobs[jb + k] = make_int4(b, c, (g >= 0 && c < sc) ? g : -1, 0);
        else
          set_status(p.status, kStatusPosRange);
      }
    }
  }
  if (tid == 0) {
    p.w.pbase[B] = run_p;
    p.w.njobs[0] = (int)min((int64_t)run_j, p.w.max_jobs);
    p.w.njobs[1] = 0;
    p.w.njobs[2] = 0;
  }
}

// ---------------------------------------------------------------- main
template <typename T, int D, int G>
struct Cfg {
  static constexpr int RB = D * (int)sizeof(T);  // bytes of one K or V row
  static constexpr int RK = RB + 16;             // padded K row stride in shared memory
  static constexpr int STAGE = kTok * (RK + RB);
  static constexpr int RING = kStages * STAGE;
  static constexpr int QS = G * D * 4;           // fp32 q of the warp's item
  static constexpr int PS = kTok * G * 4;        // probabilities of one stage
  static constexpr int BAR = kStages * 8;
  static constexpr int WARP_BYTES = (RING + QS + PS + BAR + 127) / 128 * 128;
  static constexpr int SMEM = kWarps * WARP_BYTES;
  static constexpr int DPL = D / 32;             // output columns per lane
  static_assert(RB % 16 == 0, "rows must be multiples of 16 bytes");
  static_assert(STAGE % 16 == 0 && QS % 16 == 0 && PS % 16 == 0, "alignment");
};

template <typename T>
__device__ __forceinline__ void load_cols(const char* p, float* v, int n);
template <>
__device__ __forceinline__ void load_cols<__nv_bfloat16>(const char* p, float* v, int n) {
  if (n == 4) {
    const uint2 w = *(const uint2*)p;
    v[0] = bf16lo(w.x); v[1] = bf16hi(w.x); v[2] = bf16lo(w.y); v[3] = bf16hi(w.y);
  } else {  // n == 2
    const uint32_t w = *(const uint32_t*)p;
    v[0] = bf16lo(w); v[1] = bf16hi(w);
  }
}
template <>
__device__ __forceinline__ void load_cols<float>(const char* p, float* v, int n) {
  if (n == 4) {
    const float4 w = *(const float4*)p;
    v[0] = w.x; v[1] = w.y; v[2] = w.z; v[3] = w.w;
  } else {
    const float2 w = *(const float2*)p;
    v[0] = w.x; v[1] = w.y;
  }
}

// 16 bytes of a row -> fp32 values (8 for bf16, 4 for fp32)
template <typename T>
struct Chunk16;
template <>
struct Chunk16<__nv_bfloat16> {
  static constexpr int N = 8;
  static __device__ __forceinline__ void get(const char* p, float* k) {
    const uint4 w = *(const uint4*)p;
    k[0] = bf16lo(w.x); k[1] = bf16hi(w.x); k[2] = bf16lo(w.y); k[3] = bf16hi(w.y);
    k[4] = bf16lo(w.z); k[5] = bf16hi(w.z); k[6] = bf16lo(w.w); k[7] = bf16hi(w.w);
  }
};
template <>
struct Chunk16<float> {
  static constexpr int N = 4;
  static __device__ __forceinline__ void get(const char* p, float* k) {
    const float4 w = *(const float4*)p;
    k[0] = w.x; k[1] = w.y; k[2] = w.z; k[3] = w.w;
  }
};

template <typename T, int D, int G>
__global__ void __launch_bounds__(kWarps * 32) decode_main_kernel(Params p) {
  using C = Cfg<T, D, G>;
  extern __shared__ __align__(128) char smem[];
  const int lane = threadIdx.x & 31;
  const int wid = threadIdx.x >> 5;
  char* wbase = smem + wid * C::WARP_BYTES;
  char* ring = wbase;
  float* q_s = (float*)(wbase + C::RING);
  float* p_s = (float*)(wbase + C::RING + C::QS);
  uint64_t* bars = (uint64_t*)(wbase + C::RING + C::QS + C::PS);
  if (lane == 0) {
    for (int s = 0; s < kStages; ++s) mbar_init(&bars[s], 1);
    fence_mbar_init();
  }
  __syncwarp();

  const rc_decode_args& a = p.a;
  const int Hq = a.num_q_heads, Hkv = a.num_kv_heads;
  const int n_items = p.w.njobs[0] * Hkv;
  const float qscale = a.sm_scale * kLog2e;
  const T* kpool = (const T*)a.k_pool;
  const T* vpool = (const T*)a.v_pool;
  uint32_t phases = 0;  // bit s = parity to wait for on stage buffer s
  const int t = lane & 15, half = lane >> 4;

  while (true) {
    int item = 0;
    if (lane == 0) item = atomicAdd(&p.w.njobs[1], 1);
    item = __shfl_sync(0xffffffffu, item, 0);
    if (item >= n_items) break;
    const int job = item / Hkv, h = item - job * Hkv;
    const int4 bc = p.w.jobs[job];
    const int b = bc.x, c = bc.y;
    const int64_t pslot = (int64_t)p.w.pbase[b] + c;   // partial-state slot of (b, c)
    const int L = a.seq_len[b];
    const int row = a.req_idx[b];
    const int t0 = c * p.chunk;
    const int t1 = min(L, t0 + p.chunk);
    const int nchunks = (L + p.chunk - 1) / p.chunk;
    const int nst = (t1 - t0 + kTok - 1) / kTok;
    const int32_t* rt = a.req_to_token + (int64_t)row * a.max_ctx;
    const T* knew = (const T*)a.k_new + ((int64_t)b * Hkv + h) * D;
    const T* vnew = (const T*)a.v_new + ((int64_t)b * Hkv + h) * D;

    // q of the G query heads of this KV head, pre-scaled to base-2 logits
    {
      const T* qg = (const T*)a.q + ((int64_t)b * Hq + (int64_t)h * G) * D;
      for (int e = lane; e < G * D; e += 32) q_s[e] = Elem<T>::to_f(qg[e]) * qscale;
    }

    // slot of the token this lane loads in stage s (-1: past the chunk; -2: the new token)
    auto slot_of = [&](int s) -> int {
      const int pos = t0 + s * kTok + lane;
      if (lane >= kTok || pos >= t1) return -1;
      if (pos == L - 1) return -2;
      const int sl = rt[pos];
      if (sl < 0 || (int64_t)sl >= a.num_slots) {
        set_status(p.status, kStatusSlotRange);
        return -3;
      }
      return sl;
    };
    // issue stage s (slot already resolved); returns the mask of real tokens
    auto issue = [&](int s, int sl) {
      const int buf = s % kStages;
      char* kd = ring + buf * C::STAGE + lane * C::RK;
      char* vd = ring + buf * C::STAGE + kTok * C::RK + lane * C::RB;
      const bool live = sl != -1;
      const uint32_t nlive = __popc(__ballot_sync(0xffffffffu, live));
      if (lane == 0) mbar_arrive_expect_tx(&bars[buf], nlive * 2u * C::RB);
      if (live) {
        const T* ks;
        const T* vs;
        if (sl == -2) {
          ks = knew;
          vs = vnew;
        } else {
          const int64_t r = ((int64_t)(sl < 0 ? 0 : sl) * Hkv + h) * D;  // bad slot: read row 0
          ks = kpool + r;
          vs = vpool + r;
        }
        bulk_g2s(kd, ks, C::RB, &bars[buf]);
        bulk_g2s(vd, vs, C::RB, &bars[buf]);
      }
    };

    int next_slot = slot_of(0);
    const int pro = min(nst, kStages - 1);
    for (int s = 0; s < pro; ++s) {
      issue(s, next_slot);
      next_slot = slot_of(s + 1);
    }
    __syncwarp();  // q_s visible to all lanes

    float m[G], lsum[G], acc[G][C::DPL];
#pragma unroll
    for (int g = 0; g < G; ++g) {
      m[g] = -INFINITY;
      lsum[g] = 0.f;
#pragma unroll
      for (int k = 0; k < C::DPL; ++k) acc[g][k] = 0.f;
    }

    bool ok = true;
    for (int s = 0; s < nst; ++s) {
      if (s + kStages - 1 < nst) {
        issue(s + kStages - 1, next_slot);
        next_slot = slot_of(s + kStages);
      }
      const int buf = s % kStages;
      if (!mbar_wait(&bars[buf], (phases >> buf) & 1u, p.status)) {
        ok = false;
        break;
      }
      phases ^= 1u << buf;
      const int base_pos = t0 + s * kTok;
      const int ntok = min(kTok, t1 - base_pos);
      const int my_slot_ok = (base_pos + t < t1);
      // ---- scores: lane (t, half) covers head_dim/2 columns of token t
      float sc[G];
#pragma unroll
      for (int g = 0; g < G; ++g) sc[g] = 0.f;
      {
        const char* krow = ring + buf * C::STAGE + t * C::RK + half * (C::RB / 2);
        const int d0 = half * (D / 2);
#pragma unroll
        for (int cc = 0; cc < C::RB / 2 / 16; ++cc) {
          float k[Chunk16<T>::N];
          Chunk16<T>::get(krow + cc * 16, k);
          const int dd = d0 + cc * Chunk16<T>::N;
#pragma unroll
          for (int g = 0; g < G; ++g) {
#pragma unroll
            for (int e = 0; e < Chunk16<T>::N; e += 4) {
              const float4 qv = *(const float4*)&q_s[g * D + dd + e];
              sc[g] = fmaf(qv.x, k[e], sc[g]);
              sc[g] = fmaf(qv.y, k[e + 1], sc[g]);
              sc[g] = fmaf(qv.z, k[e + 2], sc[g]);
              sc[g] = fmaf(qv.w, k[e + 3], sc[g]);
            }
          }
        }
      }
      float alpha[G];
#pragma unroll
      for (int g = 0; g < G; ++g) {
        sc[g] += __shfl_xor_sync(0xffffffffu, sc[g], 16);
        if (!my_slot_ok) sc[g] = -INFINITY;
        float mx = sc[g];
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
        const float mn = fmaxf(m[g], mx);
        alpha[g] = (mn == -INFINITY) ? 1.f : exp2f(m[g] - mn);
        const float pr = (sc[g] == -INFINITY) ? 0.f : exp2f(sc[g] - mn);
        lsum[g] = lsum[g] * alpha[g] + (half == 0 ? pr : 0.f);
        m[g] = mn;
        if (half == 0) p_s[t * G + g] = pr;
      }
      __syncwarp();
      // ---- P.V: lane owns columns [lane*DPL, lane*DPL + DPL)
#pragma unroll
      for (int g = 0; g < G; ++g)
#pragma unroll
        for (int k = 0; k < C::DPL; ++k) acc[g][k] *= alpha[g];
      const char* vb = ring + buf * C::STAGE + kTok * C::RK + lane * C::DPL * (int)sizeof(T);
      for (int tt = 0; tt < ntok; ++tt) {
        float v[C::DPL];
        load_cols<T>(vb + tt * C::RB, v, C::DPL);
#pragma unroll
        for (int g = 0; g < G; ++g) {
          const float pr = p_s[tt * G + g];
#pragma unroll
          for (int k = 0; k < C::DPL; ++k) acc[g][k] = fmaf(pr, v[k], acc[g][k]);
        }
      }
      __syncwarp();
    }
    if (!ok) {
      // a copy never landed: wait (bounded) for this warp's other copies, then stop
      for (int s = 0; s < kStages; ++s) mbar_wait(&bars[s], (phases >> s) & 1u, p.status, 100000000ull);
      return;
    }

    // ---- epilogue
#pragma unroll
    for (int g = 0; g < G; ++g) {
      float l = lsum[g];
      l += __shfl_xor_sync(0xffffffffu, l, 1);
      l += __shfl_xor_sync(0xffffffffu, l, 2);
      l += __shfl_xor_sync(0xffffffffu, l, 4);
      l += __shfl_xor_sync(0xffffffffu, l, 8);
      l += __shfl_xor_sync(0xffffffffu, l, 16);
      const float inv = l > 0.f ? 1.f / l : 0.f;
      const float lse2 = l > 0.f ? m[g] + log2f(l) : -INFINITY;
      const int hq = h * G + g;
      if (nchunks == 1) {
        T* o = (T*)a.o + ((int64_t)b * Hq + hq) * D + lane * C::DPL;
#pragma unroll
        for (int k = 0; k < C::DPL; ++k) o[k] = Elem<T>::from_f(acc[g][k] * inv);
        if (a.lse && lane == 0) a.lse[(int64_t)b * Hq + hq] = lse2 * kLn2;
      } else {
        const int64_t pi = (pslot * Hkv + h) * G + g;
        float* po = p.w.po + pi * D + lane * C::DPL;
#pragma unroll
        for (int k = 0; k < C::DPL; ++k) po[k] = acc[g][k] * inv;
        if (lane == 0) p.w.plse[pi] = lse2;
      }
    }
    // ---- the last chunk scatters the new token's K and V rows into the pool
    if (c == nchunks - 1) {
      const int sl = a.out_loc[b];
      if (sl < 0 || (int64_t)sl >= a.num_slots) {
        if (lane == 0) set_status(p.status, kStatusSlotRange);
      } else {
        const int64_t r = ((int64_t)sl * Hkv + h) * D;
        for (int e = lane; e < C::RB / 16; e += 32) {
          ((uint4*)((T*)a.k_pool + r))[e] = ((const uint4*)knew)[e];
          ((uint4*)((T*)a.v_pool + r))[e] = ((const uint4*)vnew)[e];
        }
      }
    }
    __syncwarp();
  }
}

// ---------------------------------------------------------------- main, bf16 (warp-level MMA)
// Same work split and ring as the CUDA-core kernel, but the two contractions of a stage run on
// mma.sync m16n8k16 (bf16 in, fp32 accumulate), which cuts the instruction count per KV row by
// an order of magnitude so that the kernel stays bound by HBM, not by issue:
//   S^T [16 tokens x 8] = K [16 tokens x d] . Q^T [d x 8]       (the G <= 8 query heads as N)
//   O^T [d x 8]        += V^T [d x 16 tokens] . P^T [16 x 8]
// K fragments by ldmatrix, V^T by ldmatrix.trans (both from 272-byte padded rows: conflict-free),
// Q^T fragments held in registers for the whole item, P^T from the S^T accumulator by
// movmatrix.trans. P is split into a bf16 high part and a bf16 remainder (two MMAs), so P.V
// keeps ~16 bits of the fp32 probabilities.
template <int D>
struct MmaCfg {
  static constexpr int RB = D * 2;               // bytes of one bf16 K or V row
  static constexpr int RS = RB + 16;             // padded row stride in shared memory
  static constexpr int STAGE = kTok * 2 * RS;    // K rows then V rows
  static constexpr int RING = kStages * STAGE;
  static constexpr int WARP_BYTES = (RING + kStages * 8 + 127) / 128 * 128;
  static constexpr int SMEM = kWarps * WARP_BYTES;
  static constexpr int KSTEPS = D / 16;
  static_assert(kTok == 16, "one m16 tile of tokens per stage");
};

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_arrive_noinc(uint32_t bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                          uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void mma16816(float* c, uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t movm_t(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}
__device__ __forceinline__ uint32_t bf2(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *(const uint32_t*)&v;
}

// A warp leaves the persistent loop: the last one of the grid resets the item counter, so a
// later call that reuses the plan hands out the items again.
__device__ __forceinline__ void retire_warp(const Params& p, int lane) {
  __syncwarp();
  if (lane == 0) {
    __threadfence();
    if (atomicAdd(&p.w.njobs[2], 1) == (int)gridDim.x * kWarps - 1) {
      p.w.njobs[1] = 0;
      p.w.njobs[2] = 0;
    }
  }
}

template <int D, int G>
__global__ void __launch_bounds__(kWarps * 32) decode_mma_kernel(Params p) {
  using C = MmaCfg<D>;
  extern __shared__ __align__(128) char smem[];
  const int lane = threadIdx.x & 31;
  const int wid = threadIdx.x >> 5;
  const int gid = lane >> 2, tig = lane & 3;
  char* ring = smem + wid * C::WARP_BYTES;
  uint64_t* bars = (uint64_t*)(ring + C::RING);
  if (lane == 0) {
    for (int s = 0; s < kStages; ++s) mbar_init(&bars[s], 32);   // one copy-arrival per lane
    fence_mbar_init();
  }
  __syncwarp();
  const uint32_t ring_s = smem_u32(ring);

  const rc_decode_args& a = p.a;
  const int Hq = a.num_q_heads, Hkv = a.num_kv_heads;
  const int n_items = p.w.njobs[0] * Hkv;
  const float qscale = a.sm_scale * kLog2e;
  const __nv_bfloat16* kpool = (const __nv_bfloat16*)a.k_pool;
  const __nv_bfloat16* vpool = (const __nv_bfloat16*)a.v_pool;
  uint32_t phases = 0;
  // ldmatrix row addresses (per lane, relative to a stage): K as the A operand (token rows),
  // V^T through the transposing load (token rows, d halves)
  const int k_row = (lane & 7) + ((lane >> 3) & 1) * 8, k_col = (lane >> 4) * 8;
  const int v_row = (lane & 7) + (lane >> 4) * 8, v_col = ((lane >> 3) & 1) * 8;

  while (true) {
    int item = 0;
    if (lane == 0) item = atomicAdd(&p.w.njobs[1], 1);
    item = __shfl_sync(0xffffffffu, item, 0);
    if (item >= n_items) break;
    const int job = item / Hkv, h = item - job * Hkv;
    const int4 bc = p.w.jobs[job];
    const int b = bc.x, c = bc.y;
    const int64_t pslot = (int64_t)p.w.pbase[b] + c;   // partial-state slot of (b, c)
    // a stacked chunk of a shared-context group: the leader's rows serve every member; query
    // column n of the MMA tile is member n / G, head n % G
    const int grp = bc.z;
    int nm = 1;
    const int32_t* mem = nullptr;
    if (grp >= 0) {
      const int m0 = a.group_indptr[grp];
      nm = min(a.group_indptr[grp + 1] - m0, 8 / G);
      mem = a.group_members + m0;
    }
    const int ncols = grp >= 0 ? nm * G : G;
    const int L = a.seq_len[b];
    const int row = a.req_idx[b];
    const int t0 = c * p.chunk;
    const int t1 = min(L, t0 + p.chunk);
    const int nchunks = (L + p.chunk - 1) / p.chunk;
    const int nst = (t1 - t0 + kTok - 1) / kTok;
    const int32_t* rt = a.req_to_token + (int64_t)row * a.max_ctx;
    const __nv_bfloat16* knew = (const __nv_bfloat16*)a.k_new + ((int64_t)b * Hkv + h) * D;
    const __nv_bfloat16* vnew = (const __nv_bfloat16*)a.v_new + ((int64_t)b * Hkv + h) * D;

    // slot of the token lane `lane` (< 16) copies in stage s: -2 = the new token (also used to
    // fill the rows past the chunk end, so every shared row holds finite values). The load is
    // only issued here; issue() checks the value, so it stays in flight for a stage.
    auto slot_of = [&](int s) -> int {
      const int pos = t0 + s * kTok + lane;
      if (lane >= kTok) return -1;
      if (pos >= t1 || pos == L - 1) return -2;
      return rt[pos];
    };
    // Stage s: the warp copies the 16 tokens' K and V rows with 16-byte cp.async (lane l moves
    // chunk l % CPR of rows l / CPR, l / CPR + RPI, ...), each row pointer taken by a shuffle
    // from the lane that loaded that token's slot; completion is one arrival per lane.
    auto issue = [&](int s, int sl) {
      if (sl >= 0 && (int64_t)sl >= a.num_slots) {
        set_status(p.status, kStatusSlotRange);
        sl = 0;
      } else if (sl < -2) {
        set_status(p.status, kStatusSlotRange);
        sl = 0;
      }
      const int buf = s % kStages;
      const __nv_bfloat16* ks = knew;
      const __nv_bfloat16* vs = vnew;
      if (sl >= 0) {
        const int64_t r = ((int64_t)sl * Hkv + h) * D;
        ks = kpool + r;
        vs = vpool + r;
      }
      constexpr int CPR = C::RB / 16;   // 16-byte chunks per row
      constexpr int RPI = 32 / CPR;     // rows per copy instruction
      const int cc = lane % CPR, rsub = lane / CPR;
      const uint32_t kd = ring_s + buf * C::STAGE + cc * 16;
      const uint32_t vd = kd + kTok * C::RS;
#pragma unroll
      for (int i = 0; i < kTok / RPI; ++i) {
        const int t = i * RPI + rsub;
        const char* kp = (const char*)__shfl_sync(0xffffffffu, (uint64_t)ks, t);
        const char* vp = (const char*)__shfl_sync(0xffffffffu, (uint64_t)vs, t);
        cp_async16(kd + t * C::RS, kp + cc * 16);
        cp_async16(vd + t * C::RS, vp + cc * 16);
      }
      cp_async_arrive_noinc(smem_u32(&bars[buf]));
    };

    int next_slot = slot_of(0);
    const int pro = min(nst, kStages - 1);
    for (int s = 0; s < pro; ++s) {
      issue(s, next_slot);
      next_slot = slot_of(s + 1);
    }
    // Q^T fragments: column n = gid is query head h*G + gid of request b (zero for gid >= G),
    // or, for a stacked chunk, head h*G + gid % G of member gid / G
    uint32_t qb[C::KSTEPS][2];
    {
      int qb_req = b, qh = gid;
      bool qv = gid < ncols;
      if (grp >= 0 && qv) {
        qb_req = mem[gid / G];
        qh = gid % G;
        qv = qb_req >= 0 && qb_req < a.num_reqs;
      }
      const __nv_bfloat16* qg =
          (const __nv_bfloat16*)a.q + ((int64_t)(qv ? qb_req : 0) * Hq + h * G + (qv ? qh : 0)) * D;
#pragma unroll
      for (int kk = 0; kk < C::KSTEPS; ++kk) {
        qb[kk][0] = qv ? *(const uint32_t*)(qg + kk * 16 + tig * 2) : 0u;
        qb[kk][1] = qv ? *(const uint32_t*)(qg + kk * 16 + tig * 2 + 8) : 0u;
      }
    }
    float acc[C::KSTEPS][4];
#pragma unroll
    for (int i = 0; i < C::KSTEPS; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;  // heads 2*tig, 2*tig + 1

    bool ok = true;
    for (int s = 0; s < nst; ++s) {
      if (s + kStages - 1 < nst) {
        issue(s + kStages - 1, next_slot);
        next_slot = slot_of(s + kStages);
      }
      const int buf = s % kStages;
      if (!mbar_wait(&bars[buf], (phases >> buf) & 1u, p.status)) {
        ok = false;
        break;
      }
      phases ^= 1u << buf;
      const uint32_t kb = ring_s + buf * C::STAGE;
      const uint32_t vb = kb + kTok * C::RS;
      // ---- S^T = K Q^T
      float sc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int kk = 0; kk < C::KSTEPS; ++kk) {
        uint32_t a0, a1, a2, a3;
        ldsm_x4(kb + k_row * C::RS + (kk * 16 + k_col) * 2, a0, a1, a2, a3);
        mma16816(sc, a0, a1, a2, a3, qb[kk][0], qb[kk][1]);
      }
      const int base_pos = t0 + s * kTok;
      const bool v_lo = base_pos + gid < t1, v_hi = base_pos + gid + 8 < t1;
      sc[0] = v_lo ? sc[0] * qscale : -INFINITY;
      sc[1] = v_lo ? sc[1] * qscale : -INFINITY;
      sc[2] = v_hi ? sc[2] * qscale : -INFINITY;
      sc[3] = v_hi ? sc[3] * qscale : -INFINITY;
      float x0 = fmaxf(sc[0], sc[2]), x1 = fmaxf(sc[1], sc[3]);
#pragma unroll
      for (int o = 4; o < 32; o <<= 1) {
        x0 = fmaxf(x0, __shfl_xor_sync(0xffffffffu, x0, o));
        x1 = fmaxf(x1, __shfl_xor_sync(0xffffffffu, x1, o));
      }
      // lazy rescale: move the running max only when it grows by more than 2^8
      const float n0 = fmaxf(m0, x0), n1 = fmaxf(m1, x1);
      const bool r0 = n0 > m0 + 8.f, r1 = n1 > m1 + 8.f;
      const float u0 = r0 ? n0 : m0, u1 = r1 ? n1 : m1;
      const float al0 = (r0 && m0 != -INFINITY) ? exp2f(m0 - n0) : 1.f;
      const float al1 = (r1 && m1 != -INFINITY) ? exp2f(m1 - n1) : 1.f;
      m0 = u0;
      m1 = u1;
      const float p0 = exp2f(sc[0] - u0), p1 = exp2f(sc[1] - u1);
      const float p2 = exp2f(sc[2] - u0), p3 = exp2f(sc[3] - u1);
      l0 = l0 * al0 + p0 + p2;
      l1 = l1 * al1 + p1 + p3;
      if (__any_sync(0xffffffffu, al0 != 1.f || al1 != 1.f)) {
#pragma unroll
        for (int i = 0; i < C::KSTEPS; ++i) {
          acc[i][0] *= al0;
          acc[i][1] *= al1;
          acc[i][2] *= al0;
          acc[i][3] *= al1;
        }
      }
      // ---- P^T fragments (high and remainder parts)
      const uint32_t hx = bf2(p0, p1), hy = bf2(p2, p3);
      const uint32_t lx = bf2(p0 - bf16lo(hx), p1 - bf16hi(hx));
      const uint32_t ly = bf2(p2 - bf16lo(hy), p3 - bf16hi(hy));
      const uint32_t bh0 = movm_t(hx), bh1 = movm_t(hy), bl0 = movm_t(lx), bl1 = movm_t(ly);
      // ---- O^T += V^T P^T
#pragma unroll
      for (int i = 0; i < C::KSTEPS; ++i) {
        uint32_t a0, a1, a2, a3;
        ldsm_x4_t(vb + v_row * C::RS + (i * 16 + v_col) * 2, a0, a1, a2, a3);
        mma16816(acc[i], a0, a1, a2, a3, bh0, bh1);
        mma16816(acc[i], a0, a1, a2, a3, bl0, bl1);
      }
      __syncwarp();
    }
    if (!ok) {
      asm volatile("cp.async.wait_all;" ::: "memory");   // no copy lands after the exit
      retire_warp(p, lane);
      return;
    }
    // ---- epilogue: full denominators per head, then O^T columns -> output rows
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) {
      l0 += __shfl_xor_sync(0xffffffffu, l0, o);
      l1 += __shfl_xor_sync(0xffffffffu, l1, o);
    }
    const int hA = 2 * tig, hB = 2 * tig + 1;
    const float iA = l0 > 0.f ? 1.f / l0 : 0.f, iB = l1 > 0.f ? 1.f / l1 : 0.f;
    const float lseA = l0 > 0.f ? m0 + log2f(l0) : -INFINITY;
    const float lseB = l1 > 0.f ? m1 + log2f(l1) : -INFINITY;
    if (grp >= 0) {
      // stacked chunk: column n's partial state goes to member n / G's slot for this chunk
      int64_t piA = -1, piB = -1;
      auto pidx = [&](int col) -> int64_t {
        if (col >= ncols) return -1;
        const int bm = mem[col / G];
        if (bm < 0 || bm >= a.num_reqs) return -1;
        const int64_t ps = (int64_t)p.w.pbase[bm] + c;
        if (ps >= p.w.max_jobs) return -1;
        return (ps * Hkv + h) * G + col % G;
      };
      piA = pidx(hA);
      piB = pidx(hB);
#pragma unroll
      for (int i = 0; i < C::KSTEPS; ++i) {
        const int d0 = i * 16 + gid;
        if (piA >= 0) {
          p.w.po[piA * D + d0] = acc[i][0] * iA;
          p.w.po[piA * D + d0 + 8] = acc[i][2] * iA;
        }
        if (piB >= 0) {
          p.w.po[piB * D + d0] = acc[i][1] * iB;
          p.w.po[piB * D + d0 + 8] = acc[i][3] * iB;
        }
      }
      if (gid == 0) {
        if (piA >= 0) p.w.plse[piA] = lseA;
        if (piB >= 0) p.w.plse[piB] = lseB;
      }
    } else if (nchunks == 1) {
      __nv_bfloat16* o = (__nv_bfloat16*)a.o + ((int64_t)b * Hq + h * G) * D;
#pragma unroll
      for (int i = 0; i < C::KSTEPS; ++i) {
        const int d0 = i * 16 + gid;
        if (hA < G) {
          o[hA * D + d0] = __float2bfloat16_rn(acc[i][0] * iA);
          o[hA * D + d0 + 8] = __float2bfloat16_rn(acc[i][2] * iA);
        }
        if (hB < G) {
          o[hB * D + d0] = __float2bfloat16_rn(acc[i][1] * iB);
          o[hB * D + d0 + 8] = __float2bfloat16_rn(acc[i][3] * iB);
        }
      }
      if (a.lse && gid == 0) {
        if (hA < G) a.lse[(int64_t)b * Hq + h * G + hA] = lseA * kLn2;
        if (hB < G) a.lse[(int64_t)b * Hq + h * G + hB] = lseB * kLn2;
      }
    } else {
      const int64_t pi = (pslot * Hkv + h) * G;
#pragma unroll
      for (int i = 0; i < C::KSTEPS; ++i) {
        const int d0 = i * 16 + gid;
        if (hA < G) {
          p.w.po[(pi + hA) * D + d0] = acc[i][0] * iA;
          p.w.po[(pi + hA) * D + d0 + 8] = acc[i][2] * iA;
        }
        if (hB < G) {
          p.w.po[(pi + hB) * D + d0] = acc[i][1] * iB;
          p.w.po[(pi + hB) * D + d0 + 8] = acc[i][3] * iB;
        }
      }
      if (gid == 0) {
        if (hA < G) p.w.plse[pi + hA] = lseA;
        if (hB < G) p.w.plse[pi + hB] = lseB;
      }
    }
    // ---- the last chunk scatters the new token's K and V rows into the pool
    if (grp < 0 && c == nchunks - 1) {
      const int sl = a.out_loc[b];
      if (sl < 0 || (int64_t)sl >= a.num_slots) {
        if (lane == 0) set_status(p.status, kStatusSlotRange);
      } else {
        const int64_t r = ((int64_t)sl * Hkv + h) * D;
        for (int e = lane; e < C::RB / 16; e += 32) {
          ((uint4*)((__nv_bfloat16*)a.k_pool + r))[e] = ((const uint4*)knew)[e];
          ((uint4*)((__nv_bfloat16*)a.v_pool + r))[e] = ((const uint4*)vnew)[e];
        }
      }
    }
    __syncwarp();
  }
  retire_warp(p, lane);
}

// ---------------------------------------------------------------- merge
template <typename T, int D, int G>
__global__ void decode_merge_kernel(Params p) {
  const rc_decode_args& a = p.a;
  const int b = blockIdx.x;
  const int hq = blockIdx.y;
  const int L = a.seq_len[b];
  const int row = a.req_idx[b];
  if (L < 1 || L > a.max_ctx || row < 0 || row >= a.max_reqs) return;
  const int nchunks = (L + p.chunk - 1) / p.chunk;
  if (nchunks == 1) return;
  const int Hkv = a.num_kv_heads;
  const int h = hq / G, g = hq - h * G;
  const int j0 = p.w.pbase[b];
  if ((int64_t)j0 + nchunks > p.w.max_jobs) return;
  float M = -INFINITY;
  for (int c = 0; c < nchunks; ++c) M = fmaxf(M, p.w.plse[((int64_t)(j0 + c) * Hkv + h) * G + g]);
  const int d = threadIdx.x;
  float num = 0.f, den = 0.f;
  for (int c = 0; c < nchunks; ++c) {
    const int64_t pi = ((int64_t)(j0 + c) * Hkv + h) * G + g;
    const float lc = p.w.plse[pi];
    const float w = (lc == -INFINITY) ? 0.f : exp2f(lc - M);
    den += w;
    num = fmaf(w, p.w.po[pi * D + d], num);
  }
  T* o = (T*)a.o + ((int64_t)b * a.num_q_heads + hq) * D;
  o[d] = Elem<T>::from_f(den > 0.f ? num / den : 0.f);
  if (a.lse && d == 0) a.lse[(int64_t)b * a.num_q_heads + hq] = (M + log2f(den)) * kLn2;
}

// ---------------------------------------------------------------- host side
int64_t max_jobs_for(const rc_decode_args* a, int chunk) {
  return (a->max_total_tokens + chunk - 1) / chunk + a->num_reqs;
}

int chunk_of(const rc_decode_args* a) { return a->kv_chunk > 0 ? a->kv_chunk : kDefaultChunk; }

int validate(const rc_decode_args* a) {
  RC_CHECK_ARG(a != nullptr, "rc_decode_attention: args is NULL");
  RC_CHECK_ARG(a->dtype == RC_DTYPE_BF16 || a->dtype == RC_DTYPE_F32,
               "rc_decode_attention: dtype %d", a->dtype);
  RC_CHECK_ARG(a->num_reqs >= 0 && a->num_q_heads > 0 && a->num_kv_heads > 0 &&
                   a->num_q_heads % a->num_kv_heads == 0,
               "rc_decode_attention: bad head counts");
  const int G = a->num_q_heads / a->num_kv_heads;
  RC_CHECK_ARG(G == 1 || G == 2 || G == 4 || G == 8, "rc_decode_attention: group size %d", G);
  RC_CHECK_ARG(a->head_dim == 64 || a->head_dim == 128, "rc_decode_attention: head_dim %d",
               a->head_dim);
  RC_CHECK_ARG(a->max_ctx > 0 && a->max_reqs > 0 && a->num_slots > 0 && a->max_total_tokens >= 0,
               "rc_decode_attention: bad sizes");
  RC_CHECK_ARG(a->kv_chunk == 0 || (a->kv_chunk > 0 && a->kv_chunk % 64 == 0),
               "rc_decode_attention: kv_chunk %d", a->kv_chunk);
  RC_CHECK_ARG(a->num_groups >= 0, "rc_decode_attention: num_groups %d", a->num_groups);
  RC_CHECK_ARG(a->num_groups == 0 ||
                   (a->group_indptr && a->group_members && a->group_shared),
               "rc_decode_attention: group arrays are NULL");
  return RC_OK;
}

template <typename T, int D, int G>
struct MainKernel {
  static constexpr int SMEM = Cfg<T, D, G>::SMEM;
  static constexpr auto fn = decode_main_kernel<T, D, G>;
};
template <int D, int G>
struct MainKernel<__nv_bfloat16, D, G> {
  static constexpr int SMEM = MmaCfg<D>::SMEM;
  static constexpr auto fn = decode_mma_kernel<D, G>;
};

template <typename T, int D, int G>
int launch_t(const Params& p, cudaStream_t s) {
  using C = MainKernel<T, D, G>;
  auto kern = C::fn;
  struct Setup {
    int num_sms = 0, blocks_per_sm = 0;
  };
  static PerDevice<Setup> setup;
  const Setup* su = nullptr;
  const cudaError_t init_err = setup.get(
      [&](Setup& st) {
        cudaError_t e =
            cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
        int dev = 0;
        if (e == cudaSuccess) e = cudaGetDevice(&dev);
        if (e == cudaSuccess)
          e = cudaDeviceGetAttribute(&st.num_sms, cudaDevAttrMultiProcessorCount, dev);
        if (e == cudaSuccess)
          e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&st.blocks_per_sm, kern,
                                                            kWarps * 32, C::SMEM);
        return e;
      },
      &su);
  if (init_err != cudaSuccess)
    return fail(RC_ERR_CUDA, "rc_decode_attention: setup: %s", cudaGetErrorString(init_err));
  // bf16 can reuse the plan of the previous call (the main kernel leaves the item counter reset)
  constexpr bool kMma = std::is_same<T, __nv_bfloat16>::value;
  int n = 0;
  if (!(kMma && p.a.reuse_plan)) {
    decode_plan_kernel<<<1, 1024, 0, s>>>(p);
    ++n;
  }
  const int grid = std::max(1, su->num_sms * std::max(1, su->blocks_per_sm));
  kern<<<grid, kWarps * 32, C::SMEM, s>>>(p);
  ++n;
  dim3 mg(p.a.num_reqs, p.a.num_q_heads);
  decode_merge_kernel<T, D, G><<<mg, D, 0, s>>>(p);
  ++n;
  count_launches(n);
  return check_launch("rc_decode_attention");
}

template <typename T, int D>
int launch_g(const Params& p, int G, cudaStream_t s) {
  switch (G) {
    case 1: return launch_t<T, D, 1>(p, s);
    case 2: return launch_t<T, D, 2>(p, s);
    case 4: return launch_t<T, D, 4>(p, s);
    default: return launch_t<T, D, 8>(p, s);
  }
}

}  // namespace
}  // namespace rc

extern "C" int rc_decode_workspace_bytes(const rc_decode_args* a, size_t* out_bytes) {
  const int v = rc::validate(a);
  if (v != RC_OK) return v;
  RC_CHECK_ARG(out_bytes != nullptr, "rc_decode_workspace_bytes: out_bytes is NULL");
  const int chunk = rc::chunk_of(a);
  const int G = a->num_q_heads / a->num_kv_heads;
  size_t total = 0;
  rc::carve(nullptr, a->num_reqs, G, a->head_dim, rc::max_jobs_for(a, chunk), a->num_kv_heads,
            &total);
  *out_bytes = total;
  return RC_OK;
}

extern "C" int rc_decode_attention(const rc_decode_args* a, void* workspace,
                                   size_t workspace_bytes, void* stream) {
  const int v = rc::validate(a);
  if (v != RC_OK) return v;
  if (a->num_reqs == 0) return RC_OK;
  RC_CHECK_ARG(a->q && a->k_new && a->v_new && a->out_loc && a->seq_len && a->req_idx &&
                   a->req_to_token && a->k_pool && a->v_pool && a->o && workspace,
               "rc_decode_attention: NULL pointer");
  const uintptr_t al = (uintptr_t)a->k_new | (uintptr_t)a->v_new | (uintptr_t)a->k_pool |
                       (uintptr_t)a->v_pool | (uintptr_t)workspace;
  RC_CHECK_ARG((al & 15) == 0, "rc_decode_attention: K/V pointers and workspace must be 16-byte aligned");
  const int chunk = rc::chunk_of(a);
  const int G = a->num_q_heads / a->num_kv_heads;
  size_t need = 0;
  rc::Params p{};
  p.a = *a;
  p.chunk = chunk;
  p.use_groups = (a->dtype == RC_DTYPE_BF16 && a->num_groups > 0) ? 1 : 0;
  p.max_members = 8 / G;
  p.w = rc::carve(workspace, a->num_reqs, G, a->head_dim, rc::max_jobs_for(a, chunk),
                  a->num_kv_heads, &need);
  RC_CHECK_ARG(workspace_bytes >= need, "rc_decode_attention: workspace %zu bytes < %zu needed",
               workspace_bytes, need);
  p.status = rc::device_status_ptr();
  if (!p.status) return rc::fail(RC_ERR_CUDA, "rc_decode_attention: no device status word");
  cudaStream_t s = (cudaStream_t)stream;
  if (a->dtype == RC_DTYPE_BF16)
    return a->head_dim == 128 ? rc::launch_g<__nv_bfloat16, 128>(p, G, s)
                              : rc::launch_g<__nv_bfloat16, 64>(p, G, s);
  return a->head_dim == 128 ? rc::launch_g<float, 128>(p, G, s) : rc::launch_g<float, 64>(p, G, s);
}

// ---------------------------------------------------------------- no-allocation variant
// Scratch for rc_decode_attention_noalloc: a fixed device array of this translation unit, so a
// caller that cannot allocate still gets split-K decode. Its device address is looked up once
// per device (host code may not use the symbol itself as a device pointer).
namespace {
__device__ __align__(256) unsigned char g_decode_scratch[RC_DECODE_STATIC_SCRATCH_BYTES];
void* g_decode_scratch_ptr[rc::kMaxDevices] = {};
std::mutex g_decode_scratch_mu;
}  // namespace

extern "C" int rc_decode_attention_noalloc(const rc_decode_args* a, void* stream) {
  const int v = rc::validate(a);
  if (v != RC_OK) return v;
  size_t need = 0;
  const int rc0 = rc_decode_workspace_bytes(a, &need);
  if (rc0 != RC_OK) return rc0;
  if (need > RC_DECODE_STATIC_SCRATCH_BYTES)
    return rc::fail(RC_ERR_INVALID,
                    "rc_decode_attention_noalloc: these arguments need %zu bytes of scratch but the "
                    "built-in area holds %zu; use a larger kv_chunk or rc_decode_attention",
                    need, (size_t)RC_DECODE_STATIC_SCRATCH_BYTES);
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev < 0 || dev >= rc::kMaxDevices)
    return rc::fail(RC_ERR_CUDA, "rc_decode_attention_noalloc: no usable current device");
  void* ptr = nullptr;
  {
    std::lock_guard<std::mutex> lk(g_decode_scratch_mu);
    if (!g_decode_scratch_ptr[dev]) {
      e = cudaGetSymbolAddress(&ptr, g_decode_scratch);
      if (e != cudaSuccess)
        return rc::fail(RC_ERR_CUDA, "rc_decode_attention_noalloc: scratch address lookup: %s",
                        cudaGetErrorString(e));
      g_decode_scratch_ptr[dev] = ptr;
    }
    ptr = g_decode_scratch_ptr[dev];
  }
  // The shared area's job list may come from another caller's call (or from an fp32 call,
  // which leaves the item counter as it was): always plan afresh.
  rc_decode_args local = *a;
  local.reuse_plan = 0;
  return rc_decode_attention(&local, ptr, RC_DECODE_STATIC_SCRATCH_BYTES, stream);
}
