// Extend attention on the 5th-generation tensor cores (tcgen05, TMEM accumulators), bf16,
// head_dim 128. SGLang blog Sec. 2.3 ("compute only the unmatched tokens") and paper digest
// App. A.1: the new tokens' queries attend to the request's cached prefix KV -- gathered from
// the paged pool through the slot table -- and causally to the new tokens' own K/V.
//
// One CTA = (request, KV head, tile of 128 query rows). With G = Hq / Hkv query heads per KV
// head, a tile packs floor(128 / G) query positions x G heads, so every K/V tile loaded is used
// by all heads of the group. Keys are processed in tiles of 128: first the prefix (slots from
// req_to_token, rows gathered from the pool), then the new tokens (rows of k_new / v_new), the
// causal mask applied only where a tile crosses the diagonal.
//
// Warp roles (512 threads, four warpgroups):
//   warps 0-3   producers (0-1 for K, 2-3 for V): gather the key tile's rows (256 B each, one
//               slot per row) with 16-byte cp.async copies straight into the 128-byte-swizzled
//               operand layout, two rows per warp instruction (fully coalesced); completion is
//               signalled on the stage's mbarrier with cp.async.mbarrier.arrive.noinc. (TMA tile::gather4 moves
//               only 512 B per instruction and, measured here, its issue rate capped a 256-byte
//               row gather at about 2 TB/s for the whole GPU; the copy engine path does not.)
//   warp 4      allocates TMEM and issues every tcgen05.mma from one lane:
//               S[j%2] = Q K_j^T (M=128, N=128, K=128; fp32 in TMEM), then O += P_{j-1} V_{j-1};
//   warps 5-7   scatter the tile's new K/V rows into their pool slots;
//   warps 8-15  softmax, two threads per query row (TMEM lane), 64 columns each: two passes
//               over the scores (row max -- combined with the partner thread through shared
//               memory -- then exp2 with the scale folded into one packed FMA), lazy rescale
//               of O (only when the running max grows by > 8 in log2 units), P as bf16 into
//               shared memory (the A operand of P V), epilogue O / l.
// Every mbarrier wait is bounded; on expiry the kernel records a status code and unwinds.
#include <mutex>

#include "device_common.cuh"
#include "extend_common.h"
#include "host_common.h"

namespace rc {
namespace {

constexpr int kD = 128;           // head_dim
constexpr int kM = 128;           // query rows per tile (TMEM lanes)
constexpr int kN = 128;           // keys per tile
constexpr int kStagesKV = 2;
constexpr int kTileBytes = kM * kD * 2;   // 32 KB: one 128 x 128 bf16 operand tile
constexpr int kBlockBytes = kM * 128;     // 16 KB: one 64-column block of a tile
constexpr int kThreads = 512;
constexpr int kProducers = 128;          // warps 0-3
constexpr int kMmaWarp = 4;
constexpr int kSoftmax0 = 256;           // first softmax thread (warps 8-15)
constexpr int kSoftmaxThreads = 256;     // two threads per query row, 64 columns each
constexpr float kRescaleThreshold = 8.0f; // log2 units: rescale O only if the max grows by 2^8

struct SmemLayout {
  static constexpr int Q = 0;
  static constexpr int K = Q + kTileBytes;
  static constexpr int V = K + kStagesKV * kTileBytes;
  static constexpr int P = V + kStagesKV * kTileBytes;
  static constexpr int BAR = P + 2 * kTileBytes;
  // barriers: k_full[2], k_empty[2], v_full[2], v_empty[2], s_full[2], s_free[2], p_full[2],
  //           o_done[2], x_done[2] (softmax partner exchange), e_done (epilogue exchange)
  static constexpr int NBAR = 19;
  static constexpr int TMEM_SLOT = BAR + NBAR * 8;
  static constexpr int TOTAL = TMEM_SLOT + 16;
  static constexpr int ALLOC = TOTAL + 1024;  // room to align the base to 1024 bytes
};
static_assert(SmemLayout::ALLOC <= 232448, "shared memory budget");

struct TcParams {
  rc_extend_args a;
  int* status;
  int ppt;        // query positions per tile
  float scale2;   // sm_scale * log2(e)
};

// ---------------------------------------------------------------- PTX wrappers
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_arrive_noinc(uint32_t bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ uint64_t f2pack(float a, float b) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ void f2unpack(uint64_t r, float& a, float& b) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(r));
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t add2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= (uint64_t)((addr >> 4) & 0x3FFF);
  d |= (uint64_t)((lbo >> 4) & 0x3FFF) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFF) << 32;
  d |= (uint64_t)1 << 46;   // descriptor version for tcgen05
  d |= (uint64_t)2 << 61;   // 128-byte swizzle
  return d;
}

// kind::f16 instruction descriptor: bf16 A and B, fp32 D, M = 128, N = 128
__host__ __device__ constexpr uint32_t idesc_bf16(bool b_mn_major) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((b_mn_major ? 1u : 0u) << 16) |
         ((uint32_t)(kN >> 3) << 17) | ((uint32_t)(kM >> 4) << 24);
}

__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                         uint32_t accum) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(accum));
}

__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void fence_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// 32 consecutive fp32 columns of this thread's TMEM lane
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float* v) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float* v) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,"
      "%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(
          taddr),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
      "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
      "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
      "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
      "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
      "r"(__float_as_uint(v[15])), "r"(__float_as_uint(v[16])), "r"(__float_as_uint(v[17])),
      "r"(__float_as_uint(v[18])), "r"(__float_as_uint(v[19])), "r"(__float_as_uint(v[20])),
      "r"(__float_as_uint(v[21])), "r"(__float_as_uint(v[22])), "r"(__float_as_uint(v[23])),
      "r"(__float_as_uint(v[24])), "r"(__float_as_uint(v[25])), "r"(__float_as_uint(v[26])),
      "r"(__float_as_uint(v[27])), "r"(__float_as_uint(v[28])), "r"(__float_as_uint(v[29])),
      "r"(__float_as_uint(v[30])), "r"(__float_as_uint(v[31]))
      : "memory");
}
__device__ __forceinline__ void tmem_st1(uint32_t taddr, float v) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x1.b32 [%0], {%1};" ::"r"(taddr),
               "r"(__float_as_uint(v))
               : "memory");
}
__device__ __forceinline__ float tmem_ld1(uint32_t taddr) {
  uint32_t r;
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x1.b32 {%0}, [%1];" : "=r"(r) : "r"(taddr));
  return __uint_as_float(r);
}
__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *(const uint32_t*)&v;
}

// byte offset of 16-byte chunk c (0..15) of row r inside a 128 x 128 bf16 SW128 K-major tile
__device__ __forceinline__ uint32_t sw128_off(int r, int c) {
  return (uint32_t)((c >> 3) * kBlockBytes + r * 128 + (((c & 7) ^ (r & 7)) << 4));
}

// ---------------------------------------------------------------- the kernel
__global__ void __launch_bounds__(kThreads, 1) extend_tc_kernel(const __grid_constant__ TcParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // 128-byte swizzled operand tiles must start on 1024-byte boundaries
  uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  const rc_extend_args& a = p.a;
  const int b = blockIdx.z;
  const int hk = blockIdx.y;
  const int qt = blockIdx.x;
  const int qo = a.qo_indptr[b];
  const int S = a.qo_indptr[b + 1] - qo;
  const int P = a.prefix_len[b];
  const int G = a.num_q_heads / a.num_kv_heads;
  const int i0 = qt * p.ppt;
  if (S <= 0 || i0 >= S) return;
  const int row = a.req_idx[b];
  if (P < 0 || (int64_t)P + S > a.max_ctx || row < 0 || row >= a.max_reqs || qo < 0 ||
      (int64_t)qo + S > a.num_tokens) {
    if (threadIdx.x == 0) set_status(p.status, kStatusPosRange);
    return;
  }
  const int npos = min(p.ppt, S - i0);         // query positions in this tile
  const int kend_s = i0 + npos;                // new-token keys visible to some row: [0, kend_s)
  const int n_pre = (P + kN - 1) / kN;
  const int n_suf = (kend_s + kN - 1) / kN;
  const int ntiles = n_pre + n_suf;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int Hq = a.num_q_heads, Hkv = a.num_kv_heads;

  const uint32_t sbase = smem_u32(smem);
  const uint32_t sQ = sbase + SmemLayout::Q;
  const uint32_t sK = sbase + SmemLayout::K;
  const uint32_t sV = sbase + SmemLayout::V;
  const uint32_t sP = sbase + SmemLayout::P;
  uint64_t* bars = (uint64_t*)(smem + SmemLayout::BAR);
  uint64_t* k_full = bars + 0;
  uint64_t* k_empty = bars + 2;
  uint64_t* v_full = bars + 4;
  uint64_t* v_empty = bars + 6;
  uint64_t* s_full = bars + 8;
  uint64_t* s_free = bars + 10;
  uint64_t* p_full = bars + 12;
  uint64_t* o_done = bars + 14;
  uint64_t* x_done = bars + 16;
  uint64_t* e_done = bars + 18;
  uint32_t* tmem_slot = (uint32_t*)(smem + SmemLayout::TMEM_SLOT);

  if (threadIdx.x == 0) {
    for (int s = 0; s < 2; ++s) {
      mbar_init(&k_full[s], kProducers / 2);
      mbar_init(&k_empty[s], 1);
      mbar_init(&v_full[s], kProducers / 2);
      mbar_init(&v_empty[s], 1);
      mbar_init(&s_full[s], 1);
      mbar_init(&s_free[s], kSoftmaxThreads);
      mbar_init(&p_full[s], kSoftmaxThreads);
      mbar_init(&o_done[s], 1);
      mbar_init(&x_done[s], kSoftmaxThreads);
    }
    mbar_init(e_done, kSoftmaxThreads);
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;" ::"r"(
                     smem_u32(tmem_slot))
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  // Q tile: row m = (position i0 + m / G, head hk * G + m % G); rows past the tile are zero
  {
    const __nv_bfloat16* q = (const __nv_bfloat16*)a.q;
    const int rows_used = npos * G;
    for (int e = threadIdx.x; e < kM * 16; e += kThreads) {
      const int m = e >> 4, c = e & 15;
      uint4 v = make_uint4(0, 0, 0, 0);
      if (m < rows_used) {
        const int i = i0 + m / G, hh = m % G;
        v = *(const uint4*)(q + ((int64_t)(qo + i) * Hq + hk * G + hh) * kD + c * 8);
      }
      *(uint4*)(smem + SmemLayout::Q + sw128_off(m, c)) = v;
    }
  }
  fence_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t tS0 = tmem, tO = tmem + 256;

  if (warp < 4) {
    // ------------------------------------------------------------ producers (warps 0-3)
    // Warps 0-1 load the K tiles and warps 2-3 the V tiles, each side at its own pace (a K tile
    // only waits for the QK that last read its stage, a V tile for the P.V). Warp w covers rows
    // [64 (w & 1), 64 (w & 1) + 64) of a tile in two halves of 32: lane l resolves the source
    // row of tile row 64 (w & 1) + 32 h + l, and one copy instruction moves 16-byte chunk
    // (l & 15) of two rows.
    const int32_t* rt = a.req_to_token + (int64_t)row * a.max_ctx;
    const bool is_v = warp >= 2;
    const __nv_bfloat16* pool = (const __nv_bfloat16*)(is_v ? a.v_pool : a.k_pool);
    const __nv_bfloat16* nsrc = (const __nv_bfloat16*)(is_v ? a.v_new : a.k_new);
    uint64_t* full = is_v ? v_full : k_full;
    uint64_t* empty = is_v ? v_empty : k_empty;
    const uint32_t sdst = is_v ? sV : sK;
    const int rbase = (warp & 1) * 64;
    // raw_row(j, h) only issues the slot load; row_of() checks it when the tile is issued, so
    // the load of tile j+1 stays in flight while tile j is being copied
    auto raw_row = [&](int j, int h) -> int {
      if (j < n_pre) {
        const int key = j * kN + rbase + h * 32 + lane;
        return rt[key < P ? key : P - 1];
      }
      return 0;
    };
    auto row_of = [&](int j, int h, int raw) -> int {
      if (j < n_pre) {
        int sl = raw;
        if (sl < 0 || (int64_t)sl >= a.num_slots) {
          set_status(p.status, kStatusSlotRange);
          sl = 0;
        }
        return sl * Hkv + hk;
      }
      const int s0 = (j - n_pre) * kN + rbase + h * 32 + lane;
      return (qo + min(s0, S - 1)) * Hkv + hk;
    };
    int nxt0 = raw_row(0, 0), nxt1 = raw_row(0, 1);
    bool ok = true;
    const int c = lane & 15, half = lane >> 4;
    for (int j = 0; j < ntiles && ok; ++j) {
      const int st = j & 1;
      const int cur0 = row_of(j, 0, nxt0), cur1 = row_of(j, 1, nxt1);
      if (j + 1 < ntiles) {  // in flight while this tile is issued
        nxt0 = raw_row(j + 1, 0);
        nxt1 = raw_row(j + 1, 1);
      }
      const __nv_bfloat16* src = j < n_pre ? pool : nsrc;
      if (j >= kStagesKV) ok = mbar_wait(&empty[st], ((j >> 1) - 1) & 1, p.status);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      const uint32_t dst = sdst + st * kTileBytes;
#pragma unroll 4
      for (int i = 0; i < 32; ++i) {
        const int rr = 2 * i + half;                       // 0..63 within this warp's rows
        const int srow = __shfl_sync(0xffffffffu, rr < 32 ? cur0 : cur1, rr & 31);
        cp_async16(dst + sw128_off(rbase + rr, c), src + (int64_t)srow * kD + c * 8);
      }
      cp_async_arrive_noinc(smem_u32(&full[st]));
    }
    asm volatile("cp.async.wait_all;" ::: "memory");
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    const uint32_t idq = idesc_bf16(false), idv = idesc_bf16(true);
    bool ok = true;
    auto pv = [&](int t) -> bool {
      const int pb = t & 1, st = t & 1;
      if (!mbar_wait(&p_full[pb], (t >> 1) & 1, p.status)) return false;
      if (!mbar_wait(&v_full[st], (t >> 1) & 1, p.status)) return false;
      fence_async_smem();   // V arrived through the generic proxy (cp.async)
      tc_fence_after();
      if (lane == 0) {
#pragma unroll
        for (int kk = 0; kk < kN / 16; ++kk) {
          // A = P (K-major over keys), B = V (MN-major: d contiguous, keys as rows)
          const uint64_t ad = smem_desc_sw128(sP + pb * kTileBytes + (kk >> 2) * kBlockBytes +
                                                  (kk & 3) * 32, 16, 1024);
          const uint64_t bd = smem_desc_sw128(sV + st * kTileBytes + kk * 2048, kBlockBytes, 1024);
          mma_bf16(tO, ad, bd, idv, (t > 0 || kk > 0) ? 1u : 0u);
        }
        mma_commit(smem_u32(&o_done[pb]));
        mma_commit(smem_u32(&v_empty[st]));
      }
      __syncwarp();
      return true;
    };
    // S = Q K_j^T into S[j & 1]; S[j & 1] is free again once the softmax has read S_{j-2}
    auto qk = [&](int j) -> bool {
      const int st = j & 1, sb = j & 1;
      if (!mbar_wait(&k_full[st], (j >> 1) & 1, p.status)) return false;
      if (j >= 2 && !mbar_wait(&s_free[sb], ((j >> 1) - 1) & 1, p.status)) return false;
      fence_async_smem();   // K arrived through the generic proxy (cp.async)
      tc_fence_after();
      if (lane == 0) {
#pragma unroll
        for (int kk = 0; kk < kD / 16; ++kk) {
          const uint32_t off = (kk >> 2) * kBlockBytes + (kk & 3) * 32;
          const uint64_t ad = smem_desc_sw128(sQ + off, 16, 1024);
          const uint64_t bd = smem_desc_sw128(sK + st * kTileBytes + off, 16, 1024);
          mma_bf16(tS0 + sb * 128, ad, bd, idq, kk > 0 ? 1u : 0u);
        }
        mma_commit(smem_u32(&s_full[sb]));
        mma_commit(smem_u32(&k_empty[st]));
      }
      __syncwarp();
      return true;
    };
    // two score tiles ahead of the softmax, then P.V of tile j as soon as its P is written,
    // followed by the scores of tile j + 2 into the buffer the softmax just released
    if (ntiles > 0) ok = __all_sync(0xffffffffu, qk(0));
    if (ok && ntiles > 1) ok = __all_sync(0xffffffffu, qk(1));
    for (int j = 0; j < ntiles && ok; ++j) {
      ok = __all_sync(0xffffffffu, pv(j));
      if (ok && j + 2 < ntiles) ok = __all_sync(0xffffffffu, qk(j + 2));
    }
  } else if (warp < 8) {
    // ------------------------------------------------------------ scatter of the new K/V rows
    // 96 threads copy (row, 16-byte chunk) pairs; each round issues all of a thread's loads
    // before any store so that four copies are in flight per thread.
    const int t = threadIdx.x - 160;
    const __nv_bfloat16* kn = (const __nv_bfloat16*)a.k_new;
    const __nv_bfloat16* vn = (const __nv_bfloat16*)a.v_new;
    constexpr int kU = 4;
    const int total = npos * 16;
    for (int base = t; base < total; base += 96 * kU) {
      uint4 kv[kU], vv[kU];
      int64_t dst[kU];
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const int e = base + u * 96;
        dst[u] = -1;
        if (e < total) {
          const int i = i0 + (e >> 4), c = e & 15;
          const int64_t tok = qo + i;
          const int sl = a.out_loc[tok];
          const int64_t src = (tok * Hkv + hk) * kD + c * 8;
          kv[u] = *(const uint4*)(kn + src);
          vv[u] = *(const uint4*)(vn + src);
          if (sl >= 0 && (int64_t)sl < a.num_slots)
            dst[u] = ((int64_t)sl * Hkv + hk) * kD + c * 8;
          else if (c == 0)
            set_status(p.status, kStatusSlotRange);
        }
      }
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        if (dst[u] >= 0) {
          *(uint4*)((__nv_bfloat16*)a.k_pool + dst[u]) = kv[u];
          *(uint4*)((__nv_bfloat16*)a.v_pool + dst[u]) = vv[u];
        }
      }
    }
  } else {
    // ------------------------------------------------------------ softmax warpgroups
    const int hf = (warp - 8) >> 2;                   // column half: [64 hf, 64 hf + 64)
    const int r = (warp & 3) * 32 + lane;             // query row = TMEM lane
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    const int rows_used = npos * G;
    const int ipos = min(i0 + r / G, S - 1);          // this row's new-token index (clamped)
    const float sc2 = p.scale2;
    const uint64_t sc2x2 = f2pack(sc2, sc2);
    // partner exchange through spare TMEM columns (same lane, so the same quadrant): row maxima
    // at 448 + 2 * (tile parity) + half, final sums at 452 + 2 * (which sum) + half
    const uint32_t tX = tmem + 448 + lane_off;
    float m_run = -INFINITY, l_run = 0.f, l_exact = 0.f;
    bool ok = true;
    uint8_t* pbase = smem + SmemLayout::P;
    const int c0 = hf * 64;                           // first column of this thread
    for (int j = 0; j < ntiles; ++j) {
      const int sb = j & 1;
      ok = mbar_wait(&s_full[sb], (j >> 1) & 1, p.status);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      // keys [0, lim) of this tile are visible to this row
      const int lim = j < n_pre ? min(kN, P - j * kN) : min(kN, ipos - (j - n_pre) * kN + 1);
      const bool full = __all_sync(0xffffffffu, lim >= c0 + 64);
      const uint32_t tS = tS0 + sb * 128 + lane_off + c0;
      // pass 1: row max of the raw scores, combined with the partner thread
      float mx = -INFINITY;
#pragma unroll 1
      for (int c = 0; c < 2; ++c) {
        float v[32];
        tmem_ld32(tS + c * 32, v);
        tmem_wait_ld();
        if (full) {
#pragma unroll
          for (int u = 0; u < 32; ++u) mx = fmaxf(mx, v[u]);
        } else {
#pragma unroll
          for (int u = 0; u < 32; ++u) mx = fmaxf(mx, c0 + c * 32 + u < lim ? v[u] : -INFINITY);
        }
      }
      tmem_st1(tX + sb * 2 + hf, mx);
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&x_done[sb]);
      ok = mbar_wait(&x_done[sb], (j >> 1) & 1, p.status);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      mx = fmaxf(mx, tmem_ld1(tX + sb * 2 + (hf ^ 1)));
      tmem_wait_ld();
      const float mt = mx * sc2;                      // sc2 > 0: max commutes with the scale
      const float m_new = fmaxf(m_run, mt);
      const bool rescale = m_new > m_run + kRescaleThreshold;  // also true for the first tile
      const float m_use = rescale ? m_new : m_run;
      const float alpha = (rescale && m_run != -INFINITY) ? ex2(m_run - m_new) : 1.f;
      const uint64_t negx2 = f2pack(-m_use, -m_use);
      // P[j&1] was read by the P.V of tile j-2
      if (j >= 2) {
        ok = mbar_wait(&o_done[sb], ((j >> 1) - 1) & 1, p.status);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
      }
      // pass 2: weights, written as bf16 into the P operand tile
      uint64_t rs2 = 0, re2 = 0;   // packed (even, odd) partial sums: rounded and exact
      uint8_t* prow = pbase + sb * kTileBytes;
#pragma unroll 1
      for (int c = 0; c < 2; ++c) {
        float v[32];
        tmem_ld32(tS + c * 32, v);
        tmem_wait_ld();
        if (!full) {
#pragma unroll
          for (int u = 0; u < 32; ++u) v[u] = c0 + c * 32 + u < lim ? v[u] : -INFINITY;
        }
        uint32_t pk[16];
#pragma unroll
        for (int u = 0; u < 16; ++u) {
          float x0, x1;
          f2unpack(fma2(f2pack(v[2 * u], v[2 * u + 1]), sc2x2, negx2), x0, x1);
          const float p0 = ex2(x0), p1 = ex2(x1);
          pk[u] = pack_bf16(p0, p1);
          // O is normalised by the sum of the rounded weights P.V uses; the log-sum-exp
          // output uses the exact sum
          rs2 = add2(rs2, f2pack(bf16lo(pk[u]), bf16hi(pk[u])));
          re2 = add2(re2, f2pack(p0, p1));
        }
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4)
          *(uint4*)(prow + sw128_off(r, hf * 8 + c * 4 + q4)) =
              make_uint4(pk[4 * q4], pk[4 * q4 + 1], pk[4 * q4 + 2], pk[4 * q4 + 3]);
      }
      tc_fence_before();
      mbar_arrive(&s_free[sb]);
      // O is touched only after the P.V of tile j-1; each thread rescales its half of O
      const bool any_rescale = __any_sync(0xffffffffu, rescale && m_run != -INFINITY) && j > 0;
      if (any_rescale) {
        ok = mbar_wait(&o_done[(j - 1) & 1], ((j - 1) >> 1) & 1, p.status);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        tc_fence_after();
#pragma unroll 1
        for (int c = 0; c < 2; ++c) {
          float o[32];
          tmem_ld32(tO + lane_off + c0 + c * 32, o);
          tmem_wait_ld();
#pragma unroll
          for (int u = 0; u < 32; ++u) o[u] *= alpha;
          tmem_st32(tO + lane_off + c0 + c * 32, o);
        }
        tmem_wait_st();
      }
      float a0, a1, b0, b1;
      f2unpack(rs2, a0, a1);
      f2unpack(re2, b0, b1);
      l_run = l_run * alpha + (a0 + a1);
      l_exact = l_exact * alpha + (b0 + b1);
      m_run = m_use;
      fence_async_smem();
      tc_fence_before();
      mbar_arrive(&p_full[sb]);
    }
    // epilogue: full denominators from both halves, then this thread's half of the O row
    if (ok && ntiles > 0) {
      const int t = ntiles - 1;
      ok = mbar_wait(&o_done[t & 1], (t >> 1) & 1, p.status);
      ok = __all_sync(0xffffffffu, ok);
    }
    tmem_st1(tX + 4 + hf, l_run);
    tmem_st1(tX + 6 + hf, l_exact);
    tmem_wait_st();
    tc_fence_before();
    mbar_arrive(e_done);
    if (ok) ok = __all_sync(0xffffffffu, mbar_wait(e_done, 0, p.status));
    tc_fence_after();
    l_run += tmem_ld1(tX + 4 + (hf ^ 1));
    l_exact += tmem_ld1(tX + 6 + (hf ^ 1));
    tmem_wait_ld();
    if (ok && ntiles > 0) {
      tc_fence_after();
      const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
      const bool store = r < rows_used;
      const int i = i0 + r / G, hh = r % G;
      __nv_bfloat16* orow =
          (__nv_bfloat16*)a.o + ((int64_t)(qo + i) * Hq + hk * G + hh) * kD + c0;
#pragma unroll 1
      for (int c = 0; c < 2; ++c) {
        float o[32];
        tmem_ld32(tO + lane_off + c0 + c * 32, o);
        tmem_wait_ld();
        if (store) {
#pragma unroll
          for (int u = 0; u < 32; u += 8) {
            *(uint4*)(orow + c * 32 + u) =
                make_uint4(pack_bf16(o[u] * inv, o[u + 1] * inv),
                           pack_bf16(o[u + 2] * inv, o[u + 3] * inv),
                           pack_bf16(o[u + 4] * inv, o[u + 5] * inv),
                           pack_bf16(o[u + 6] * inv, o[u + 7] * inv));
          }
        }
      }
      if (store && hf == 0 && a.lse)
        a.lse[(int64_t)(qo + i) * Hq + hk * G + hh] = (m_run + log2f(l_exact)) * kLn2;
    }
  }
  // every tcgen05 op has completed once the softmax observed the last o_done; free TMEM
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;" ::"r"(tmem) : "memory");
  }
}

}  // namespace

int launch_extend_tc(const rc_extend_args* a, int* status, cudaStream_t s) {
  if (a->head_dim != kD) return fail(RC_ERR_INVALID, "extend (tensor cores): head_dim must be 128");
  const int G = a->num_q_heads / a->num_kv_heads;
  if (G > kM) return fail(RC_ERR_INVALID, "extend (tensor cores): group size %d > 128", G);
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, []() {
    attr_err = cudaFuncSetAttribute(extend_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    SmemLayout::ALLOC);
  });
  if (attr_err != cudaSuccess)
    return fail(RC_ERR_CUDA, "extend (tensor cores): %s", cudaGetErrorString(attr_err));
  TcParams p;
  p.a = *a;
  p.status = status;
  p.ppt = kM / G;
  p.scale2 = a->sm_scale * kLog2e;
  dim3 grid((a->max_q_len + p.ppt - 1) / p.ppt, a->num_kv_heads, a->num_reqs);
  extend_tc_kernel<<<grid, kThreads, SmemLayout::ALLOC, s>>>(p);
  count_launches(1);
  return check_launch("rc_extend_attention (tensor cores)");
}

}  // namespace rc
