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
// Warp roles (256 threads):
//   warp 0      producer: per key tile, 32 lanes each gather 4 rows x 2 column blocks with TMA
//               tile::gather4 (box 64 columns x 1 row, 128-byte swizzle) into K and V stages;
//   warp 1      allocates TMEM and issues every tcgen05.mma from one lane:
//               S[j%2] = Q K_j^T (M=128, N=128, K=128; fp32 in TMEM), then O += P_{j-1} V_{j-1};
//   warps 2-3   scatter the tile's new K/V rows into their pool slots;
//   warps 4-7   softmax, one thread per query row (TMEM lane): scores from TMEM, online softmax
//               in base 2 with a lazy rescale of O (only when the running max grows by > 8),
//               P as bf16 into shared memory (the A operand of P V), epilogue O / l.
// Every mbarrier wait is bounded; on expiry the kernel records a status code and unwinds.
#include <cuda.h>

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
constexpr int kThreads = 256;
constexpr float kRescaleThreshold = 8.0f; // log2 units: rescale O only if the max grows by 2^8

struct SmemLayout {
  static constexpr int Q = 0;
  static constexpr int K = Q + kTileBytes;
  static constexpr int V = K + kStagesKV * kTileBytes;
  static constexpr int P = V + kStagesKV * kTileBytes;
  static constexpr int BAR = P + 2 * kTileBytes;
  // barriers: k_full[2], k_empty[2], v_full[2], v_empty[2], s_full[2], s_free[2], p_full[2],
  //           o_done[2]
  static constexpr int NBAR = 16;
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
__device__ __forceinline__ void tma_gather4(uint32_t dst, const CUtensorMap* map, int col, int r0,
                                            int r1, int r2, int r3, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cta.global.tile::gather4.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4, %5, %6}], [%7];" ::"r"(dst),
      "l"(map), "r"(col), "r"(r0), "r"(r1), "r"(r2), "r"(r3), "r"(bar)
      : "memory");
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
__global__ void __launch_bounds__(kThreads, 1)
    extend_tc_kernel(const __grid_constant__ TcParams p, const __grid_constant__ CUtensorMap tk_pool,
                     const __grid_constant__ CUtensorMap tv_pool,
                     const __grid_constant__ CUtensorMap tk_new,
                     const __grid_constant__ CUtensorMap tv_new) {
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
  uint32_t* tmem_slot = (uint32_t*)(smem + SmemLayout::TMEM_SLOT);

  if (threadIdx.x == 0) {
    for (int s = 0; s < 2; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&k_empty[s], 1);
      mbar_init(&v_full[s], 1);
      mbar_init(&v_empty[s], 1);
      mbar_init(&s_full[s], 1);
      mbar_init(&s_free[s], 128);
      mbar_init(&p_full[s], 128);
      mbar_init(&o_done[s], 1);
    }
    fence_mbar_init();
  }
  if (warp == 1) {
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

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    const int32_t* rt = a.req_to_token + (int64_t)row * a.max_ctx;
    // slots of this lane's 4 keys of prefix tile j (invalid ones replaced by slot 0 and reported)
    auto load_slots = [&](int j, int* sl) {
      const int k0 = j * kN + lane * 4;
      if (k0 + 3 < P) {
        const int4 v4 = *(const int4*)(rt + k0);
        sl[0] = v4.x; sl[1] = v4.y; sl[2] = v4.z; sl[3] = v4.w;
      } else {
#pragma unroll
        for (int u = 0; u < 4; ++u) sl[u] = (k0 + u < P) ? rt[k0 + u] : rt[0];
      }
    };
    int nxt[4] = {0, 0, 0, 0};
    if (n_pre > 0) load_slots(0, nxt);
    bool ok = true;
    for (int j = 0; j < ntiles && ok; ++j) {
      const int st = j & 1;
      const uint32_t par_empty = ((j >> 1) - 1) & 1;
      int r[4];
      const CUtensorMap* mk;
      const CUtensorMap* mv;
      if (j < n_pre) {
        int sl[4] = {nxt[0], nxt[1], nxt[2], nxt[3]};
        if (j + 1 < n_pre) load_slots(j + 1, nxt);   // in flight while this tile is issued
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          if (sl[u] < 0 || (int64_t)sl[u] >= a.num_slots) {
            set_status(p.status, kStatusSlotRange);
            sl[u] = 0;
          }
          r[u] = sl[u] * Hkv + hk;
        }
        mk = &tk_pool;
        mv = &tv_pool;
      } else {
        const int s0 = (j - n_pre) * kN + lane * 4;
#pragma unroll
        for (int u = 0; u < 4; ++u) r[u] = (qo + min(s0 + u, S - 1)) * Hkv + hk;
        mk = &tk_new;
        mv = &tv_new;
      }
      if (j >= kStagesKV) ok = mbar_wait(&k_empty[st], par_empty, p.status);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      if (lane == 0) mbar_arrive_expect_tx(&k_full[st], kTileBytes);
      __syncwarp();
      const uint32_t kdst = sK + st * kTileBytes + lane * 4 * 128;
      tma_gather4(kdst, mk, 0, r[0], r[1], r[2], r[3], smem_u32(&k_full[st]));
      tma_gather4(kdst + kBlockBytes, mk, 64, r[0], r[1], r[2], r[3], smem_u32(&k_full[st]));
      if (j >= kStagesKV) ok = mbar_wait(&v_empty[st], par_empty, p.status);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      if (lane == 0) mbar_arrive_expect_tx(&v_full[st], kTileBytes);
      __syncwarp();
      const uint32_t vdst = sV + st * kTileBytes + lane * 4 * 128;
      tma_gather4(vdst, mv, 0, r[0], r[1], r[2], r[3], smem_u32(&v_full[st]));
      tma_gather4(vdst + kBlockBytes, mv, 64, r[0], r[1], r[2], r[3], smem_u32(&v_full[st]));
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    const uint32_t idq = idesc_bf16(false), idv = idesc_bf16(true);
    bool ok = true;
    auto pv = [&](int t) -> bool {
      const int pb = t & 1, st = t & 1;
      if (!mbar_wait(&p_full[pb], (t >> 1) & 1, p.status)) return false;
      if (!mbar_wait(&v_full[st], (t >> 1) & 1, p.status)) return false;
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
    for (int j = 0; j < ntiles && ok; ++j) {
      const int st = j & 1, sb = j & 1;
      ok = mbar_wait(&k_full[st], (j >> 1) & 1, p.status);
      if (ok && j >= 2) ok = mbar_wait(&s_free[sb], ((j >> 1) - 1) & 1, p.status);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
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
      if (j >= 1) ok = __all_sync(0xffffffffu, pv(j - 1));
    }
    if (ok && ntiles > 0) pv(ntiles - 1);
  } else if (warp == 2 || warp == 3) {
    // ------------------------------------------------------------ scatter of the new K/V rows
    // 64 threads copy (row, 16-byte chunk) pairs; each round issues all of a thread's loads
    // before any store so that eight copies are in flight per thread.
    const int t = threadIdx.x - 64;
    const __nv_bfloat16* kn = (const __nv_bfloat16*)a.k_new;
    const __nv_bfloat16* vn = (const __nv_bfloat16*)a.v_new;
    constexpr int kU = 8;
    const int total = npos * 16;
    for (int base = t; base < total; base += 64 * kU) {
      uint4 kv[kU], vv[kU];
      int64_t dst[kU];
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const int e = base + u * 64;
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
    // ------------------------------------------------------------ softmax warpgroup
    const int r = threadIdx.x - 128;                  // query row = TMEM lane
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    const int rows_used = npos * G;
    const int ipos = min(i0 + r / G, S - 1);          // this row's new-token index (clamped)
    float m_run = -INFINITY, l_run = 0.f, l_exact = 0.f;
    bool ok = true;
    uint8_t* pbase = smem + SmemLayout::P;
    for (int j = 0; j < ntiles; ++j) {
      const int sb = j & 1;
      ok = mbar_wait(&s_full[sb], (j >> 1) & 1, p.status);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      float s[128];
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_ld32(tS0 + sb * 128 + lane_off + c * 32, s + c * 32);
      tmem_wait_ld();
      tc_fence_before();
      mbar_arrive(&s_free[sb]);
      // mask and scale; tile max
      int lim;  // keys [0, lim) of this tile are visible to this row
      if (j < n_pre) {
        lim = min(kN, P - j * kN);
      } else {
        lim = min(kN, ipos - (j - n_pre) * kN + 1);
      }
      float mt = -INFINITY;
#pragma unroll
      for (int c = 0; c < 128; ++c) {
        s[c] = c < lim ? s[c] * p.scale2 : -INFINITY;
        mt = fmaxf(mt, s[c]);
      }
      const float m_new = fmaxf(m_run, mt);
      const bool rescale = m_new > m_run + kRescaleThreshold;  // also true for the first tile
      const float m_use = rescale ? m_new : m_run;
      const float alpha = (rescale && m_run != -INFINITY) ? exp2f(m_run - m_new) : 1.f;
      float rs = 0.f, re = 0.f;
      uint32_t pk[64];
#pragma unroll
      for (int c = 0; c < 64; ++c) {
        const float p0 = exp2f(s[2 * c] - m_use);
        const float p1 = exp2f(s[2 * c + 1] - m_use);
        pk[c] = pack_bf16(p0, p1);
        // O is normalised by the sum of the rounded weights P.V uses (so they stay normalised);
        // the log-sum-exp output uses the exact sum
        rs += bf16lo(pk[c]) + bf16hi(pk[c]);
        re += p0 + p1;
      }
      // P[j&1] was read by the P.V of tile j-2; O is touched only after P.V of tile j-1
      if (j >= 2) {
        ok = mbar_wait(&o_done[sb], ((j >> 1) - 1) & 1, p.status);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
      }
      const bool any_rescale = __any_sync(0xffffffffu, rescale && m_run != -INFINITY) && j > 0;
      if (any_rescale) {
        ok = mbar_wait(&o_done[(j - 1) & 1], ((j - 1) >> 1) & 1, p.status);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        tc_fence_after();
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          float o[32];
          tmem_ld32(tO + lane_off + c * 32, o);
          tmem_wait_ld();
#pragma unroll
          for (int u = 0; u < 32; ++u) o[u] *= alpha;
          tmem_st32(tO + lane_off + c * 32, o);
        }
        tmem_wait_st();
      }
      l_run = l_run * alpha + rs;
      l_exact = l_exact * alpha + re;
      m_run = m_use;
      uint8_t* prow = pbase + sb * kTileBytes;
#pragma unroll
      for (int c = 0; c < 16; ++c)
        *(uint4*)(prow + sw128_off(r, c)) =
            make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
      fence_async_smem();
      tc_fence_before();
      mbar_arrive(&p_full[sb]);
    }
    // epilogue
    if (ok && ntiles > 0) {
      const int t = ntiles - 1;
      ok = mbar_wait(&o_done[t & 1], (t >> 1) & 1, p.status);
      ok = __all_sync(0xffffffffu, ok);
    }
    if (ok && ntiles > 0) {
      tc_fence_after();
      const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
      const bool store = r < rows_used;
      const int i = i0 + r / G, hh = r % G;
      __nv_bfloat16* orow = (__nv_bfloat16*)a.o + ((int64_t)(qo + i) * Hq + hk * G + hh) * kD;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        float o[32];
        tmem_ld32(tO + lane_off + c * 32, o);
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
      if (store && a.lse) a.lse[(int64_t)(qo + i) * Hq + hk * G + hh] = (m_run + log2f(l_exact)) * kLn2;
    }
  }
  // drain: every tcgen05 op issued by warp 1 has completed once o_done / s_full of the last
  // tiles were observed; make sure before freeing TMEM
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;" ::"r"(tmem) : "memory");
  }
}

// ---------------------------------------------------------------- host side
using EncodeFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                              const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                              const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                              CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeFn encode_fn() {
  static EncodeFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, []() {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = (EncodeFn)p;
  });
  return fn;
}

// rows x 128 bf16 matrix, gathered one row at a time in 64-column boxes with 128-byte swizzle
int make_row_map(CUtensorMap* m, const void* base, int64_t rows) {
  EncodeFn fn = encode_fn();
  if (!fn) return fail(RC_ERR_CUDA, "extend: cuTensorMapEncodeTiled unavailable");
  const cuuint64_t dims[2] = {(cuuint64_t)kD, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)kD * 2};
  const cuuint32_t box[2] = {64, 1};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(RC_ERR_CUDA, "extend: tensor map encode failed (%d)", (int)r);
  return RC_OK;
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
  CUtensorMap mk, mv, mkn, mvn;
  const int64_t pool_rows = a->num_slots * a->num_kv_heads;
  const int64_t new_rows = a->num_tokens * a->num_kv_heads;
  int rc;
  if ((rc = make_row_map(&mk, a->k_pool, pool_rows)) != RC_OK) return rc;
  if ((rc = make_row_map(&mv, a->v_pool, pool_rows)) != RC_OK) return rc;
  if ((rc = make_row_map(&mkn, a->k_new, new_rows)) != RC_OK) return rc;
  if ((rc = make_row_map(&mvn, a->v_new, new_rows)) != RC_OK) return rc;
  TcParams p;
  p.a = *a;
  p.status = status;
  p.ppt = kM / G;
  p.scale2 = a->sm_scale * kLog2e;
  dim3 grid((a->max_q_len + p.ppt - 1) / p.ppt, a->num_kv_heads, a->num_reqs);
  extend_tc_kernel<<<grid, kThreads, SmemLayout::ALLOC, s>>>(p, mk, mv, mkn, mvn);
  count_launches(1);
  return check_launch("rc_extend_attention (tensor cores)");
}

}  // namespace rc
