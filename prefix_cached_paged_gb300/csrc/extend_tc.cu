// Extend attention on the 5th-generation tensor cores (tcgen05, TMEM accumulators), bf16,
// head_dim 128. SGLang blog Sec. 2.3 ("compute only the unmatched tokens") and paper digest
// App. A.1: the new tokens' queries attend to the request's cached prefix KV -- gathered from
// the paged pool through the slot table -- and causally to the new tokens' own K/V.
//
// One CTA = (request, KV head, two tiles A and B of 128 query rows). With G = Hq / Hkv query
// heads per KV head, a tile packs floor(128 / G) query positions x G heads, so every K/V tile
// gathered serves all heads of the group and both query tiles. Keys are processed in tiles of
// 128: first the prefix (slots from req_to_token, rows gathered from the pool), then the new
// tokens (rows of k_new / v_new); the causal mask is applied only where a tile crosses the
// diagonal, and a query tile skips key tiles that lie entirely in its future.
//
// The two query tiles ping-pong on the tensor core: while the softmax of tile A turns its scores
// into weights, the MMA warp runs P.V and the next Q K^T of tile B, and the other way round.
// A CTA with a single query tile (short suffixes) splits its key tiles instead: the even key
// tiles form virtual tile 0 and the odd ones virtual tile 1, each with its own running max, sum
// and O accumulator, merged with log-sum-exp weights at the end.
//
// TMEM (512 columns): S_A [0,128) S_B [128,256) scores (fp32); O_A [256,384) O_B [384,512)
// outputs (fp32). The bf16 weights P overwrite the first 64 columns of the scores they came from
// (two weights per 32-bit column) and feed P.V straight from TMEM as the A operand.
//
// The two Q tiles arrive by TMA (one tensor box of 64 columns x G heads x 128 / G positions per
// 64-column block, 128-byte swizzled), issued by thread 0 right after the barrier set-up.
//
// Warp roles (512 threads):
//   warp 0       allocates TMEM and issues every tcgen05.mma from one lane;
//   warps 1-4    producers, two for K and two for V, each filling half of a key tile's rows
//                (256 B, one slot per row) with 16-byte cp.async copies straight into the
//                128-byte-swizzled operand layout, two rows per instruction (fully coalesced);
//                completion is signalled with cp.async.mbarrier.arrive.noinc. (TMA
//                tile::gather4 moves 512 B per instruction and, measured here, its issue rate
//                capped a 256-byte row gather at about 2 TB/s GPU-wide; the copy path does not.
//                The copy path is itself bound by instruction issue, hence two warps per
//                operand and one shuffled row pointer per copy.)
//   warps 5-7    scatter the new tokens' K/V rows into their pool slots;
//   warps 8-11   softmax of query tile A, warps 12-15 of tile B: one thread per query row holds
//                the row's 128 scores in registers; one pass (row max, then exp2 with the scale
//                folded into one packed FMA); lazy rescale of O (only when the running max
//                grows by more than 8 in log2 units); weights rounded to bf16, normalised by
//                the sum of the rounded weights; epilogue O / l.
// Every mbarrier wait is bounded; on expiry the kernel records a status code and unwinds.
#include <cuda.h>
#include <cudaTypedefs.h>

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
constexpr int kMmaWarp = 0;
constexpr int kProdWarps = 2;             // producer warps per operand
constexpr int kKWarp0 = 1, kVWarp0 = kKWarp0 + kProdWarps;
constexpr int kScatterWarp0 = kVWarp0 + kProdWarps, kScatterWarps = 3;
constexpr int kSoftmaxWarp0 = kScatterWarp0 + kScatterWarps;
static_assert(kSoftmaxWarp0 == 8 && kThreads == 32 * (kSoftmaxWarp0 + 8), "warp roles");
constexpr int kGroupThreads = 128;        // softmax threads of one query tile (one per row)
// control warpgroups (warps 0-7) give registers up, the softmax warpgroups (8-15) take them
// The kernel exists twice: without prefix-stacking support, and with it (the stacked pass and
// the merge in the epilogue need a few more registers in the softmax warps).
constexpr int kRegsLaunch = 128;
template <bool kStack> struct Regs {
  static constexpr int control = kStack ? 64 : 72, softmax = kStack ? 192 : 184;
  static_assert(kThreads * kRegsLaunch <= 65536, "register file");
  static_assert(256 * control + 256 * softmax <= kThreads * kRegsLaunch,
                "a register split above the launch allocation never completes");
};
constexpr float kRescaleThreshold = 8.0f; // log2 units: rescale O only if the max grows by 2^8
constexpr int kFoldTiles = 512;           // remainder tiles of one CTA of a folded pass, at most
constexpr int kFoldMembers = 256;         // members of one CTA of a folded pass, at most

struct SmemLayout {
  static constexpr int Q = 0;                                   // Q_A, Q_B
  static constexpr int K = Q + 2 * kTileBytes;
  static constexpr int V = K + kStagesKV * kTileBytes;
  static constexpr int BAR = V + kStagesKV * kTileBytes;
  // k_full[2] k_empty[2] v_full[2] v_empty[2] s_full[2] (unused)[2] o_done[2] e_done q_full drain
  static constexpr int NBAR = 4 * kStagesKV + 9;
  static constexpr int TMEM_SLOT = BAR + NBAR * 8;   // TMEM address; MMA_DONE 8 bytes on
  static constexpr int MMA_DONE = TMEM_SLOT + 8;     // set once the MMA warp syncs no more
  // split-mode merge: row maxima, rounded and exact sums of each virtual tile [X][row]
  static constexpr int XMRG = TMEM_SLOT + 16;
  // folded stacked pass: remainder tile u -> (member offset << 16 | tile of member), and the
  // first remainder tile of each member of the CTA
  static constexpr int FMAP = XMRG + 3 * 2 * 128 * 4;
  static constexpr int FU0 = FMAP + 4 * 512;
  static constexpr int TOTAL = FU0 + 4 * 260;
  static constexpr int ALLOC = TOTAL + 1024;  // room to align the base to 1024 bytes
};
static_assert(SmemLayout::ALLOC <= 232448, "shared memory budget");

struct TcParams {
  CUtensorMap tmap_q;   // q as (head_dim, heads, tokens), boxes of 64 x G x 128 / G, 128-byte swizzle
  rc_extend_args a;
  int* status;
  int ppt;           // query positions per tile
  float scale2;      // sm_scale * log2(e)
  int pass;          // 0: one request per CTA z; 1: stacked prefix pass, one group per CTA z
  float* lse_part;   // [T, Hq] log2-sum-exp of the stacked pass's partial results
  int group_lo;      // stacked pass: group of CTA z = group_lo + z (one launch per level)
  int nlevels;       // levels of stacking groups (>= 1 when num_groups > 0)
  int level_lo[RC_MAX_STACK_LEVELS + 1];   // groups of level l: [level_lo[l], level_lo[l+1])
  uint64_t wait_limit_ns;   // bound of every wait except the final drain
};

// The group among groups [g0, g1) holding request b (ranges ascending and disjoint within a
// level), -1 if none.
__device__ __forceinline__ int group_index_of(const rc_extend_args& a, int b, int g0, int g1) {
  int lo = g0, hi = g1 - 1;
  while (lo <= hi) {
    const int mid = (lo + hi) >> 1;
    if (b < a.group_range[2 * mid]) hi = mid - 1;
    else if (b >= a.group_range[2 * mid + 1]) lo = mid + 1;
    else return mid;
  }
  return -1;
}

// The request among [b0, b1) whose new tokens hold stacked position pos (positions counted from
// qo_indptr[b0] = qo): the last one starting at or before pos.
__device__ __forceinline__ int request_of_pos(const rc_extend_args& a, int b0, int b1, int qo,
                                              int pos) {
  int lo = b0, hi = b1 - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (a.qo_indptr[mid] - qo <= pos) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}

// Folded stacked pass: member r of the group (new tokens at stacked positions [st, en) from
// the group's first) has priv = prefix_len[r] - P cached keys past the shared prefix P, then
// its new tokens. Its remainder keys in the CTA, in 128-key tiles: up to the key its last row
// before stacked position `end` sees.
__device__ __forceinline__ int fold_tiles(const rc_extend_args& a, int r, int qo, int P, int end) {
  const int st = a.qo_indptr[r] - qo, en = a.qo_indptr[r + 1] - qo;
  const int last = min(en, end) - 1 - st;   // member-relative index of its last row here
  return last < 0 ? 0 : (a.prefix_len[r] - P + last + 1 + kN - 1) / kN;
}

// ---------------------------------------------------------------- PTX wrappers
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_arrive_noinc(uint32_t bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}
// one box of a 3-D tensor map into shared memory, completing bytes on `bar`
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int x, int y,
                                            int z, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst), "l"(map), "r"(x), "r"(y), "r"(z), "r"(bar)
      : "memory");
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
// s0 += low bf16 of x, s1 += high bf16 of x (each widened exactly, one rounding in the add)
__device__ __forceinline__ void add_bf16x2(float& s0, float& s1, uint32_t x) {
  asm("{\n .reg .b16 lo, hi;\n mov.b32 {lo, hi}, %2;\n add.rn.f32.bf16 %0, lo, %0;\n"
      " add.rn.f32.bf16 %1, hi, %1;\n}" : "+f"(s0), "+f"(s1) : "r"(x));
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

// A descriptor advanced by `bytes` (a multiple of 16): only the 14-bit start-address field
// changes, and shared-memory addresses stay below 2^18, so the low word takes the add without a
// carry into the next field.
__device__ __forceinline__ uint64_t desc_add(uint64_t d, uint32_t bytes) {
  uint32_t lo, hi;
  asm("mov.b64 {%0, %1}, %2;" : "=r"(lo), "=r"(hi) : "l"(d));
  lo += bytes >> 4;
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "r"(lo), "r"(hi));
  return r;
}

// kind::f16 instruction descriptor: bf16 A and B, fp32 D, M = 128, N = 128
__host__ __device__ constexpr uint32_t idesc_bf16(bool b_mn_major) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((b_mn_major ? 1u : 0u) << 16) |
         ((uint32_t)(kN >> 3) << 17) | ((uint32_t)(kM >> 4) << 24);
}


// Eight K = 16 steps of one 128 x 128 x 128 product in one block, issued by the lane whose
// `leader` is non-zero (the warp runs the schedule converged; one thread issues). Each step
// advances the low descriptor words by a constant (no carry: see desc_add).
// Q K^T: A and B K-major SW128 tiles in shared memory; the steps of a 64-column block are
// 32 bytes apart, the blocks kBlockBytes apart. The first step overwrites D.
__device__ __forceinline__ void mma_qk8(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc,
                                        uint32_t leader) {
  asm volatile(
      "{\n .reg .pred e, pf, pt;\n .reg .b32 alo, ahi, blo, bhi, x, y;\n .reg .b64 ad, bd;\n"
      " setp.ne.b32 e, %4, 0;\n setp.ne.b32 pf, %4, %4;\n setp.eq.b32 pt, %4, %4;\n"
      " mov.b64 {alo, ahi}, %1;\n mov.b64 {blo, bhi}, %2;\n"
      " @e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, pf;\n"
#define RC_QK_STEP(OFF)                                                              \
      " add.u32 x, alo, " #OFF ";\n mov.b64 ad, {x, ahi};\n"                        \
      " add.u32 y, blo, " #OFF ";\n mov.b64 bd, {y, bhi};\n"                        \
      " @e tcgen05.mma.cta_group::1.kind::f16 [%0], ad, bd, %3, pt;\n"
      RC_QK_STEP(2) RC_QK_STEP(4) RC_QK_STEP(6) RC_QK_STEP(1024) RC_QK_STEP(1026)
      RC_QK_STEP(1028) RC_QK_STEP(1030)
#undef RC_QK_STEP
      "}\n" ::"r"(d), "l"(a), "l"(b), "r"(idesc), "r"(leader));
}
static_assert(kBlockBytes == 1024 * 16, "step offsets of mma_qk8 are in 16-byte units");
// P V: A = the weights in TMEM (keys 16 kk.. in columns 8 kk..), B = V MN-major in shared
// memory (16 key rows of 128 bytes = 2048 bytes = 128 descriptor units per step). The first step
// accumulates iff `accum`.
__device__ __forceinline__ void mma_pv8(uint32_t d, uint32_t a_tmem, uint64_t b, uint32_t idesc,
                                        uint32_t accum, uint32_t leader) {
  asm volatile(
      "{\n .reg .pred e, pf, pt;\n .reg .b32 blo, bhi, x, y;\n .reg .b64 bd;\n"
      " setp.ne.b32 e, %5, 0;\n setp.ne.b32 pf, %4, 0;\n setp.eq.b32 pt, %5, %5;\n"
      " mov.b64 {blo, bhi}, %2;\n"
      " @e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, pf;\n"
#define RC_PV_STEP(COL, OFF)                                                         \
      " add.u32 x, %1, " #COL ";\n add.u32 y, blo, " #OFF ";\n mov.b64 bd, {y, bhi};\n" \
      " @e tcgen05.mma.cta_group::1.kind::f16 [%0], [x], bd, %3, pt;\n"
      RC_PV_STEP(8, 128) RC_PV_STEP(16, 256) RC_PV_STEP(24, 384) RC_PV_STEP(32, 512)
      RC_PV_STEP(40, 640) RC_PV_STEP(48, 768) RC_PV_STEP(56, 896)
#undef RC_PV_STEP
      "}\n" ::"r"(d), "r"(a_tmem), "l"(b), "r"(idesc), "r"(accum), "r"(leader));
}
// tcgen05.commit from the issuing lane only
__device__ __forceinline__ void mma_commit_by(uint32_t bar, uint32_t leader) {
  asm volatile(
      "{\n .reg .pred e;\n setp.ne.b32 e, %1, 0;\n"
      " @e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n}" ::"r"(bar),
      "r"(leader)
      : "memory");
}


__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// Hardware named barriers (not shared memory): the weights hand-off from a softmax warpgroup
// to the MMA warp. A poll of an mbarrier by the MMA warp queues behind the tensor core's
// shared-memory operand reads; a named barrier does not.
constexpr int kHandoffBar0 = 1;                       // ids 1 (tile A) and 2 (tile B); 0 is __syncthreads
constexpr int kHandoffThreads = 128 + 32;             // a softmax warpgroup and the MMA warp
__device__ __forceinline__ void named_bar_arrive(int id, int count) {
  asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(count) : "memory");
}
__device__ __forceinline__ void named_bar_sync(int id, int count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
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
// 16 consecutive fp32 columns of this thread's TMEM lane
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float* v) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
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


// Ties 32 registers written by tcgen05.ld to a point after tcgen05.wait::ld, so that no use of
// them is scheduled before the wait.
__device__ __forceinline__ void reg_fence32(float* v) {
  asm volatile(""
               : "+f"(v[0]), "+f"(v[1]), "+f"(v[2]), "+f"(v[3]), "+f"(v[4]), "+f"(v[5]),
                 "+f"(v[6]), "+f"(v[7]), "+f"(v[8]), "+f"(v[9]), "+f"(v[10]), "+f"(v[11]),
                 "+f"(v[12]), "+f"(v[13]), "+f"(v[14]), "+f"(v[15]), "+f"(v[16]), "+f"(v[17]),
                 "+f"(v[18]), "+f"(v[19]), "+f"(v[20]), "+f"(v[21]), "+f"(v[22]), "+f"(v[23]),
                 "+f"(v[24]), "+f"(v[25]), "+f"(v[26]), "+f"(v[27]), "+f"(v[28]), "+f"(v[29]),
                 "+f"(v[30]), "+f"(v[31]));
}
__device__ __forceinline__ void reg_fence16(float* v) {
  asm volatile(""
               : "+f"(v[0]), "+f"(v[1]), "+f"(v[2]), "+f"(v[3]), "+f"(v[4]), "+f"(v[5]),
                 "+f"(v[6]), "+f"(v[7]), "+f"(v[8]), "+f"(v[9]), "+f"(v[10]), "+f"(v[11]),
                 "+f"(v[12]), "+f"(v[13]), "+f"(v[14]), "+f"(v[15]));
}
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}
__device__ __forceinline__ void tmem_st16u(uint32_t taddr, const uint32_t* v) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
      "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]),
      "r"(v[15])
      : "memory");
}

__device__ __forceinline__ bool mbar_test_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.test_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Wait for a phase for at most limit_ns (the launch's bound: 2 s, or a test hook's shorter
// one). On expiry: status code, false. done != nullptr: also give up (without a status code)
// once *done is set. A bound under 1 ms polls without suspending (test_wait): a suspended
// try_wait may sleep until the phase completes, which would hide a short bound.
__device__ __forceinline__ bool wait_lim(uint64_t* bar, uint32_t parity, int* status,
                                         uint64_t limit_ns, volatile int* done = nullptr) {
  const bool short_limit = limit_ns < 1000000;
  if (!short_limit && mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  while (!(short_limit ? mbar_test_wait(bar, parity) : mbar_try_wait(bar, parity))) {
    if (done && *done) return false;
    if (global_timer_ns() - t0 > limit_ns) {
      set_status(status, kStatusWaitExpired);
      return false;
    }
  }
  return true;
}

// ---------------------------------------------------------------- the kernel
template <bool kStack>
__global__ void __launch_bounds__(kThreads, 1) extend_tc_kernel(const __grid_constant__ TcParams p) {
  constexpr int kRegsControl = Regs<kStack>::control, kRegsSoftmax = Regs<kStack>::softmax;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // 128-byte swizzled operand tiles must start on 1024-byte boundaries
  uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  const rc_extend_args& a = p.a;
  const int hk = blockIdx.y;
  const int G = a.num_q_heads / a.num_kv_heads;
  const int iA = blockIdx.x * 2 * p.ppt;       // first query position of tile A
  // The CTA's rows and keys. Per-request pass: request b's new tokens against keys
  // [kstart, P) of its prefix -- kstart the shared length of its stacking group, 0 outside
  // groups -- and causally its own new tokens. Stacked pass: the new tokens of group g's
  // members, stacked in batch order, against keys [0, shared) only.
  const bool stacked = kStack && p.pass == 1;
  int b, qo, S, P, row, kstart = 0;
  // folded stacked pass: the CTA also takes each of its members' remainders -- a run of key
  // tiles per member, members r_first, r_first + 1, ... of the group [gb0, gb1) in order, n_rem
  // tiles in all, of which query tile A needs the first n_rem_a -- and is final
  bool fold = false;
  int gb0 = 0, gb1 = 0, r_first = 0, r_last = 0, n_rem = 0, n_rem_a = 0;
  if (stacked) {
    const int g = p.group_lo + blockIdx.z;
    const int b0 = a.group_range[2 * g], b1 = a.group_range[2 * g + 1];
    if (b0 < 0 || b1 <= b0 || b1 > a.num_reqs) {
      if (threadIdx.x == 0 && blockIdx.x == 0 && hk == 0) set_status(p.status, kStatusPosRange);
      return;
    }
    b = b0;
    qo = a.qo_indptr[b0];
    S = a.qo_indptr[b1] - qo;
    P = a.group_shared[g];
    row = a.req_idx[b0];
    fold = a.group_fold && a.group_fold[g];
    gb0 = b0;
    gb1 = b1;
    if (threadIdx.x == 0 && blockIdx.x == 0 && hk == 0) {
      for (int bb = b0; bb < b1; ++bb) {  // every member matched the shared prefix
        if (a.prefix_len[bb] < P) set_status(p.status, kStatusPosRange);
      }
    }
    if (S <= 0 || iA >= S) return;
    // a deeper level covers only the keys after its parent's shared prefix
    kstart = a.group_start ? a.group_start[g] : 0;
    if (fold) {
      const int endA = min(iA + p.ppt, S), endC = min(iA + 2 * p.ppt, S);
      r_first = request_of_pos(a, b0, b1, qo, iA);
      const int r_lastA = request_of_pos(a, b0, b1, qo, endA - 1);
      r_last = request_of_pos(a, b0, b1, qo, endC - 1);
      // query tile A needs the remainder tiles of its own members only, which come first (of
      // its last member, those up to its last row in A)
      for (int r = r_first; r <= r_last; ++r) {
        const int nt = fold_tiles(a, r, qo, P, endC);
        n_rem += nt;
        if (r < r_lastA) n_rem_a += nt;
        else if (r == r_lastA) n_rem_a += fold_tiles(a, r, qo, P, endA);
      }
      // the CTA's remainder-tile map must fit its shared-memory table (the host folds only
      // groups whose CTAs do)
      if (n_rem > kFoldTiles || r_last - r_first + 1 > kFoldMembers) {
        if (threadIdx.x == 0) set_status(p.status, kStatusPosRange);
        return;
      }
    }
    if (P < 1 || P > a.prefix_len[b0] || P > a.max_ctx || row < 0 || row >= a.max_reqs ||
        qo < 0 || (int64_t)qo + S > a.num_tokens || kstart < 0 || kstart >= P) {
      if (threadIdx.x == 0) set_status(p.status, kStatusPosRange);
      return;
    }
  } else {
    b = blockIdx.z;
    qo = a.qo_indptr[b];
    S = a.qo_indptr[b + 1] - qo;
    P = a.prefix_len[b];
    if (S <= 0 || iA >= S) return;
    row = a.req_idx[b];
    if (P < 0 || (int64_t)P + S > a.max_ctx || row < 0 || row >= a.max_reqs || qo < 0 ||
        (int64_t)qo + S > a.num_tokens) {
      if (threadIdx.x == 0) set_status(p.status, kStatusPosRange);
      return;
    }
    if (kStack && a.num_groups > 0) {
      int deepest = -1;
      for (int l = 0; l < p.nlevels; ++l) {   // the deepest group holding b shares the most
        const int gi = group_index_of(a, b, p.level_lo[l], p.level_lo[l + 1]);
        if (gi >= 0 && a.group_shared[gi] > kstart) {
          kstart = a.group_shared[gi];
          deepest = gi;
        }
      }
      // a folded group's stacked pass computed its members completely
      if (deepest >= 0 && a.group_fold && a.group_fold[deepest]) return;
      if (kstart < 0 || kstart > P) {
        if (threadIdx.x == 0) set_status(p.status, kStatusPosRange);
        kstart = 0;
      }
    }
  }
  // rows merged in the epilogue with the partial result the stacked passes before left: the
  // per-request pass after any group, a deeper level's stacked pass after its parent's
  const bool merge = kStack && kstart > 0;
  const int iB = iA + p.ppt;
  const int nposA = min(p.ppt, S - iA);
  const int nposB = max(0, min(p.ppt, S - iB));
  // TMEM lane of a query tile's first row: a tile of at most 96 rows starts at lane 32, so that
  // lane quadrant 0 holds no rows. Its softmax warps share a sub-partition with the MMA warp,
  // and a busy warp there slows the MMA warp's issue (measured: one tcgen05.mma per ~89 cycles
  // with idle neighbours, ~123 with one arithmetic-bound warp beside it, ~159 with two). The
  // Q box then starts 32 / G positions early, so G must divide 32.
  const bool can_shift = 32 % G == 0;
  const int shA = can_shift && nposA * G <= 96 ? 32 : 0;
  const int shB = can_shift && nposB * G <= 96 ? 32 : 0;
  const int n_pre = (P - kstart + kN - 1) / kN;     // prefix key tiles: keys [kstart, P)
  // key tiles of each query tile: the prefix, then (per-request pass) new-token keys up to its
  // last position
  const int nA = n_pre + (stacked ? n_rem_a : (iA + nposA + kN - 1) / kN);
  const int nB = nposB > 0 ? n_pre + (stacked ? n_rem : (iB + nposB + kN - 1) / kN) : 0;
  // the epilogue leaves a partial result (unfolded stacked pass) or the final one
  const bool partial = stacked && !fold;
  const int ntiles = max(nA, nB);
  const int kend = nposB > 0 ? iB + nposB : iA + nposA;  // new-token keys loaded: [0, kend)
  // virtual tiles: pair mode (query tiles A and B, every key tile each) or split mode (query
  // tile A only; key tile 2t + X is local tile t of virtual tile X)
  const bool split = nposB == 0 && nA >= 2;
  const int nt0 = split ? (nA + 1) / 2 : nA;
  const int nt1 = split ? nA / 2 : nB;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int Hq = a.num_q_heads, Hkv = a.num_kv_heads;
  (void)b;

  const uint32_t sbase = smem_u32(smem);
  const uint32_t sQ = sbase + SmemLayout::Q;
  const uint32_t sK = sbase + SmemLayout::K;
  const uint32_t sV = sbase + SmemLayout::V;
  uint64_t* bars = (uint64_t*)(smem + SmemLayout::BAR);
  uint64_t* k_full = bars;                      // [stage]
  uint64_t* k_empty = k_full + kStagesKV;       // [stage]
  uint64_t* v_full = k_empty + kStagesKV;       // [stage]
  uint64_t* v_empty = v_full + kStagesKV;       // [stage]
  uint64_t* s_full = v_empty + kStagesKV;       // [tile]
  uint64_t* o_done = s_full + 4;                // [tile]
  uint64_t* e_done = o_done + 2;                // split-mode merge
  uint64_t* q_full = e_done + 1;                // both Q tiles in shared memory
  uint64_t* drain = q_full + 1;                 // every issued MMA has completed
  static_assert(4 * kStagesKV + 9 == SmemLayout::NBAR, "barrier count");
  uint32_t* tmem_slot = (uint32_t*)(smem + SmemLayout::TMEM_SLOT);
  volatile int* mma_done = (volatile int*)(smem + SmemLayout::MMA_DONE);
  const uint64_t lim = p.wait_limit_ns;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStagesKV; ++s) {
      mbar_init(&k_full[s], 32 * kProdWarps);
      mbar_init(&k_empty[s], 1);
      mbar_init(&v_full[s], 32 * kProdWarps);
      mbar_init(&v_empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&s_full[s], 1);
      mbar_init(&o_done[s], 1);
    }
    mbar_init(e_done, 2 * kGroupThreads);
    mbar_init(q_full, 1);
    mbar_init(drain, 1);
    *mma_done = 0;
    fence_mbar_init();
    // Q tiles: smem row (= TMEM lane) m of tile X holds position iX + (m - shX) / G, head
    // hk * G + m % G -- one TMA box of 128 / G positions x G heads per 64-column block, starting
    // shX / G positions early. Rows outside the tile hold other tokens' queries, or zeros past
    // either end of the batch; their results are never stored. The MMA warp waits on q_full.
    const int nq = nposB > 0 ? 2 : 1;
    mbar_arrive_expect_tx(q_full, nq * (kM / G) * G * kD * 2);
    for (int X = 0; X < nq; ++X) {
      const int z = qo + (X ? iB : iA) - (X ? shB : shA) / G;
      for (int blk = 0; blk < 2; ++blk)
        tma_load_3d(sQ + X * kTileBytes + blk * kBlockBytes, &p.tmap_q, blk * 64, hk * G, z,
                    smem_u32(q_full));
    }
  }
  if (warp == kMmaWarp) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;" ::"r"(
                     smem_u32(tmem_slot))
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  // ---- producer state (warps 1-4). Producer w of an operand fills tile rows [64 w, 64 w + 64):
  // lane l resolves rows 64 w + l and 64 w + 32 + l to a row pointer; one copy instruction then
  // moves 16-byte chunk (l & 15) of two rows, the row pointer taken from its owner lane by a
  // shuffle.
  const bool producer = warp >= kKWarp0 && warp < kScatterWarp0;
  const int32_t* rt = a.req_to_token + (int64_t)row * a.max_ctx;
  const bool is_v = warp >= kVWarp0;
  const int w = warp - (is_v ? kVWarp0 : kKWarp0);
  constexpr int kRowsPerWarp = kN / kProdWarps;
  constexpr int kGroups = kRowsPerWarp / 32;
  static_assert(kGroups == 2, "two 32-row groups per producer warp");
  const __nv_bfloat16* pool = (const __nv_bfloat16*)(is_v ? a.v_pool : a.k_pool);
  const __nv_bfloat16* nsrc = (const __nv_bfloat16*)(is_v ? a.v_new : a.k_new);
  uint64_t* full = is_v ? v_full : k_full;
  uint64_t* empty = is_v ? v_empty : k_empty;
  const int c = lane & 15, half = lane >> 4;
  // destination of row 2 i + half (i = 0..15) of a 32-row group, chunk c: the swizzle term
  // repeats every four values of i; the row term adds 1024 bytes per four
  uint32_t d4[4];
#pragma unroll
  for (int m = 0; m < 4; ++m) d4[m] = sw128_off(2 * m + half, c);
  const uint32_t sbuf = (is_v ? sV : sK) + (uint32_t)(w * kRowsPerWarp * 128);
  // raw(j, q) only issues the slot load; rowptr() checks it when the tile is issued, so the
  // loads of tile j+1 stay in flight while tile j is being copied
  // folded remainder tile j >= n_pre: tile qt of member r (the CTA's map, filled before the
  // set-up barrier); the member's key k = 128 qt + row is its own cached token P + k while
  // k < priv (= its prefix past the shared P), then its new token k - priv
  const int endC = min(iA + 2 * p.ppt, S);
  const uint32_t* fmap = (const uint32_t*)(smem + SmemLayout::FMAP);
  const int* fu0 = (const int*)(smem + SmemLayout::FU0);
  auto fold_tile = [&](int j, int& qt) -> int {
    const uint32_t e = fmap[min(max(j - n_pre, 0), kFoldTiles - 1)];
    qt = (int)(e & 0xFFFFu);
    return min(r_first + (int)(e >> 16), gb1 - 1);
  };
  auto raw = [&](int j, int q) -> int {
    if (j < n_pre) {
      const int key = kstart + j * kN + w * kRowsPerWarp + q * 32 + lane;
      return rt[key < P ? key : P - 1];
    }
    if (fold) {
      int qt;
      const int r = fold_tile(j, qt);
      const int k = qt * kN + w * kRowsPerWarp + q * 32 + lane;
      const int rr = a.req_idx[r];
      if (k < a.prefix_len[r] - P && rr >= 0 && rr < a.max_reqs && P + k < a.max_ctx)
        return a.req_to_token[(int64_t)rr * a.max_ctx + P + k];
      return -1;   // a new token (or padding): resolved by rowptr
    }
    return 0;
  };
  auto rowptr = [&](int j, int q, int rv) -> const __nv_bfloat16* {
    if (fold && j >= n_pre) {
      int qt;
      const int r = fold_tile(j, qt);
      const int k = qt * kN + w * kRowsPerWarp + q * 32 + lane;
      const int priv = a.prefix_len[r] - P;
      if (k < priv) {
        int sl = rv;
        if (sl < 0 || (int64_t)sl >= a.num_slots) {
          set_status(p.status, kStatusSlotRange);
          sl = 0;
        }
        return pool + ((int64_t)sl * Hkv + hk) * kD;
      }
      // new token k - priv of member r (past its last: its last, masked anyway)
      const int q0 = a.qo_indptr[r], nr = a.qo_indptr[r + 1] - q0;
      const int tok = min(max(q0 + min(k - priv, nr - 1), 0), (int)a.num_tokens - 1);
      return nsrc + ((int64_t)tok * Hkv + hk) * kD;
    }
    if (j < n_pre) {
      int sl = rv;
      if (sl < 0 || (int64_t)sl >= a.num_slots) {
        set_status(p.status, kStatusSlotRange);
        sl = 0;
      }
      return pool + ((int64_t)sl * Hkv + hk) * kD;
    }
    const int s0 = (j - n_pre) * kN + w * kRowsPerWarp + q * 32 + lane;
    return nsrc + ((int64_t)(qo + min(s0, kend - 1)) * Hkv + hk) * kD;
  };
  auto copy_tile = [&](int j, const __nv_bfloat16* p0, const __nv_bfloat16* p1) {
    const uint32_t dst = sbuf + (j % kStagesKV) * kTileBytes;
#pragma unroll
    for (int q = 0; q < kGroups; ++q) {
      const uint64_t rp = (uint64_t)(q == 0 ? p0 : p1);
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const __nv_bfloat16* src =
            (const __nv_bfloat16*)__shfl_sync(0xffffffffu, rp, 2 * i + half) + c * 8;
        cp_async16(dst + q * 32 * 128 + (i >> 2) * 1024 + d4[i & 3], src);
      }
    }
  };
  // stage 0 is free at the start: the first key tile's copies go out before the setup barrier
  if (producer && ntiles > 0) copy_tile(0, rowptr(0, 0, raw(0, 0)), rowptr(0, 1, raw(0, 1)));

  // the folded pass's remainder-tile map: one thread walks the CTA's members (its loads overlap
  // the other threads' first copies)
  if (fold && threadIdx.x == kThreads - 1) {
    uint32_t* map = (uint32_t*)(smem + SmemLayout::FMAP);
    int* u0 = (int*)(smem + SmemLayout::FU0);
    int u = 0;
    for (int r = r_first; r <= r_last; ++r) {
      u0[r - r_first] = u;
      const int nt = fold_tiles(a, r, qo, P, endC);
      for (int qt = 0; qt < nt; ++qt) map[u++] = ((uint32_t)(r - r_first) << 16) | (uint32_t)qt;
    }
  }
  tc_fence_before();
  __syncthreads();   // barrier initialisation and the TMEM address are visible from here
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // register split (each role branch starts with its setmaxnreg, so that its code is compiled
  // for its own budget): launched with kRegsLaunch per thread; the control warpgroup (warps 0-3)
  // gives registers up, the two softmax warpgroups take them
  if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsControl));
    // The warp runs the whole schedule converged (waits, fences); lane 0 alone issues the MMAs
    // and the commits that track them.
    {
      const uint32_t leader = lane == 0;
      const uint32_t idq = idesc_bf16(false), idv = idesc_bf16(true);
      // base descriptors (Q tile A, K stage 0, V stage 0), built once
      const uint64_t dq0 = smem_desc_sw128(sQ, 16, 1024);
      const uint64_t dk0 = smem_desc_sw128(sK, 16, 1024);
      const uint64_t dv0 = smem_desc_sw128(sV, kBlockBytes, 1024);
      // local tile t of virtual tile X reads key tile kt; in pair mode key tile j is read first
      // by tile A (if j < nA) and last by tile B (if j < nB), in split mode by one virtual tile
      auto kt_of = [&](int X, int t) { return split ? 2 * t + X : t; };
      auto qk = [&](int X, int t) -> bool {
        const int kt = kt_of(X, t), st = kt % kStagesKV;
        const bool first = split || X == 0 || kt >= nA;
        const bool last = split || X == 1 || kt >= nB;
        if (first) {
          if (!wait_lim(&k_full[st], (kt / kStagesKV) & 1, p.status, lim)) return false;
          // K arrived through the generic proxy (cp.async); one fence covers every later
          // MMA issued on the stage
          fence_async_smem();
        }
        tc_fence_after();
        mma_qk8(tmem + X * 128, desc_add(dq0, (split ? 0 : X) * kTileBytes),
                desc_add(dk0, st * kTileBytes), idq, leader);
        mma_commit_by(smem_u32(&s_full[X]), leader);
        if (last) mma_commit_by(smem_u32(&k_empty[st]), leader);
        return true;
      };
      auto pv = [&](int X, int t) -> bool {
        const int kt = kt_of(X, t), st = kt % kStagesKV;
        // the weights P of tile X: every softmax thread of the tile arrives once per local tile,
        // also after a wait of its own gave up, so this sync always completes
        named_bar_sync(kHandoffBar0 + X, kHandoffThreads);
        const bool first = split || X == 0 || kt >= nA;
        const bool last = split || X == 1 || kt >= nB;
        if (first) {
          if (!wait_lim(&v_full[st], (kt / kStagesKV) & 1, p.status, lim)) return false;
          fence_async_smem();   // V arrived through the generic proxy (cp.async)
        }
        tc_fence_after();
        mma_pv8(tmem + 256 + X * 128, tmem + X * 128, desc_add(dv0, st * kTileBytes), idv,
                t > 0 ? 1u : 0u, leader);
        if (t == (X ? nt1 : nt0) - 1) mma_commit_by(smem_u32(&o_done[X]), leader);
        if (last) mma_commit_by(smem_u32(&v_empty[st]), leader);
        return true;
      };
      bool ok = wait_lim(q_full, 0, p.status, lim);   // Q by TMA: the async proxy already
      if (ok) ok = qk(0, 0);
      if (ok && nt1 > 0) ok = qk(1, 0);
      for (int t = 0; t < max(nt0, nt1) && ok; ++t) {
        if (t < nt0) {
          ok = pv(0, t);
          if (ok && t + 1 < nt0) ok = qk(0, t + 1);
        }
        if (ok && t < nt1) {
          ok = pv(1, t);
          if (ok && t + 1 < nt1) ok = qk(1, t + 1);
        }
      }
      // no weights sync follows: a softmax group shadowing this warp may stop
      if (leader) *mma_done = 1;
      // every MMA issued above completes before TMEM is freed, also when a wait gave up early
      // (this wait keeps the full bound whatever the launch's: it guards the deallocation)
      mma_commit_by(smem_u32(drain), leader);
      mbar_wait(drain, 0, p.status);
      // the Q boxes have landed before the CTA exits, also when the wait above for them gave up
      mbar_wait(q_full, 0, p.status);
    }
    __syncwarp();
  } else if (warp < kScatterWarp0) {
    // ------------------------------------------------------------ producers (K: warps 1-2, V: 3-4)
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsControl));
    // tile 0 was issued before the barrier; its arrival can only follow the barrier
    // initialisation
    bool ok = true;
    if (ntiles > 0) cp_async_arrive_noinc(smem_u32(&full[0]));
    int n0 = ntiles > 1 ? raw(1, 0) : 0, n1 = ntiles > 1 ? raw(1, 1) : 0;
    for (int j = 1; j < ntiles && ok; ++j) {
      const int st = j % kStagesKV;
      const __nv_bfloat16* p0 = rowptr(j, 0, n0);
      const __nv_bfloat16* p1 = rowptr(j, 1, n1);
      if (j + 1 < ntiles) {
        n0 = raw(j + 1, 0);
        n1 = raw(j + 1, 1);
      }
      if (j >= kStagesKV) ok = wait_lim(&empty[st], ((j / kStagesKV) - 1) & 1, p.status, lim);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      copy_tile(j, p0, p1);
      cp_async_arrive_noinc(smem_u32(&full[st]));
    }
    asm volatile("cp.async.wait_all;" ::: "memory");
  } else if (warp < kSoftmaxWarp0) {
    // ------------------------------------------------------------ scatter of the new K/V rows
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsControl));
    // (row, 16-byte chunk) pairs of both query tiles' positions; each round issues all of a
    // lane's loads before any store, four copies in flight per lane.
    const __nv_bfloat16* kn = (const __nv_bfloat16*)a.k_new;
    const __nv_bfloat16* vn = (const __nv_bfloat16*)a.v_new;
    constexpr int kU = 4;
    // an unfolded stacked pass writes no K/V (each member's own pass does)
    const int total = partial ? 0 : (nposA + nposB) * 16;
    for (int base = (warp - kScatterWarp0) * 32 + lane; base < total; base += 32 * kScatterWarps * kU) {
      uint4 kv[kU], vv[kU];
      int64_t dst[kU];
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const int e = base + u * 32 * kScatterWarps;
        dst[u] = -1;
        if (e < total) {
          const int i = iA + (e >> 4), cc = e & 15;
          const int64_t tok = qo + i;
          const int sl = a.out_loc[tok];
          const int64_t src = (tok * Hkv + hk) * kD + cc * 8;
          kv[u] = *(const uint4*)(kn + src);
          vv[u] = *(const uint4*)(vn + src);
          if (sl >= 0 && (int64_t)sl < a.num_slots)
            dst[u] = ((int64_t)sl * Hkv + hk) * kD + cc * 8;
          else if (cc == 0)
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
    // ------------------------------------------------------------ softmax groups
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsSoftmax));
    const int X = (warp - kSoftmaxWarp0) >> 2;        // query tile (virtual tile in split mode)
    const int quad = warp & 3;                        // TMEM lane quadrant of this warp
    const int r = quad * 32 + lane;                   // query row = TMEM lane
    const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
    const int nX = X ? nt1 : nt0;
    const int iX = (X && !split) ? iB : iA;
    const int rows_used = ((X && !split) ? nposB : nposA) * G;
    const int mrow = r - ((X && !split) ? shB : shA);  // tile row of this lane (< 0: none)
    const bool row_valid = mrow >= 0 && mrow < rows_used;
    // a warp with no row of the tile only paces the weights hand-off
    const bool warp_idle = !__any_sync(0xffffffffu, row_valid);
    const int ipos = min(iX + max(mrow, 0) / G, S - 1);  // this row's new-token index (clamped)
    // folded stacked pass: the member this row belongs to, its index among that member's new
    // tokens, the remainder keys it sees (its member's cached keys past P, then its new tokens up
    // to its own), and where its member's remainder tiles start in the CTA's list (u0_row)
    int req_row = -1, row_keys = 0, u0_row = 0;
    if (fold) {
      req_row = request_of_pos(a, gb0, gb1, qo, ipos);
      row_keys = a.prefix_len[req_row] - P + ipos - (a.qo_indptr[req_row] - qo) + 1;
      u0_row = fu0[min(max(req_row - r_first, 0), kFoldMembers - 1)];
    }
    const float sc2 = p.scale2;
    const uint64_t sc2x2 = f2pack(sc2, sc2);
    const uint32_t tS = tmem + X * 128 + lane_off;
    const uint32_t tO = tmem + 256 + X * 128 + lane_off;
    float m_run = -INFINITY, l_run = 0.f, l_exact = 0.f;
    bool ok = true;
    int j = 0;
    for (; j < nX; ++j) {
      ok = wait_lim(&s_full[X], j & 1, p.status, lim);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      if (warp_idle) {
        // arriving only after this tile's scores exist keeps every arrival in the generation
        // the MMA warp syncs on next
        named_bar_arrive(kHandoffBar0 + X, kHandoffThreads);
        continue;
      }
      tc_fence_after();
      // keys [0, lim) of key tile kt are visible to this row (lim <= 0: none)
      const int kt = split ? 2 * j + X : j;
      int lim;
      if (kt < n_pre) {
        lim = min(kN, P - kstart - kt * kN);
      } else if (fold) {
        // remainder tiles of other members are invisible to this row
        const int qt = kt - n_pre - u0_row;
        lim = qt < 0 ? 0 : min(kN, row_keys - qt * kN);
      } else {
        lim = min(kN, ipos - (kt - n_pre) * kN + 1);
      }
      float v[kN];
#pragma unroll
      for (int c = 0; c < kN / 32; ++c) tmem_ld32(tS + c * 32, v + c * 32);
      tmem_wait_ld();
#pragma unroll
      for (int c = 0; c < kN / 32; ++c) reg_fence32(v + c * 32);
      if (!__all_sync(0xffffffffu, lim >= kN)) {
#pragma unroll
        for (int u = 0; u < kN; ++u) v[u] = u < lim ? v[u] : -INFINITY;
      }
      // row max of the raw scores: four running three-input maxima
      float m4[4] = {fmaxf(v[0], v[1]), fmaxf(v[2], v[3]), fmaxf(v[4], v[5]), fmaxf(v[6], v[7])};
#pragma unroll
      for (int u = 8; u < kN; u += 8) {
#pragma unroll
        for (int k = 0; k < 4; ++k) m4[k] = fmax3(m4[k], v[u + 2 * k], v[u + 2 * k + 1]);
      }
      const float mx = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
      const float mt = mx * sc2;                   // sc2 > 0: max commutes with the scale
      const float m_new = fmaxf(m_run, mt);
      const bool rescale = m_new > m_run + kRescaleThreshold;  // also true for the first tile
      const float m_use = rescale ? m_new : m_run;
      const float alpha = (rescale && m_run != -INFINITY) ? ex2(m_run - m_new) : 1.f;
      // a row with no visible key so far keeps m = -inf; subtract 0 so masked scores give 0
      const float m_sub = m_use == -INFINITY ? 0.f : m_use;
      const uint64_t negx2 = f2pack(-m_sub, -m_sub);
      // weights, rounded to bf16, two per column in the first 64 score columns (kept in pk for
      // the rounded sum after the hand-off); the exact sum in packed (even, odd) form, two chains
      uint32_t pk[kN / 2];
      uint64_t re2[2] = {0, 0};
#pragma unroll
      for (int h = 0; h < kN / 32; ++h) {
#pragma unroll
        for (int u = 0; u < 16; ++u) {
          float x0, x1;
          f2unpack(fma2(f2pack(v[32 * h + 2 * u], v[32 * h + 2 * u + 1]), sc2x2, negx2), x0, x1);
          const float p0 = ex2(x0), p1 = ex2(x1);
          pk[16 * h + u] = pack_bf16(p0, p1);
          re2[u & 1] = add2(re2[u & 1], f2pack(p0, p1));
        }
        tmem_st16u(tS + 16 * h, pk + 16 * h);
      }
      // rescale O: the last P.V of this tile completed before these scores did
      // (16 columns at a time: the rounded weights stay live in registers until the hand-off)
      if (__any_sync(0xffffffffu, rescale && m_run != -INFINITY) && j > 0) {
#pragma unroll 1
        for (int c = 0; c < kD / 16; ++c) {
          float o[16];
          tmem_ld16(tO + c * 16, o);
          tmem_wait_ld();
          reg_fence16(o);
          uint32_t ou[16];
#pragma unroll
          for (int u = 0; u < 16; ++u) ou[u] = __float_as_uint(o[u] * alpha);
          tmem_st16u(tO + c * 16, ou);
        }
      }
      tmem_wait_st();
      tc_fence_before();
      named_bar_arrive(kHandoffBar0 + X, kHandoffThreads);
      // The rounded sum is not needed for the hand-off: it runs while the tensor core does P.V.
      // O is normalised by the sum of the rounded weights P.V uses; the log-sum-exp output
      // uses the exact sum. Each rounded weight enters the sum through one f32 + bf16 add (four
      // chains), without unpacking it first.
      float rs[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int u = 0; u < kN / 2; ++u) add_bf16x2(rs[2 * (u & 1)], rs[2 * (u & 1) + 1], pk[u]);
      float b0, b1;
      f2unpack(add2(re2[0], re2[1]), b0, b1);
      l_run = l_run * alpha + ((rs[0] + rs[1]) + (rs[2] + rs[3]));
      l_exact = l_exact * alpha + (b0 + b1);
      m_run = m_use;
    }
    // A wait that gave up ends the loop early (the status word records the failure; the
    // outputs are not valid). The MMA warp's weights syncs cannot time out, so the group keeps
    // answering them: one arrival for each further Q.K^T of its tile the MMA warp completes (an
    // arrival thus never runs ahead of the sync it answers), until the MMA warp has left its
    // schedule (mma_done); the bound is a backstop beyond any wait of the MMA warp.
    const uint64_t shadow_lim = 8 * lim + 1000000000ull;
    for (; j < nX; ++j) {
      if (!__all_sync(0xffffffffu, wait_lim(&s_full[X], j & 1, p.status, shadow_lim, mma_done)))
        break;
      named_bar_arrive(kHandoffBar0 + X, kHandoffThreads);
    }
    // The row's result over this pass's keys is (O, lse2): O the accumulator(s) times `scale`,
    // lse2 its log2-sum-exp. The stacked pass stores it as a partial (O in o, lse2 in the
    // workspace); a group member's per-request pass merges it with that partial, weights
    // 2^(lse2 - M) and 2^(lse_p - M); every other row is final as it is.
    auto combine = [&](int64_t rowidx, float lse2, float& fs, float& fp, float& lse_out) {
      fs = 1.f;
      fp = 0.f;
      lse_out = lse2;
      if (merge) {
        const float lp = p.lse_part[rowidx];
        const float M = fmaxf(lse2, lp);
        const float es = ex2(lse2 - M), ep = ex2(lp - M);
        const float inv = 1.f / (es + ep);
        fs = es * inv;
        fp = ep * inv;
        lse_out = M + log2f(es + ep);
      }
    };
    // 8 output columns: acc * scale (+ fp * the partial already in o) -> bf16
    auto store8 = [&](__nv_bfloat16* dst, const float* acc, float scale, float fp) {
      float v8[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) v8[k] = acc[k] * scale;
      if (merge) {
        const uint4 old = *(const uint4*)dst;
        v8[0] += fp * bf16lo(old.x); v8[1] += fp * bf16hi(old.x);
        v8[2] += fp * bf16lo(old.y); v8[3] += fp * bf16hi(old.y);
        v8[4] += fp * bf16lo(old.z); v8[5] += fp * bf16hi(old.z);
        v8[6] += fp * bf16lo(old.w); v8[7] += fp * bf16hi(old.w);
      }
      *(uint4*)dst = make_uint4(pack_bf16(v8[0], v8[1]), pack_bf16(v8[2], v8[3]),
                                pack_bf16(v8[4], v8[5]), pack_bf16(v8[6], v8[7]));
    };
    if (nX > 0 && !split) {
      // epilogue: O / l for this thread's row
      if (ok) ok = __all_sync(0xffffffffu, wait_lim(&o_done[X], 0, p.status, lim));
      if (ok) {
        tc_fence_after();
        const bool store = row_valid;
        const int i = iX + max(mrow, 0) / G, hh = max(mrow, 0) % G;
        const int64_t rowidx = (int64_t)(qo + i) * Hq + hk * G + hh;
        __nv_bfloat16* orow = (__nv_bfloat16*)a.o + rowidx * kD;
        const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
        float fs = 1.f, fp = 0.f, lse2 = m_run + log2f(l_exact);
        if (store) combine(rowidx, lse2, fs, fp, lse2);
#pragma unroll 1
        for (int c = 0; c < kD / 32; ++c) {
          float o[32];
          tmem_ld32(tO + c * 32, o);
          tmem_wait_ld();
          reg_fence32(o);
          if (store) {
#pragma unroll
            for (int u = 0; u < 32; u += 8) store8(orow + c * 32 + u, o + u, inv * fs, fp);
          }
        }
        if (store) {
          if (partial) p.lse_part[rowidx] = lse2;
          else if (a.lse) a.lse[rowidx] = lse2 * kLn2;
        }
      }
    } else if (split) {
      // merge the two virtual tiles: every softmax thread publishes its row max and sums;
      // thread (X, row) then writes columns [64 X, 64 X + 64) of the merged row
      if (ok) ok = __all_sync(0xffffffffu, wait_lim(&o_done[X], 0, p.status, lim));
      float* xm = (float*)(smem + SmemLayout::XMRG);     // [X][row] maxima
      float* xl = xm + 2 * 128;                          // [X][row] rounded-weight sums
      float* xe = xl + 2 * 128;                          // [X][row] exact sums
      xm[X * 128 + r] = m_run;
      xl[X * 128 + r] = l_run;
      xe[X * 128 + r] = l_exact;
      mbar_arrive(e_done);
      if (ok) ok = __all_sync(0xffffffffu, wait_lim(e_done, 0, p.status, lim));
      if (ok) {
        const float m0 = xm[r], m1 = xm[128 + r];
        const float M = fmaxf(m0, m1);
        const float w0 = m0 == -INFINITY ? 0.f : ex2(m0 - M);
        const float w1 = m1 == -INFINITY ? 0.f : ex2(m1 - M);
        const float lt = w0 * xl[r] + w1 * xl[128 + r];
        const float inv = lt > 0.f ? 1.f / lt : 0.f;
        tc_fence_after();
        const bool store = row_valid;
        const int i = iA + max(mrow, 0) / G, hh = max(mrow, 0) % G;
        const int64_t rowidx = (int64_t)(qo + i) * Hq + hk * G + hh;
        __nv_bfloat16* orow = (__nv_bfloat16*)a.o + rowidx * kD;
        float fs = 1.f, fp = 0.f, lse2 = M + log2f(w0 * xe[r] + w1 * xe[128 + r]);
        if (store) combine(rowidx, lse2, fs, fp, lse2);
        const float a0 = w0 * inv * fs, a1 = w1 * inv * fs;
#pragma unroll 1
        for (int c = 0; c < 2; ++c) {
          const int col = 64 * X + 32 * c;
          float o0[32], o1[32];
          tmem_ld32(tmem + 256 + lane_off + col, o0);
          tmem_ld32(tmem + 384 + lane_off + col, o1);
          tmem_wait_ld();
          reg_fence32(o0);
          reg_fence32(o1);
          if (store) {
#pragma unroll
            for (int u = 0; u < 32; u += 8) {
              float v8[8];
#pragma unroll
              for (int k = 0; k < 8; ++k) v8[k] = o0[u + k] * a0 + o1[u + k] * a1;
              store8(orow + col + u, v8, 1.f, fp);
            }
          }
        }
        if (store && X == 0) {
          if (partial) p.lse_part[rowidx] = lse2;
          else if (a.lse) a.lse[rowidx] = lse2 * kLn2;
        }
      }
    }
  }
  // every tcgen05 op has completed once the softmax observed o_done of both tiles; free TMEM
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;" ::"r"(tmem) : "memory");
  }
}

}  // namespace

// The driver's tensor-map encoder, looked up once per process through the runtime.
static PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static const PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      f = nullptr;
    return (PFN_cuTensorMapEncodeTiled_v12000)f;
  }();
  return fn;
}

int launch_extend_tc(const rc_extend_args* a, int* status, cudaStream_t s) {
  if (a->head_dim != kD) return fail(RC_ERR_INVALID, "extend (tensor cores): head_dim must be 128");
  const int G = a->num_q_heads / a->num_kv_heads;
  if (G > kM) return fail(RC_ERR_INVALID, "extend (tensor cores): group size %d > 128", G);
  if (((uintptr_t)a->q & 15) != 0)
    return fail(RC_ERR_INVALID, "extend (tensor cores): q must be 16-byte aligned");
  // per instantiation and device: opt in to the shared memory, and check that the launch
  // allocation covers the register split (the softmax warpgroups' setmaxnreg.inc would never
  // return)
  struct Setup {
    int regs[2] = {0, 0};
  };
  static PerDevice<Setup> setup;
  const Setup* su = nullptr;
  const cudaError_t err = setup.get(
      [](Setup& st) {
        int i = 0;
        for (const void* kern : {(const void*)extend_tc_kernel<false>,
                                 (const void*)extend_tc_kernel<true>}) {
          cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               SmemLayout::ALLOC);
          cudaFuncAttributes fa;
          if (e == cudaSuccess) e = cudaFuncGetAttributes(&fa, kern);
          if (e != cudaSuccess) return e;
          st.regs[i++] = fa.numRegs;
        }
        return cudaSuccess;
      },
      &su);
  if (err != cudaSuccess)
    return fail(RC_ERR_CUDA, "extend (tensor cores): %s", cudaGetErrorString(err));
  for (int regs : su->regs)
    if (regs < kRegsLaunch)
      return fail(RC_ERR_CUDA, "extend (tensor cores): kernel built with %d registers per "
                  "thread, the register split needs %d", regs, kRegsLaunch);
  TcParams p;
  // q [T, Hq, 128] bf16 as a 3-D tensor (columns, heads, tokens); one box is the 64-column block
  // of 128 / G positions x the G heads of a query tile
  const PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
  if (!encode) return fail(RC_ERR_CUDA, "extend (tensor cores): no tensor-map encoder in the driver");
  {
    const cuuint64_t dims[3] = {(cuuint64_t)kD, (cuuint64_t)a->num_q_heads,
                                (cuuint64_t)(a->num_tokens > 0 ? a->num_tokens : 1)};
    const cuuint64_t strides[2] = {(cuuint64_t)kD * 2, (cuuint64_t)a->num_q_heads * kD * 2};
    const cuuint32_t box[3] = {64, (cuuint32_t)G, (cuuint32_t)(kM / G)};
    const cuuint32_t elem[3] = {1, 1, 1};
    const CUresult r = encode(&p.tmap_q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(a->q),
                              dims, strides, box, elem, CU_TENSOR_MAP_INTERLEAVE_NONE,
                              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
      return fail(RC_ERR_CUDA, "extend (tensor cores): tensor map for q (error %d)", (int)r);
  }
  p.a = *a;
  p.status = status;
  p.ppt = kM / G;
  p.scale2 = a->sm_scale * kLog2e;
  p.lse_part = (float*)a->workspace;
  p.wait_limit_ns = wait_limit_ns();
  int launches = 0;
  p.group_lo = 0;
  p.nlevels = a->num_levels > 1 ? a->num_levels : 1;
  p.level_lo[0] = 0;
  p.level_lo[1] = a->num_groups;
  if (a->num_levels > 1)
    for (int l = 0; l <= a->num_levels; ++l) p.level_lo[l] = a->level_indptr[l];
  if (a->num_groups > 0) {
    // stacked prefix passes first, level by level: every member's partial result over the keys
    // above is in place before the next level (or the per-request pass) merges into it (same
    // stream)
    p.pass = 1;
    for (int l = 0; l < p.nlevels; ++l) {
      p.group_lo = p.level_lo[l];
      dim3 g1((a->max_group_rows + 2 * p.ppt - 1) / (2 * p.ppt), a->num_kv_heads,
              p.level_lo[l + 1] - p.level_lo[l]);
      extend_tc_kernel<true><<<g1, kThreads, SmemLayout::ALLOC, s>>>(p);
      ++launches;
    }
  }
  p.pass = 0;
  dim3 grid((a->max_q_len + 2 * p.ppt - 1) / (2 * p.ppt), a->num_kv_heads, a->num_reqs);
  if (a->num_groups > 0 && a->skip_request_pass) {
    // every request is in a folded group: the stacked passes computed everything
  } else if (a->num_groups > 0) {
    extend_tc_kernel<true><<<grid, kThreads, SmemLayout::ALLOC, s>>>(p);
    ++launches;
  } else {
    extend_tc_kernel<false><<<grid, kThreads, SmemLayout::ALLOC, s>>>(p);
    ++launches;
  }
  count_launches(launches);
  return check_launch("rc_extend_attention (tensor cores)");
}

}  // namespace rc
