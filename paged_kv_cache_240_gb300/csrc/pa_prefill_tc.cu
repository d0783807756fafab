// pa_prefill_tc.cu -- chunked-prefill attention on the 5th-generation tensor
// cores (tcgen05.mma, accumulators in tensor memory) for fp16/bf16 caches
// ("PyTorch LLM Serving Engine", "What is implemented": chunked prefill; "Loading":
// online softmax while walking the block table).
//
// A work item is 256 query rows (two tiles of 128) of one sequence's chunk and
// one kv head: row R = c*G + j is query token c, query head kvh*G + j.  The keys
// the rows can see are walked in tiles of 128 (eight 16-token blocks), each tile
// used by both query tiles:
//   S_q = Q_q K_t^T   tcgen05.mma M=128 N=128 K=head_dim, A and B in shared memory
//   P_q = exp2(S_q*scale - m)   one softmax thread per row; P (f16/bf16) is written
//                     back into the first 64 columns of S_q's tensor memory
//   O_q += P_q V_t    tcgen05.mma M=128 N=head_dim K=128, A = P from tensor memory
// Tensor memory (512 columns): per query tile S_q (128) and O_q (128).  Keeping P
// in tensor memory and taking 128 keys per S MMA halves the shared-memory traffic
// per key of a 64-key tile with P in shared memory; shared-memory bandwidth, not
// the tensor core, bounded that design.
//
// Warps: warpgroup 0 = warp 0 the Q and K producer, warp 3 the V producer (TMA
// into separate rings, each paced only by its own ring), warp 1 the MMA warp (it
// runs the schedule, one elected lane issues) and tensor-memory owner, warp 2 the
// scheduler of the key-split instance; warpgroups 1 and 2 = softmax of query
// tiles 0 and 1, one TMEM lane (row) per thread.  Registers move from warpgroup 0
// to the softmax warpgroups (setmaxnreg), which hold a row's 128 scores.
//
// MMA order per key tile t:  P V_0 of tile t-1, S_0 of t, P V_1 of t-1, S_1 of t
// (P V_1 moves ahead of S_0 when its P is ready).  S_q of tile t overwrites the
// columns holding P_q of tile t-1, so it waits for that P V to complete; queued
// MMAs of the other query tile run meanwhile.  The
// running maximum is rescaled lazily: O and the normaliser only when a row's
// maximum grows by more than 2^8, so the exponentials stay below 256.  A parity
// wait only tells a barrier's current phase from the one before, so every
// barrier is waited on at every phase, in order (or provably within one phase);
// every wait is bounded.
//
// Key split (a second instance, for chunks of at most 128 rows, such as a
// speculative-decode verification of a few drafts): both query slots hold the
// same rows and take the item's key tiles alternately, so two S -> softmax ->
// P V chains run at once; the query tile the item does not need becomes a third
// V stage; at the item's end slot 1 divides its O by its normaliser in tensor
// memory and hands its weight log2(l) + m to slot 0, which combines the two.
#include <algorithm>
#include <cstring>
#include <type_traits>

#include "pa_attn_common.cuh"
#include "pa_internal.h"

namespace pa_dev {
namespace tc {

constexpr int kRows = 128;      // query rows per tile (MMA M)
constexpr int kQTiles = 2;      // query tiles per item
constexpr int kCtaRows = kQTiles * kRows;
constexpr int kKeys = 128;      // keys per tile (MMA N of S, K of P V)
constexpr int kTileBlocks = kKeys / kBlock;  // 8
constexpr int kKS = 3;          // K stages
constexpr int kVS = 2;          // V stages (the key split adds a third, see Layout)
constexpr int kVSMax = 3;
constexpr int kFlagRing = 8;    // tiles whose block-validity masks are kept
constexpr int kSoftmaxThreads = 128;  // per query tile
constexpr int kThreads = 128 + kQTiles * kSoftmaxThreads;  // 12 warps, 3 warpgroups
constexpr int kLaunchRegs = 168;      // registers per thread at launch (65536 / 384)
constexpr int kCtlRegs = 112;          // warpgroup 0 after setmaxnreg.dec
constexpr int kSoftmaxRegs = 192;     // softmax warpgroups after setmaxnreg.inc
static_assert(128 * kCtlRegs + 256 * kSoftmaxRegs <= kThreads * kLaunchRegs,
              "the register split must fit the launch's registers");
static_assert(kCtlRegs + 2 * kSoftmaxRegs <= 512, "per sub-partition register file");
constexpr float kLazyRescale = 8.0f;  // log2 of the growth that forces a rescale
constexpr float kNoMax = -1.0e30f;    // running-maximum sentinel: 2^(-inf - kNoMax) = 0
constexpr int kMaxPlan = 512;         // (sequence, tile) pairs the CTA orders by cost
constexpr int kItemCost = 6;          // per-item overhead, in key tiles (measured best of 1, 3, 6, 10)

template <int D>
struct Layout {
  static constexpr int kChunks = D / 64;               // 128-byte chunks of a row
  static constexpr int kQBytes = kRows * D * 2;        // per tile: [chunk][128 rows][128 B]
  static constexpr int kKVChunk = kKeys * 128;         // one chunk of a K or V tile
  static constexpr int kKVBytes = kChunks * kKVChunk;  // [chunk][128 keys][128 B]
  static constexpr int kQOff = 0;
  static constexpr int kKOff = kQOff + kQTiles * kQBytes;
  static constexpr int kVOff = kKOff + kKS * kKVBytes;
  static constexpr int kBarOff = kVOff + kVS * kKVBytes;
  // barriers: k_full[KS], k_free[KS], v_full[VS], v_free[VS], q_full, q_free,
  // then per query tile s_full, p_full, pv_done
  static constexpr int kNumBars = 2 * kKS + 2 * kVSMax + 2 + 3 * kQTiles + 2;
  static constexpr int kFlagOff = kBarOff + kNumBars * 8;  // block masks [kFlagRing]
  static constexpr int kTmemSlotOff = kFlagOff + kFlagRing * 4;
  static constexpr int kOrderOff = kTmemSlotOff + 16;  // work order [kMaxPlan] uint16
  static constexpr int kXchOff = kOrderOff + kMaxPlan * 2;  // key split: slot 1's weight per row
  // greedy work assignment: this CTA's work-list positions, their count, a done
  // flag, and the cost totals it is decided on
  static constexpr int kSchedOff = kXchOff + kRows * 4;
  static constexpr int kSchedItems = 128;
  static constexpr int kUsed = kSchedOff + kSchedItems * 2 + 6 * 4;
  // key split: both slots read query tile 0, and tile 1's space is a third V
  // stage (a V tile is exactly a Q tile: 128 rows of D 16-bit values)
  static constexpr int kV2Off = kQOff + kQBytes;
  static_assert(kKVBytes == kQBytes, "the third V stage fills query tile 1");
  static __host__ __device__ constexpr int v_off(int s) {
    return s < kVS ? kVOff + s * kKVBytes : kV2Off;
  }
  static constexpr int kBytes = kUsed + 1024;  // room to align the base to 1024
  // tensor memory columns per query tile: S (P in its first 64), then O
  static constexpr uint32_t kSCol = 0, kOCol = kKeys;
  static constexpr uint32_t kTileCols = 256;
  static constexpr uint32_t kTmemCols = kQTiles * kTileCols;
  static_assert(kOCol + D <= kTileCols, "tensor memory budget");
  static_assert(kBytes <= 232448, "shared memory budget");
  static_assert(kMaxPlan * 4 <= kVS * kKVBytes, "cost scratch fits the V stages");
};

// Shared-memory matrix descriptor, 128-byte swizzle (sm_100 family layout:
// start >> 4 in bits 0-13, leading byte offset >> 4 in 16-29, stride byte
// offset >> 4 in 32-45, version 1 in 46-47, swizzle mode 2 in 61-63).
__device__ __forceinline__ uint64_t sw128_desc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((addr >> 4) & 0x3FFF) | ((uint64_t)((lbo >> 4) & 0x3FFF) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFF) << 32) | (1ull << 46) | (2ull << 61);
}

// Instruction descriptor of kind::f16 with f32 accumulate: D format bits 4-5,
// A/B formats bits 7-9 / 10-12 (0 f16, 1 bf16), B major bit 16 (1 = MN-major),
// N >> 3 in bits 17-22, M >> 4 in bits 24-28.
template <bool BF16>
__host__ __device__ constexpr uint32_t idesc(int M, int N, bool b_mn_major) {
  return (1u << 4) | ((BF16 ? 1u : 0u) << 7) | ((BF16 ? 1u : 0u) << 10) |
         ((b_mn_major ? 1u : 0u) << 16) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// The MMA warp runs its schedule with all 32 lanes, so the descriptors stay
// warp-uniform, and one elected lane issues each MMA and commit.
__device__ __forceinline__ void mma_elect(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t id,
                                          uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\telect.sync _|e, 0xffffffff;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(id), "r"(accumulate));
}

// As mma_elect with the A operand in tensor memory: row m of A in lane m, two
// 16-bit elements per 32-bit column (the even k in the low half).
__device__ __forceinline__ void mma_elect_tmem_a(uint32_t d_tmem, uint32_t a_tmem, uint64_t b,
                                                 uint32_t id, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\telect.sync _|e, 0xffffffff;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b), "r"(id), "r"(accumulate));
}

__device__ __forceinline__ void commit_elect(uint64_t* bar) {
  asm volatile(
      "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(
          smem_u32(bar))
      : "memory");
}

// Whether the phase with the given parity has completed, without waiting
// (every lane asks; the verdict is the warp's).
__device__ __forceinline__ bool warp_test(uint64_t* bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return __all_sync(0xffffffffu, done != 0);
}

// Bounded wait by every lane of a warp; the verdict is the warp's (uniform).
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity) {
  return __all_sync(0xffffffffu, mbar_wait(bar, parity));
}


__device__ __forceinline__ void fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

template <int N>
__device__ __forceinline__ void setmaxnreg_inc() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}
template <int N>
__device__ __forceinline__ void setmaxnreg_dec() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}

// 32 consecutive fp32 columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 32; i++) v[i] = __uint_as_float(r[i]);
}

// 16 columns of this thread's TMEM lane (as tmem_ld32).
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15}, [%16];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 16; i++) v[i] = __uint_as_float(r[i]);
}

// 128 consecutive fp32 columns of this thread's TMEM lane, one load and one wait
// in the same asm statement (no use of the registers can move before the wait).
__device__ __forceinline__ void tmem_ld128(uint32_t taddr, float (&v)[128]) {
  uint32_t r[128];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x128.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63,%64,%65,%66,%67,%68,%69,%70,%71,%72,%73,%74,%75,%76,%77,%78,%79,%80,%81,%82,%83,%84,%85,%86,%87,%88,%89,%90,%91,%92,%93,%94,%95,%96,%97,%98,%99,%100,%101,%102,%103,%104,%105,%106,%107,%108,%109,%110,%111,%112,%113,%114,%115,%116,%117,%118,%119,%120,%121,%122,%123,%124,%125,%126,%127}, [%128];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]), "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63]), "=r"(r[64]), "=r"(r[65]), "=r"(r[66]), "=r"(r[67]), "=r"(r[68]), "=r"(r[69]), "=r"(r[70]), "=r"(r[71]), "=r"(r[72]), "=r"(r[73]), "=r"(r[74]), "=r"(r[75]), "=r"(r[76]), "=r"(r[77]), "=r"(r[78]), "=r"(r[79]), "=r"(r[80]), "=r"(r[81]), "=r"(r[82]), "=r"(r[83]), "=r"(r[84]), "=r"(r[85]), "=r"(r[86]), "=r"(r[87]), "=r"(r[88]), "=r"(r[89]), "=r"(r[90]), "=r"(r[91]), "=r"(r[92]), "=r"(r[93]), "=r"(r[94]), "=r"(r[95]), "=r"(r[96]), "=r"(r[97]), "=r"(r[98]), "=r"(r[99]), "=r"(r[100]), "=r"(r[101]), "=r"(r[102]), "=r"(r[103]), "=r"(r[104]), "=r"(r[105]), "=r"(r[106]), "=r"(r[107]), "=r"(r[108]), "=r"(r[109]), "=r"(r[110]), "=r"(r[111]), "=r"(r[112]), "=r"(r[113]), "=r"(r[114]), "=r"(r[115]), "=r"(r[116]), "=r"(r[117]), "=r"(r[118]), "=r"(r[119]), "=r"(r[120]), "=r"(r[121]), "=r"(r[122]), "=r"(r[123]), "=r"(r[124]), "=r"(r[125]), "=r"(r[126]), "=r"(r[127])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 128; i++) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float (&v)[32]) {
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
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// 64 consecutive 32-bit columns (a row of P: 128 packed 16-bit values).
__device__ __forceinline__ void tmem_st64(uint32_t taddr, const uint32_t (&v)[64]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x64.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63,%64};\n\t"
      "tcgen05.wait::st.sync.aligned;" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]), "r"(v[16]), "r"(v[17]), "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]), "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]), "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31]), "r"(v[32]), "r"(v[33]), "r"(v[34]), "r"(v[35]), "r"(v[36]), "r"(v[37]), "r"(v[38]), "r"(v[39]), "r"(v[40]), "r"(v[41]), "r"(v[42]), "r"(v[43]), "r"(v[44]), "r"(v[45]), "r"(v[46]), "r"(v[47]), "r"(v[48]), "r"(v[49]), "r"(v[50]), "r"(v[51]), "r"(v[52]), "r"(v[53]), "r"(v[54]), "r"(v[55]), "r"(v[56]), "r"(v[57]), "r"(v[58]), "r"(v[59]), "r"(v[60]), "r"(v[61]), "r"(v[62]), "r"(v[63])
      : "memory");
}

// Three-input maximum and packed fp32 pairs (two IEEE operations per instruction).
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}
__device__ __forceinline__ unsigned long long f2pack(float a, float b) {
  unsigned long long r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ void f2unpack(unsigned long long r, float& a, float& b) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(r));
}
__device__ __forceinline__ unsigned long long ffma2(unsigned long long a, unsigned long long b,
                                                    unsigned long long c) {
  unsigned long long d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ unsigned long long fadd2(unsigned long long a, unsigned long long b) {
  unsigned long long d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

// Byte offset of 16-byte unit u (0..7) of row r in a 128-byte-row swizzled chunk.
__device__ __forceinline__ uint32_t sw_unit(int r, int u) {
  return (uint32_t)(r * 128 + (((u ^ r) & 7) << 4));
}
// Zero the V rows of block-start key `key0` (within a V stage) from row
// `valid_rows` on: slots past the context end, which were never written.  Split
// over the 128 threads of query tile 0; the writes are made visible to the
// tensor core's (async proxy) reads.
template <class LY>
__device__ __forceinline__ void zero_v_tail(uint8_t* vbase, int key0, int valid_rows, int stid) {
  const int nz = (kBlock - valid_rows) * LY::kChunks * 8;
  for (int idx = stid; idx < nz; idx += kSoftmaxThreads) {
    const int key = key0 + valid_rows + idx / (LY::kChunks * 8);
    const int rest = idx % (LY::kChunks * 8);
    *reinterpret_cast<uint4*>(vbase + (rest / 8) * LY::kKVChunk + sw_unit(key, rest % 8)) =
        make_uint4(0, 0, 0, 0);
  }
  fence_proxy_async();
}

// One work item: 256 query rows (two tiles) of one sequence's chunk and one kv
// head, and the key range those rows can see.
struct Item {
  bool valid;  // rows exist (a sequence whose chunk is shorter has fewer items)
  int n, kvh, q0, C, L, R0, nrows, lo_u, hi_u, first, ntiles;
};

// The item from its sequence's raw lengths (q0, q1 = cu_q_lens[n], cu_q_lens[n+1],
// Lraw = context_lens[n]), with the checks of clamp_context.
__device__ __forceinline__ Item item_make(const AttnParams& p, int n, int kvh, int tile, int q0,
                                          int q1, int Lraw, bool report) {
  Item it;
  it.valid = false;
  it.ntiles = 0;
  it.n = n;
  it.kvh = kvh;
  report = report && kvh == 0 && tile == 0;  // one report per sequence
  if (q0 < 0 || q1 < q0 || q1 > p.num_q_tokens) {
    if (report) set_flag(p.err, PA_FLAG_Q_LEN);
    return it;
  }
  int C = q1 - q0;
  if (C > p.max_q_len) {
    if (report) set_flag(p.err, PA_FLAG_Q_LEN);
    C = p.max_q_len;
  }
  const int cap = p.max_blocks_per_seq * kBlock;
  int L = Lraw;
  if (L < 0 || L > cap) {
    if (report) set_flag(p.err, PA_FLAG_CONTEXT_LEN);
    L = L < 0 ? 0 : cap;
  }
  if (C > L && report) set_flag(p.err, PA_FLAG_Q_LEN);
  it.q0 = q0;
  it.C = C;
  it.L = L;
  it.R0 = tile * kCtaRows;
  it.nrows = C * p.group;
  if (it.R0 >= it.nrows) return it;
  it.valid = true;
  const int c_first = it.R0 / p.group;
  const int c_last = (min(it.R0 + kCtaRows, it.nrows) - 1) / p.group;
  it.hi_u = L - C + c_last;
  it.lo_u = p.window > 0 ? max(0, L - C + c_first - p.window + 1) : 0;
  it.first = it.lo_u / kBlock;
  const int last = it.hi_u / kBlock;
  it.ntiles = it.hi_u >= it.lo_u ? (last - it.first) / kTileBlocks + 1 : 0;
  return it;
}

__device__ __forceinline__ Item item_info(const AttnParams& p, int n, int kvh, int tile,
                                          bool report) {
  return item_make(p, n, kvh, tile, p.cu_q_lens[n], p.cu_q_lens[n + 1], p.context_lens[n],
                   report);
}

// The work list: items ordered by cost (key tiles + a fixed overhead), longest
// first, when the CTA could rank the (sequence, tile) pairs (every kv head of a
// pair costs the same); in (sequence, kv head, tile) order otherwise.  With the
// ranked list of a short-chunk (key-split) launch the CTAs take the items
// greedily, each next item to the CTA with
// the least work so far (ties to the lower index; warp 2 of every CTA computes
// the same assignment and publishes its own CTA's part, see the kernel), when a
// bound guarantees that no CTA gets more than kSchedItems items; otherwise
// round r of the list goes to the CTAs in alternating directions (CTA b takes
// position r*grid + b in even rounds, r*grid + grid-1-b in odd ones).  Either
// way CTA b's first item is position b.  Returns false past the end (or when a
// bounded wait for the assignment ran out).
struct WorkList {
  // Only the CTA-wide decisions are held (in registers of every role); the
  // ranked order [num_pairs] and the greedy positions live in shared memory at
  // the layout's offsets, and the sizes come from the parameters.
  bool ranked;      // the order of the pairs by cost exists
  bool greedy;      // greedy assignment (ranked list of a key-split launch)
  int first_items;  // positions of cost > 0 (ranked list)

  template <class LY>
  __device__ __forceinline__ bool at(const AttnParams& p, int num_pairs, const uint8_t* smem,
                                     int j, int& n, int& kvh, int& tile) const {
    const int grid = gridDim.x, b = blockIdx.x;
    const int kv_heads = p.num_kv_heads, q_tiles = p.q_tiles;
    long long s;
    if (greedy) {
      const volatile int* count = reinterpret_cast<const volatile int*>(
          smem + LY::kSchedOff + LY::kSchedItems * 2);
      if (j == 0) {
        if (b >= first_items) return false;
        s = b;
      } else {
        const long long t0 = clock64();
        while (count[0] <= j) {
          if (count[1]) {  // all are published
            if (count[0] <= j) return false;
            break;
          }
          if (clock64() - t0 > kWaitLimitCycles) return false;
        }
        __threadfence_block();
        s = reinterpret_cast<const volatile uint16_t*>(smem + LY::kSchedOff)[j];
      }
    } else {
      s = (long long)j * grid + ((j & 1) ? grid - 1 - b : b);
    }
    if (s >= (long long)num_pairs * kv_heads) return false;
    if (ranked) {
      const int pair = reinterpret_cast<const uint16_t*>(smem + LY::kOrderOff)[s / kv_heads] & 0x1FF;
      kvh = (int)(s % kv_heads);
      n = pair / q_tiles;
      tile = pair % q_tiles;
    } else {
      const int per_seq = q_tiles * kv_heads;
      n = (int)(s / per_seq);
      kvh = (int)(s % per_seq) / q_tiles;
      tile = (int)(s % per_seq) % q_tiles;
    }
    return true;
  }
  // whether position j is known without waiting (greedy: published, or the
  // list is complete)
  template <class LY>
  __device__ __forceinline__ bool ready(const uint8_t* smem, int j) const {
    if (!greedy || j == 0) return true;
    const volatile int* count =
        reinterpret_cast<const volatile int*>(smem + LY::kSchedOff + LY::kSchedItems * 2);
    return count[0] > j || count[1] != 0;
  }
};

// A role's walk over its CTA's items.  fetch() looks up the next item and
// starts the loads of its sequence's lengths; take() hands it out (fetching
// first if that has not happened).  Calling fetch() early -- at an item's start,
// or after its last tile -- lets the global-memory latency pass while the
// current item's work runs instead of at the next item's start.  A greedy
// list publishes its positions as the scheduler warp assigns them: an early
// fetch does not wait for one (take() will).
template <class LY>
struct ItemStream {
  WorkList wl;
  int j, n, kvh, tile, q0, q1, L;
  bool have, fetched;

  __device__ __forceinline__ explicit ItemStream(const WorkList& w) : wl(w), j(0), fetched(false) {}
  __device__ __forceinline__ void load(const AttnParams& p, int num_pairs, const uint8_t* smem) {
    fetched = true;
    have = wl.template at<LY>(p, num_pairs, smem, j, n, kvh, tile);
    if (have) {
      q0 = p.cu_q_lens[n];
      q1 = p.cu_q_lens[n + 1];
      L = p.context_lens[n];
    }
  }
  __device__ __forceinline__ void fetch(const AttnParams& p, int num_pairs, const uint8_t* smem) {
    if (!fetched && wl.template ready<LY>(smem, j)) load(p, num_pairs, smem);
  }
  __device__ __forceinline__ bool take(const AttnParams& p, int num_pairs, const uint8_t* smem,
                                       Item& it, bool report) {
    if (!fetched) load(p, num_pairs, smem);
    if (!have) return false;
    it = item_make(p, n, kvh, tile, q0, q1, L, report);
    j++;
    fetched = false;
    return true;
  }
};

// Persistent: each CTA walks its part of the work list.  Every role walks the
// same items; the tile counter g (and the item counter k for Q) runs on across
// items, so each barrier keeps stepping one phase at a time, and the next
// item's Q and first K/V tiles load while the current item's last tiles finish.
//
// KS (key split; an item of at most 128 rows): both query slots hold the same
// rows (query tile 0) and take the item's key tiles alternately, slot t & 1
// taking tile t, so that two S -> softmax -> P V chains are in flight at once;
// each slot keeps its own running maximum, normaliser and O, and slot 0's
// threads merge the two at the end of the item (reading slot 1's O from the
// same tensor-memory lanes and its (m, l) from shared memory).
template <int D, typename QT, bool KS>
__global__ void __launch_bounds__(kThreads, 1)
    pa_prefill_tc_kernel(const __grid_constant__ AttnParams p,
                         const __grid_constant__ CUtensorMap tmk,
                         const __grid_constant__ CUtensorMap tmv,
                         const __grid_constant__ CUtensorMap tmq, int num_seqs, int q_tma) {
  using LY = Layout<D>;
  constexpr bool BF = std::is_same<QT, __nv_bfloat16>::value;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  pdl_wait();  // the kernel before (say, the K/V write) is complete
  pdl_launch_dependents();
  uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + LY::kBarOff);
  uint64_t* k_full = bars;
  uint64_t* k_free = k_full + kKS;
  uint64_t* v_full = k_free + kKS;
  uint64_t* v_free = v_full + kVSMax;
  uint64_t* q_full = v_free + kVSMax;
  uint64_t* q_free = q_full + 1;
  uint64_t* s_full = q_free + 1;          // [kQTiles]: S_q of the current tile is in TMEM
  uint64_t* p_full = s_full + kQTiles;    // [kQTiles]: P_q is in TMEM (128 arrivals)
  uint64_t* pv_done = p_full + kQTiles;   // [kQTiles]: the P V that read P_q finished
  uint64_t* merge_ready = pv_done + kQTiles;  // KS: slot 1's (m, l) are in shared memory
  uint64_t* merge_done = merge_ready + 1;     // KS: slot 0 has read slot 1's O
  float* xch = reinterpret_cast<float*>(smem + LY::kXchOff);
  uint16_t* sched_items = reinterpret_cast<uint16_t*>(smem + LY::kSchedOff);
  int* sched = reinterpret_cast<int*>(smem + LY::kSchedOff + LY::kSchedItems * 2);
  // sched[0] count, [1] done, [2] total cost, [3] largest, [4] smallest nonzero,
  // [5] pairs of nonzero cost
  constexpr int VS = KS ? kVSMax : kVS;  // V stages in use
  uint32_t* bmask = reinterpret_cast<uint32_t*>(smem + LY::kFlagOff);  // loaded blocks per tile
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + LY::kTmemSlotOff);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = p.group;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kKS; i++) {
      mbar_init(&k_full[i], 1);
      mbar_init(&k_free[i], 1);
    }
    for (int i = 0; i < VS; i++) {
      mbar_init(&v_full[i], 1);
      mbar_init(&v_free[i], 1);
    }
    mbar_init(q_full, 32);  // the producer warp's lanes
    mbar_init(q_free, 1);
    for (int q = 0; q < kQTiles; q++) {
      mbar_init(&s_full[q], 1);
      mbar_init(&p_full[q], kSoftmaxThreads);
      mbar_init(&pv_done[q], 1);
    }
    mbar_init(merge_ready, kSoftmaxThreads);
    mbar_init(merge_done, kSoftmaxThreads);
    sched[0] = sched[1] = sched[2] = sched[3] = sched[5] = 0;
    sched[4] = 0x7fffffff;
    fence_mbar_init();
  }
  // Tensor memory: per query tile, S (P in its first half) and O -- all 512
  // columns of the SM.  The allocation does not wait on another CTA of this
  // launch: the 231.6 KB of dynamic shared memory leaves room for one CTA per SM,
  // and the library's other kernels allocate no tensor memory.
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(tmem_slot)),
                 "r"(LY::kTmemCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  // the work order (the V stages serve as scratch: nothing has been loaded yet)
  const int num_pairs = num_seqs * p.q_tiles;
  WorkList wl;
  wl.ranked = false;
  wl.greedy = false;
  wl.first_items = 0;
  __syncthreads();  // the scheduler's counters are set
  if (num_pairs <= kMaxPlan) {
    int* cost = reinterpret_cast<int*>(smem + LY::kVOff);
    uint16_t* order = reinterpret_cast<uint16_t*>(smem + LY::kOrderOff);
    for (int j = threadIdx.x; j < num_pairs; j += kThreads) {
      const Item it = item_info(p, j / p.q_tiles, 0, j % p.q_tiles, false);
      const int c = it.valid ? min(it.ntiles + kItemCost, 127) : 0;
      cost[j] = c;
      if (c > 0) {
        atomicAdd(&sched[2], c * p.num_kv_heads);
        atomicMax(&sched[3], c);
        atomicMin(&sched[4], c);
        atomicAdd(&sched[5], 1);
      }
    }
    __syncthreads();
    for (int j = threadIdx.x; j < num_pairs; j += kThreads) {
      const int cj = cost[j];
      int rank = 0;
      for (int i2 = 0; i2 < num_pairs; i2++) {
        const int ci = cost[i2];
        rank += (ci > cj || (ci == cj && i2 < j)) ? 1 : 0;
      }
      order[rank] = (uint16_t)(j | (cj << 9));
    }
    wl.ranked = true;
  }
  fence_before();
  __syncthreads();
  fence_after();
  if (KS && wl.ranked && sched[5] > 0 && gridDim.x <= 160) {
    // greedy (short chunks: many items of very different lengths; the long
    // chunks' few large items keep the alternating order, which measured
    // better there) when it provably fits: a CTA's work stays below
    // total/grid + the largest cost, so it holds at most that over the smallest
    // cost items
    const long long bound =
        ((long long)sched[2] / gridDim.x + sched[3] + sched[4] - 1) / sched[4] + 1;
    wl.greedy = bound <= LY::kSchedItems;
    wl.first_items = sched[5] * p.num_kv_heads;
  }
  const uint32_t tmem = *tmem_slot;
  bool timed_out = false;

  if (warp < 4) {
    setmaxnreg_dec<kCtlRegs>();
    if (warp == 0 || warp == 3) {
      // ---------------- producers: warp 0 loads each item's Q and its K tiles,
      // warp 3 its V tiles, so that neither ring waits for the other's stages
      // (a V stage frees a tile later than a K stage does)
      const bool kprod = warp == 0;
      int gk = 0, gv = 0, k = 0;  // K tiles, V tiles and items with tiles so far
      ItemStream<LY> items(wl);
      Item it;
      while (!timed_out && items.take(p, num_pairs, smem, it, threadIdx.x == 0)) {
        items.fetch(p, num_pairs, smem);
        if (!it.valid || it.ntiles == 0) continue;
        // Q of this item, once the previous item's S MMAs have finished with it
        if (kprod && k > 0 && !warp_wait(q_free, (k - 1) & 1)) {
          timed_out = true;
          break;
        }
        uint8_t* qs = smem + LY::kQOff;
        constexpr int kQLoad = KS ? 1 : kQTiles;  // key split: tile 0 only
        if (!kprod) {
          // V producer: no Q
        } else if (q_tma) {
          // box [128/G tokens][G heads][64 columns] = 128 rows of the tile
          if (lane == 0) mbar_arrive_expect_tx(q_full, kQLoad * LY::kQBytes);
          __syncwarp();
          if (lane < kQLoad * LY::kChunks) {
            const int q = lane / LY::kChunks, h = lane % LY::kChunks;
            tma_load_3d(qs + q * LY::kQBytes + h * (kRows * 128), &tmq, 64 * h, it.kvh * G,
                        it.q0 + (it.R0 + q * kRows) / G, q_full);
          }
          if (lane != 0) mbar_arrive(q_full);
        } else {
          const QT* qg = static_cast<const QT*>(p.q);
          for (int r = lane; r < kQLoad * kRows; r += 32) {
            const int R = it.R0 + r;
            const bool rv = R < it.nrows;
            const long long orow =
                rv ? (long long)(it.q0 + R / G) * p.num_q_heads + it.kvh * G + R % G : 0;
            const uint4* src = reinterpret_cast<const uint4*>(qg + orow * D);
            uint8_t* qt = qs + (r / kRows) * LY::kQBytes;
#pragma unroll
            for (int u = 0; u < D / 8; u++)
              cp_async_16_or_zero(qt + (u / 8) * (kRows * 128) + sw_unit(r % kRows, u % 8),
                                  src + u, rv);
          }
          cp_async_wait_all();
          fence_proxy_async();
          mbar_arrive(q_full);
        }
        k++;
        // block ids 32 at a time (lane l holds entry 32*b + l of batch b), the
        // next batch loaded while this one is used
        const int32_t* table =
            p.block_tables + (long long)it.n * p.max_blocks_per_seq + it.first;
        const int nblk = it.hi_u / kBlock - it.first + 1;
        constexpr int kTilesPerBatch = 32 / kTileBlocks;
        auto batch = [&](int b) { return 32 * b + lane < nblk ? table[32 * b + lane] : -1; };
        int ids = batch(0), ids_next = batch(1);
        for (int t = 0; t < it.ntiles; t++) {
          if (t > 0 && t % kTilesPerBatch == 0) {
            ids = ids_next;
            ids_next = batch(t / kTilesPerBatch + 1);
          }
          const int from = __shfl_sync(0xffffffffu, ids, (kTileBlocks * t + lane) & 31);
          const bool inside = lane < kTileBlocks && kTileBlocks * t + lane < nblk;
          const int mine = inside ? from : -1;
          const bool ok = inside && mine >= 0 && mine < p.num_blocks;
          if (kprod && inside && !ok) set_flag(p.err, PA_FLAG_BLOCK_ID);
          const unsigned okmask = __ballot_sync(0xffffffffu, ok);
          const uint32_t tile_bytes = __popc(okmask) * LY::kChunks * kBlock * 128;
          const int row0 = (mine * p.num_kv_heads + it.kvh) * kBlock;
          if (kprod) {
            // K of tile gk
            const int ks = gk % kKS;
            if (gk >= kKS && !warp_wait(&k_free[ks], ((gk / kKS) - 1) & 1)) {
              timed_out = true;
              break;
            }
            if (lane == 0) {
              bmask[gk % kFlagRing] = okmask;
              mbar_arrive_expect_tx(&k_full[ks], tile_bytes);
            }
            __syncwarp();
            if (ok) {
              uint8_t* kbase = smem + LY::kKOff + ks * LY::kKVBytes;
#pragma unroll
              for (int h = 0; h < LY::kChunks; h++)
                tma_load_2d(kbase + h * LY::kKVChunk + lane * kBlock * 128, &tmk, 64 * h, row0,
                            &k_full[ks]);
            }
            gk++;
          } else {
            // V of tile gv
            const int vs = gv % VS;
            if (gv >= VS && !warp_wait(&v_free[vs], ((gv / VS) - 1) & 1)) {
              timed_out = true;
              break;
            }
            if (lane == 0) mbar_arrive_expect_tx(&v_full[vs], tile_bytes);
            __syncwarp();
            if (ok) {
              uint8_t* vbase = smem + LY::v_off(vs);
#pragma unroll
              for (int h = 0; h < LY::kChunks; h++)
                tma_load_2d(vbase + h * LY::kKVChunk + lane * kBlock * 128, &tmv, 64 * h, row0,
                            &v_full[vs]);
            }
            gv++;
          }
        }
      }
      // no copy may still be landing in shared memory when the CTA exits; the
      // last fills issued are their barriers' current phases
      if (lane == 0) {
        for (int t = gk > kKS ? gk - kKS : 0; t < gk; t++)
          if (!mbar_wait(&k_full[t % kKS], (t / kKS) & 1)) break;
        for (int t = gv > VS ? gv - VS : 0; t < gv; t++)
          if (!mbar_wait(&v_full[t % VS], (t / VS) & 1)) break;
        if (kprod && k > 0 && !mbar_wait(q_full, (k - 1) & 1)) timed_out = true;
      }
      if (timed_out && lane == 0) set_flag(p.err, PA_FLAG_TIMEOUT);
    } else if (warp == 2) {
      // ---------------- scheduler: the greedy assignment, every CTA alike (lane
      // l keeps the work of CTAs l, l+32, ..., l+128 as keys work << 8 | CTA)
      if (wl.greedy) {
        uint32_t load[5] = {0u, 0u, 0u, 0u, 0u};
        int mine = 0;
        const int grid = gridDim.x;
        for (int s = 0; s < wl.first_items; s++) {
          const uint32_t c = reinterpret_cast<const uint16_t*>(smem + LY::kOrderOff)[s / p.num_kv_heads] >> 9;
          uint32_t best = 0xffffffffu;
#pragma unroll
          for (int q = 0; q < 5; q++)
            if (lane + 32 * q < grid) best = min(best, (load[q] << 8) | (uint32_t)(lane + 32 * q));
          best = __reduce_min_sync(0xffffffffu, best);
          const int win = (int)(best & 0xffu);
#pragma unroll
          for (int q = 0; q < 5; q++)
            if (win == lane + 32 * q) load[q] += c;
          if (win == (int)blockIdx.x) {
            if (lane == 0 && mine < LY::kSchedItems) {  // the bound keeps it below
              sched_items[mine] = (uint16_t)s;
              __threadfence_block();
              *reinterpret_cast<volatile int*>(&sched[0]) = mine + 1;
            }
            mine++;
          }
        }
        if (lane == 0) {
          __threadfence_block();
          *reinterpret_cast<volatile int*>(&sched[1]) = 1;
        }
      }
    } else if (warp == 1) {
      // ---------------- MMA warp (one elected lane issues)
      const uint32_t idS = idesc<BF>(kRows, kKeys, false);
      const uint32_t idO = idesc<BF>(kRows, D, true);
      // descriptors advance by adding (byte offset >> 4) to the start-address
      // field: every shared-memory address here is below 256 KB, so no carry
      const uint64_t dQ0 = sw128_desc(smem_u32(smem + LY::kQOff), 16, 1024);
      const uint64_t dK0 = sw128_desc(smem_u32(smem + LY::kKOff), 16, 1024);
      const uint64_t dV0 = sw128_desc(smem_u32(smem + LY::kVOff), LY::kKVChunk, 1024);
      bool started0 = false, started1 = false;  // O_q holds this item's first product
      // O_q (+)= P_q V of tile gg, skipping the blocks that were not loaded
      bool live1 = true;  // query tile 1 of the current item has rows (short chunks may not)
      auto pv = [&](int q, int gg, bool& started) -> bool {
        if (!warp_wait(&p_full[q], gg & 1)) return false;
        fence_after();
        if (q == 1 && !live1) {  // nothing to compute; the commit keeps the phases
          commit_elect(&pv_done[q]);
          return true;
        }
        const uint64_t dV = dV0 + (uint64_t)(((gg % kVS) * LY::kKVBytes) >> 4);
        // lane 0's copy: the compiler sees one value for the warp
        const uint32_t mask = __shfl_sync(0xffffffffu, bmask[gg % kFlagRing], 0);
        const uint32_t dO = tmem + q * LY::kTileCols + LY::kOCol;
        const uint32_t aP = tmem + q * LY::kTileCols + LY::kSCol;
        if (mask == 0xFFu && started) {
#pragma unroll
          for (int s = 0; s < kTileBlocks; s++)
            mma_elect_tmem_a(dO, aP + 8 * s, dV + (uint64_t)((2048 * s) >> 4), idO, 1u);
        } else {
#pragma unroll
          for (int s = 0; s < kTileBlocks; s++)
            if ((mask >> s) & 1u) {
              mma_elect_tmem_a(dO, aP + 8 * s, dV + (uint64_t)((2048 * s) >> 4), idO,
                               started ? 1u : 0u);
              started = true;
            }
        }
        commit_elect(&pv_done[q]);
        return true;
      };
      // S_q of tile gg; it overwrites the columns that held P_q of tile gg-1
      auto s_mma = [&](int q, int gg, uint64_t dK) -> bool {
        if (gg >= 1 && !warp_wait(&pv_done[q], (gg - 1) & 1)) return false;
        fence_after();
        if (q == 1 && !live1) {
          commit_elect(&s_full[q]);
          return true;
        }
        const uint64_t dQ = dQ0 + (uint64_t)((q * LY::kQBytes) >> 4);
        const uint32_t dS = tmem + q * LY::kTileCols + LY::kSCol;
#pragma unroll
        for (int s = 0; s < D / 16; s++)
          mma_elect(dS, dQ + (uint64_t)(((s / 4) * (kRows * 128) + (s % 4) * 32) >> 4),
                    dK + (uint64_t)(((s / 4) * LY::kKVChunk + (s % 4) * 32) >> 4), idS,
                    s > 0 ? 1u : 0u);
        commit_elect(&s_full[q]);
        return true;
      };
      static_assert(kQTiles == 2, "the MMA schedule is written for two query tiles");
      bool ok = true;
      if constexpr (KS) {
        // slot q's tiles so far (c[q]) step its barriers; per tile: S into the
        // tile's slot, then P V of the previous tile (the other slot)
        // P V of tile gg into slot q (its c-th tile); returns whether O_q now holds
        // a product, or -1 if the wait ran out
        auto pvk = [&](int q, int c, int gg, bool started) -> int {
          if (!warp_wait(&p_full[q], c & 1)) return -1;
          fence_after();
          const uint64_t dV = sw128_desc(smem_u32(smem + LY::v_off(gg % VS)), LY::kKVChunk, 1024);
          const uint32_t mask = bmask[gg % kFlagRing];
          const uint32_t dO = tmem + q * LY::kTileCols + LY::kOCol;
          const uint32_t aP = tmem + q * LY::kTileCols + LY::kSCol;
#pragma unroll
          for (int s = 0; s < kTileBlocks; s++)
            if ((mask >> s) & 1u) {
              mma_elect_tmem_a(dO, aP + 8 * s, dV + (uint64_t)((2048 * s) >> 4), idO,
                               started ? 1u : 0u);
              started = true;
            }
          commit_elect(&pv_done[q]);
          return started ? 1 : 0;
        };
        auto sk = [&](int q, int c, uint64_t dK) -> bool {
          if (c >= 1 && !warp_wait(&pv_done[q], (c - 1) & 1)) return false;
          fence_after();
          const uint32_t dS = tmem + q * LY::kTileCols + LY::kSCol;
#pragma unroll
          for (int s = 0; s < D / 16; s++)
            mma_elect(dS, dQ0 + (uint64_t)(((s / 4) * (kRows * 128) + (s % 4) * 32) >> 4),
                      dK + (uint64_t)(((s / 4) * LY::kKVChunk + (s % 4) * 32) >> 4), idS,
                      s > 0 ? 1u : 0u);
          commit_elect(&s_full[q]);
          return true;
        };
        int g = 0, k = 0, c0 = 0, c1 = 0;  // c_q: slot q's tiles so far
        ItemStream<LY> items(wl);
        Item it;
        while (ok && items.take(p, num_pairs, smem, it, false)) {
          items.fetch(p, num_pairs, smem);
          if (!it.valid || it.ntiles == 0) continue;
          ok = warp_wait(q_full, k & 1);
          k++;
          bool st0 = false, st1 = false;  // O_q holds this item's first product
          int pq = 0, pc = 0;             // slot and slot count of the previous tile
          auto pv_prev = [&]() {
            ok = warp_wait(&v_full[(g - 1) % VS], ((g - 1) / VS) & 1);
            if (!ok) return;
            const int r = pvk(pq, pc, g - 1, pq ? st1 : st0);
            if (r < 0) {
              ok = false;
              return;
            }
            if (pq) st1 = r != 0;
            else st0 = r != 0;
            commit_elect(&v_free[(g - 1) % VS]);
          };
          for (int t = 0; t < it.ntiles && ok; t++, g++) {
            const int q = t & 1;
            const int cq = q ? c1 : c0;
            ok = warp_wait(&k_full[g % kKS], (g / kKS) & 1);
            const uint64_t dK = dK0 + (uint64_t)(((g % kKS) * LY::kKVBytes) >> 4);
            if (ok) ok = sk(q, cq, dK);
            if (ok) commit_elect(&k_free[g % kKS]);
            if (ok && t == it.ntiles - 1) commit_elect(q_free);  // Q is no longer read
            if (ok && t >= 1) pv_prev();
            pq = q;
            pc = cq;
            if (q) c1++;
            else c0++;
          }
          if (ok) pv_prev();  // the item's last tile
        }
      } else {
        int g = 0, k = 0;
        ItemStream<LY> items(wl);
        Item it;
        while (ok && items.take(p, num_pairs, smem, it, false)) {
          items.fetch(p, num_pairs, smem);
          if (!it.valid || it.ntiles == 0) continue;
          ok = warp_wait(q_full, k & 1);
          k++;
          started0 = started1 = false;
          live1 = it.R0 + kRows < it.nrows;
          // Per tile g: P V of tile g-1 and S of tile g for each query tile, in the
          // order P V_0, S_0, P V_1, S_1, except that P V_1 goes first when its P is
          // already there.  The issuing thread blocks while an MMA waits for the
          // tensor pipe, so the pipe idles whenever the warp does anything else:
          // the wait for the next tile's K (loaded well ahead) is taken while
          // P V_1 runs, just before the wait for it to finish.
          if (ok) ok = warp_wait(&k_full[g % kKS], (g / kKS) & 1);
          for (int t = 0; t < it.ntiles && ok; t++, g++) {
            const uint64_t dK = dK0 + (uint64_t)(((g % kKS) * LY::kKVBytes) >> 4);
            const bool more = t + 1 < it.ntiles;
            if (t >= 1) {
              ok = warp_wait(&v_full[(g - 1) % kVS], ((g - 1) / kVS) & 1);
              if (ok) ok = pv(0, g - 1, started0);
              bool pv1 = false;
              if (ok && warp_test(&p_full[1], (g - 1) & 1)) {
                ok = pv(1, g - 1, started1);
                pv1 = true;
              }
              if (ok) ok = s_mma(0, g, dK);
              if (ok && !pv1) ok = pv(1, g - 1, started1);
              if (ok) commit_elect(&v_free[(g - 1) % kVS]);
            } else {
              ok = s_mma(0, g, dK);
            }
            // the next tile's K
            if (ok && more) ok = warp_wait(&k_full[(g + 1) % kKS], ((g + 1) / kKS) & 1);
            if (ok) ok = s_mma(1, g, dK);
            if (ok) commit_elect(&k_free[g % kKS]);
            if (ok && !more) commit_elect(q_free);  // Q is no longer read
          }
          if (ok) {  // the item's last tile
            ok = warp_wait(&v_full[(g - 1) % kVS], ((g - 1) / kVS) & 1);
            if (ok) ok = pv(0, g - 1, started0);
            if (ok) ok = pv(1, g - 1, started1);
            if (ok) commit_elect(&v_free[(g - 1) % kVS]);
          }
        }
      }
      if (!ok && lane == 0) set_flag(p.err, PA_FLAG_TIMEOUT);
      __syncwarp();
    }
  } else {
    setmaxnreg_inc<kSoftmaxRegs>();
    // ---------------- softmax: query tile q, thread <-> row (TMEM lane 32*(warp%4) + lane)
    const int q = (warp - 4) / 4;
    const int stid = threadIdx.x - 128 - q * kSoftmaxThreads;  // 0..127 within the tile
    const int row = 32 * (warp & 3) + lane;
    const uint32_t lane_base = tmem + q * LY::kTileCols + ((uint32_t)(32 * (warp & 3)) << 16);
    const float sc = p.scale_log2;
    QT* out = static_cast<QT*>(p.out);
    int g = 0;
    // KS: this slot's tiles so far (its barriers' phases), slot 1's tiles so far
    // (slot 0 waits on its P V), and items merged so far
    int cq = 0, c1 = 0, kk = 0;
    ItemStream<LY> items(wl);
    Item it;
    while (!timed_out && items.take(p, num_pairs, smem, it, false)) {
      if (!it.valid) continue;
      const int R = it.R0 + (KS ? 0 : q * kRows) + row;
      const bool rvalid = R < it.nrows;
      const int c = rvalid ? R / G : 0;
      const int pos = it.L - it.C + c;
      const int row_hi = rvalid ? pos : -1;
      const int row_lo = p.window > 0 ? max(0, pos - p.window + 1) : 0;
      const long long orow =
          (long long)(it.q0 + c) * p.num_q_heads + it.kvh * G + (rvalid ? R % G : 0);
      QT* dst = out + orow * D;
      if (it.ntiles == 0) {  // no row sees a key: zeros
        if (rvalid && (!KS || q == 0))
#pragma unroll
          for (int u = 0; u < D / 8; u++) reinterpret_cast<uint4*>(dst)[u] = make_uint4(0, 0, 0, 0);
        continue;
      }
      // a warp whose 32 rows are all past the chunk (short chunks) only keeps
      // the barriers stepping and clears its share of the V tail
      const bool warp_live = __any_sync(0xffffffffu, rvalid);
      // the block holding position L-1 may carry unwritten slots past it
      const int tail_blk = (it.L - 1) / kBlock;
      const int tail_rows = it.L % kBlock;  // valid rows of that block (0: all 16)
      const bool two = KS && it.ntiles >= 2;  // KS: slot 1 has tiles, the slots merge
      if (!warp_live) {
        for (int t = 0; t < it.ntiles; t++, g++) {
          if (KS && (t & 1) != q) continue;  // the other slot's tile
          if (!mbar_wait(&s_full[q], (KS ? cq : g) & 1)) {
            timed_out = true;
            break;
          }
          if (KS) cq++;
          fence_after();
          const int blk0 = it.first + kTileBlocks * t;
          const uint32_t mask = bmask[g % kFlagRing];
          if ((KS || q == 0) && tail_rows != 0 && tail_blk >= blk0 &&
              tail_blk < blk0 + kTileBlocks && ((mask >> (tail_blk - blk0)) & 1u)) {
            if (!mbar_wait(&v_full[g % VS], (g / VS) & 1)) {
              timed_out = true;
              break;
            }
            zero_v_tail<LY>(smem + LY::v_off(g % VS),
                            (tail_blk - blk0) * kBlock, tail_rows, stid);
          }
          fence_before();
          mbar_arrive(&p_full[q]);
        }
        if (timed_out) break;
        if (two) {  // the merge handshake, without data
          if (q == 1) {
            mbar_arrive(merge_ready);
            if (!mbar_wait(merge_done, kk & 1)) timed_out = true;
          } else {
            if (!mbar_wait(merge_ready, kk & 1)) timed_out = true;
            mbar_arrive(merge_done);
          }
          kk++;
        }
        if (KS && q == 0) c1 += it.ntiles / 2;
        continue;
      }
      float m_used = kNoMax, l = 0.0f;
      for (int t = 0; t < it.ntiles; t++, g++) {
        if (KS && (t & 1) != q) continue;  // the other slot's tile
        if (!mbar_wait(&s_full[q], (KS ? cq : g) & 1)) {
          timed_out = true;
          break;
        }
        if (KS) cq++;
        // S of tile g is complete, and with it (it was issued after waiting for
        // it) the P V of tile g-1: O holds every earlier tile
        fence_after();
        const int blk0 = it.first + kTileBlocks * t;
        const int pos0 = blk0 * kBlock;
        const uint32_t mask = bmask[g % kFlagRing];
        float x[kKeys];
        tmem_ld128(lane_base + LY::kSCol, x);
        // maximum of the scaled scores this row can see.  With sm_scale > 0 the
        // scores stay raw (the scale is folded into the exponent's FFMA and applied
        // to the maximum); an inner tile (every key visible to every row of the
        // warp) needs no mask, an edge tile masks the keys outside the row's range
        // [a, b] and the blocks that were not loaded (the same for every row: a
        // uniform branch per block).  Eight partial maxima (three-input max) keep
        // the dependency chains short.  (Rows past the chunk do not hold it back:
        // their outputs are not stored, and each row of O depends on its own row
        // of P only.)
        const bool raw = sc > 0.0f;
        const bool inner = raw && (mask & 0xFFu) == 0xFFu &&
                           __all_sync(0xffffffffu, !rvalid || (pos0 >= row_lo &&
                                                               pos0 + kKeys - 1 <= row_hi));
        if (!inner) {
          // keys this row sees: [a, b] of the tile (rows past the chunk: all)
          const int a = rvalid ? row_lo - pos0 : 0, b = rvalid ? row_hi - pos0 : kKeys - 1;
          if (raw) {
            // 16-key blocks are classed for the whole warp (its rows' bounds differ
            // by a few keys): masked for every row (or not loaded), visible to
            // every row, or mixed -- only mixed blocks are masked key by key
            uint32_t dead, mixed;  // per block: masked for every row / for some rows
            {
              const int amin = __reduce_min_sync(0xffffffffu, rvalid ? a : 0x7fffffff);
              const int amax = __reduce_max_sync(0xffffffffu, rvalid ? a : (int)0x80000000);
              const int bmin = __reduce_min_sync(0xffffffffu, rvalid ? b : 0x7fffffff);
              const int bmax = __reduce_max_sync(0xffffffffu, rvalid ? b : (int)0x80000000);
              dead = ~mask & 0xFFu;
              mixed = 0u;
#pragma unroll
              for (int s = 0; s < kTileBlocks; s++) {
                const int i0 = kBlock * s, i1 = i0 + kBlock - 1;
                if (i1 < amin || i0 > bmax) dead |= 1u << s;
                if (i0 < amax || i1 > bmin) mixed |= 1u << s;
              }
              mixed &= ~dead;
            }
#pragma unroll
            for (int s = 0; s < kTileBlocks; s++) {
              if (((dead | mixed) >> s) & 1u) {
                const bool d = (dead >> s) & 1u;
                const int ea = d ? kKeys : a, eb = d ? -1 : b;
#pragma unroll
                for (int j = 0; j < kBlock; j++) {
                  const int i = kBlock * s + j;
                  x[i] = (i >= ea && i <= eb) ? x[i] : -INFINITY;
                }
              }
            }
          } else {
#pragma unroll
            for (int i = 0; i < kKeys; i++)
              x[i] = (i >= a && i <= b && ((mask >> (i / kBlock)) & 1u)) ? x[i] * sc : -INFINITY;
          }
        }
        float pm[8];
#pragma unroll
        for (int j = 0; j < 8; j++) pm[j] = fmaxf(x[j], x[j + 8]);
#pragma unroll
        for (int k16 = 1; k16 < kKeys / 16; k16++)
#pragma unroll
          for (int j = 0; j < 8; j++) pm[j] = fmax3(pm[j], x[16 * k16 + j], x[16 * k16 + 8 + j]);
        float mt = fmax3(fmax3(pm[0], pm[1], pm[2]), fmax3(pm[3], pm[4], pm[5]), fmaxf(pm[6], pm[7]));
        if (raw) mt *= sc;
        // lazy rescale: only when this row's maximum grew by more than 2^8 (O is
        // scaled below, once the scores are no longer held in registers)
        const bool need = mt > m_used + kLazyRescale;
        const bool rescale = __any_sync(0xffffffffu, need);
        float factor = 1.0f;
        if (rescale) {
          const float m_new = need ? mt : m_used;
          factor = need ? fast_exp2(m_used - m_new) : 1.0f;
          l *= factor;
          m_used = m_new;
        }
        // raw scores (-inf where masked) take the scale in one FFMA, prescaled
        // ones (sm_scale <= 0) do not; pairs of keys share one packed FMA and one
        // packed add into four pairs of partial sums
        const unsigned long long mul2 = f2pack(raw ? sc : 1.0f, raw ? sc : 1.0f);
        const unsigned long long sub2 = f2pack(-m_used, -m_used);
        unsigned long long acc[4] = {0ull, 0ull, 0ull, 0ull};
        uint32_t pk[kKeys / 2];
#pragma unroll
        for (int i = 0; i < kKeys; i += 2) {
          float a0, a1;
          f2unpack(ffma2(f2pack(x[i], x[i + 1]), mul2, sub2), a0, a1);
          const float e0 = fast_exp2(a0), e1 = fast_exp2(a1);
          acc[(i / 2) & 3] = fadd2(acc[(i / 2) & 3], f2pack(e0, e1));
          pk[i / 2] = pack2<BF>(e0, e1);
        }
        {
          float sp[8];
#pragma unroll
          for (int j = 0; j < 4; j++) f2unpack(acc[j], sp[2 * j], sp[2 * j + 1]);
          l += ((sp[0] + sp[1]) + (sp[2] + sp[3])) + ((sp[4] + sp[5]) + (sp[6] + sp[7]));
        }
        // P over the first 64 columns of S (this thread's S values are all read)
        tmem_st64(lane_base + LY::kSCol, pk);
        if (rescale && t > (KS ? 1 : 0)) {
          // O holds this item's earlier tiles (their P V is complete): scale it in place
#pragma unroll
          for (int c0 = 0; c0 < D; c0 += 32) {
            float v[32];
            tmem_ld32(lane_base + LY::kOCol + c0, v);
#pragma unroll
            for (int i = 0; i < 32; i++) v[i] *= factor;
            tmem_st32(lane_base + LY::kOCol + c0, v);
          }
        }
        // unwritten slots past L-1 in a loaded block: zero their V rows, so that
        // 0 * V stays 0 (query tile 0's warps; the MMA warp waits for both tiles' P)
        if ((KS || q == 0) && tail_rows != 0 && tail_blk >= blk0 &&
            tail_blk < blk0 + kTileBlocks && ((mask >> (tail_blk - blk0)) & 1u)) {
          if (!mbar_wait(&v_full[g % VS], (g / VS) & 1)) {
            timed_out = true;
            break;
          }
          zero_v_tail<LY>(smem + LY::v_off(g % VS),
                          (tail_blk - blk0) * kBlock, tail_rows, stid);
        }
        fence_before();
        mbar_arrive(&p_full[q]);
      }
      if (timed_out) break;
      items.fetch(p, num_pairs, smem);  // the next item's lengths load during the epilogue
      if constexpr (KS) {
        if (q == 1) {
          // slot 1, if it had tiles: hand (m, l) to slot 0, which reads O_1; the
          // next item's first P V into O_1 waits for this slot's next P
          if (two) {
            // O_1 / l_1 in place, and its weight log2(l_1) + m_1 for slot 0
            if (!mbar_wait(&pv_done[1], (cq - 1) & 1)) {
              timed_out = true;
              break;
            }
            fence_after();
            {
              // the whole warp takes part in the tensor-memory copies (they are
              // .sync.aligned); a row without weight is scaled by 0 and slot 0
              // leaves it out by its weight
              const float inv1 = l > 0.0f ? 1.0f / l : 0.0f;
#pragma unroll
              for (int c0 = 0; c0 < D; c0 += 32) {
                float v[32];
                tmem_ld32(lane_base + LY::kOCol + c0, v);
#pragma unroll
                for (int i = 0; i < 32; i++) v[i] *= inv1;
                tmem_st32(lane_base + LY::kOCol + c0, v);
              }
            }
            xch[row] = l > 0.0f ? m_used + __log2f(l) : kNoMax;
            fence_before();
            mbar_arrive(merge_ready);
            if (!mbar_wait(merge_done, kk & 1)) {
              timed_out = true;
              break;
            }
            kk++;
          }
          continue;
        }
        c1 += it.ntiles / 2;
        // slot 0: both slots' last P V, then O = (O_0 2^(m_0 - M) + O_1 2^(m_1 - M)) /
        // (l_0 2^(m_0 - M) + l_1 2^(m_1 - M)), a slot without weight left out
        if (!mbar_wait(&pv_done[0], (cq - 1) & 1) ||
            (two && (!mbar_wait(merge_ready, kk & 1) || !mbar_wait(&pv_done[1], (c1 - 1) & 1)))) {
          timed_out = true;
          break;
        }
        fence_after();
        // slot 1 left O_1 / l_1 and lam = log2(l_1) + m_1 (kNoMax: no weight), so
        // O = (O_0 2^(m_0 - M) + (O_1 / l_1) 2^(lam - M)) / (l_0 2^(m_0 - M) + 2^(lam - M))
        const float lam = two ? xch[row] : kNoMax;
        const bool has1 = lam > 0.5f * kNoMax;
        const float mM = fmaxf(l > 0.0f ? m_used : kNoMax, has1 ? lam : kNoMax);
        const float f0 = l > 0.0f ? fast_exp2(m_used - mM) : 0.0f;
        const float f1 = has1 ? fast_exp2(lam - mM) : 0.0f;
        const float lt = l * f0 + f1;
        const float inv = lt > 0.0f ? 1.0f / lt : 0.0f;
        const float w0 = f0 * inv, w1 = f1 * inv;
        const uint32_t lane_base1 = lane_base + LY::kTileCols;  // slot 1, the same lanes
#pragma unroll
        for (int c0 = 0; c0 < D; c0 += 16) {
          float v[16], v1[16];
          tmem_ld16(lane_base + LY::kOCol + c0, v);
          if (two) tmem_ld16(lane_base1 + LY::kOCol + c0, v1);
          if (rvalid) {
            float w[16];
#pragma unroll
            for (int i = 0; i < 16; i++) {
              const float a0 = l > 0.0f ? v[i] * w0 : 0.0f;
              const float a1 = has1 ? v1[i] * w1 : 0.0f;
              w[i] = a0 + a1;
            }
#pragma unroll
            for (int u = 0; u < 2; u++) {
              uint4 o4;
              o4.x = pack2<BF>(w[8 * u + 0], w[8 * u + 1]);
              o4.y = pack2<BF>(w[8 * u + 2], w[8 * u + 3]);
              o4.z = pack2<BF>(w[8 * u + 4], w[8 * u + 5]);
              o4.w = pack2<BF>(w[8 * u + 6], w[8 * u + 7]);
              *reinterpret_cast<uint4*>(dst + c0 + 8 * u) = o4;
            }
          }
        }
        fence_before();  // O's reads are ordered before the next item's first P V
        if (two) {
          mbar_arrive(merge_done);
          kk++;
        }
        continue;
      }
      // epilogue: wait for this item's last P V (tile g-1)
      if (!mbar_wait(&pv_done[q], (g - 1) & 1)) {
        timed_out = true;
        break;
      }
      fence_after();
      const float inv = l > 0.0f ? 1.0f / l : 0.0f;
#pragma unroll
      for (int c0 = 0; c0 < D; c0 += 32) {
        float v[32];
        tmem_ld32(lane_base + LY::kOCol + c0, v);
        if (rvalid) {
#pragma unroll
          for (int u = 0; u < 4; u++) {
            float w[8];
#pragma unroll
            for (int i = 0; i < 8; i++) w[i] = l > 0.0f ? v[8 * u + i] * inv : 0.0f;
            uint4 o4;
            o4.x = pack2<BF>(w[0], w[1]);
            o4.y = pack2<BF>(w[2], w[3]);
            o4.z = pack2<BF>(w[4], w[5]);
            o4.w = pack2<BF>(w[6], w[7]);
            *reinterpret_cast<uint4*>(dst + c0 + 8 * u) = o4;
          }
        }
      }
      fence_before();  // O's reads are ordered before the next item's first P V
    }
    if (timed_out && lane == 0) set_flag(p.err, PA_FLAG_TIMEOUT);
  }
  fence_before();
  __syncthreads();
  fence_after();
  if (warp == 1)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(LY::kTmemCols));
}

}  // namespace tc

namespace {

int sm_count() {
  static int count[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  if (count[dev] == 0 &&
      cudaDeviceGetAttribute(&count[dev], cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    count[dev] = 0;
  return count[dev];
}

// Q as a 3-D tensor map [tokens][q heads][head_dim] whose box is one query tile:
// 128/G tokens x G heads x 64 columns (128-byte swizzle).  Possible when G
// divides 128 and the strides are multiples of 16 bytes.
bool encode_q_map(CUtensorMap* m, const AttnParams& p, int D, bool bf16) {
  if (tc::kRows % p.group != 0 || !pa_internal::aligned16(p.q)) return false;
  pa_internal::EncodeTiledFn fn = pa_internal::encode_tiled_fn();
  if (!fn || p.num_q_tokens <= 0) return false;
  const cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)p.num_q_heads,
                              (cuuint64_t)p.num_q_tokens};
  const cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)p.num_q_heads * D * 2};
  const cuuint32_t box[3] = {64, (cuuint32_t)p.group, (cuuint32_t)(tc::kRows / p.group)};
  const cuuint32_t estr[3] = {1, 1, 1};
  return fn(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3,
            const_cast<void*>(p.q), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

template <int D, typename QT, bool KS>
cudaError_t launch_prefill_tc_ks(const AttnParams& p, const CUtensorMap& tmk,
                                 const CUtensorMap& tmv, int num_seqs, cudaStream_t stream) {
  constexpr int smem = tc::Layout<D>::kBytes;
  auto kern = tc::pa_prefill_tc_kernel<D, QT, KS>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  // setmaxnreg moves registers between warpgroups inside the CTA's launch
  // allocation; an increase beyond it would wait forever, so the compiled
  // register count must cover the split before anything is launched
  cudaFuncAttributes fa;
  e = cudaFuncGetAttributes(&fa, kern);
  if (e != cudaSuccess) return e;
  if ((long long)fa.numRegs * tc::kThreads <
      128LL * tc::kCtlRegs + (long long)tc::kQTiles * tc::kSoftmaxThreads * tc::kSoftmaxRegs)
    return cudaErrorInvalidConfiguration;
  AttnParams pt = p;
  pt.q_tiles = (int)(((long long)p.max_q_len * p.group + tc::kCtaRows - 1) / tc::kCtaRows);
  const long long items = (long long)pt.q_tiles * pt.num_kv_heads * num_seqs;
  if (items <= 0) return cudaSuccess;
  if (items > 0x7fffffffLL) return cudaErrorInvalidValue;
  CUtensorMap tmq;
  memset(&tmq, 0, sizeof(tmq));
  const bool q_tma = encode_q_map(&tmq, pt, D, std::is_same<QT, __nv_bfloat16>::value);
  const int sms = sm_count();
  if (sms <= 0) return cudaErrorInvalidDevice;
  const unsigned grid = (unsigned)std::min<long long>(items, sms);
  return pa_internal::launch_dependent(kern, dim3(grid), dim3(tc::kThreads), smem, stream, 1u, pt,
                                       tmk, tmv, tmq, num_seqs, q_tma ? 1 : 0);
}

// Chunks of at most 128 query rows (a few queries per sequence, e.g. a draft
// verification) take the key-split kernel: one query tile's rows in both slots.
template <int D, typename QT>
cudaError_t launch_prefill_tc(const AttnParams& p, const CUtensorMap& tmk,
                              const CUtensorMap& tmv, int num_seqs, cudaStream_t stream) {
  if ((long long)p.max_q_len * p.group <= tc::kRows)
    return launch_prefill_tc_ks<D, QT, true>(p, tmk, tmv, num_seqs, stream);
  return launch_prefill_tc_ks<D, QT, false>(p, tmk, tmv, num_seqs, stream);
}

template cudaError_t launch_prefill_tc<64, __half>(const AttnParams&, const CUtensorMap&,
                                                   const CUtensorMap&, int, cudaStream_t);
template cudaError_t launch_prefill_tc<128, __half>(const AttnParams&, const CUtensorMap&,
                                                    const CUtensorMap&, int, cudaStream_t);
template cudaError_t launch_prefill_tc<64, __nv_bfloat16>(const AttnParams&, const CUtensorMap&,
                                                          const CUtensorMap&, int, cudaStream_t);
template cudaError_t launch_prefill_tc<128, __nv_bfloat16>(const AttnParams&, const CUtensorMap&,
                                                           const CUtensorMap&, int, cudaStream_t);

}  // namespace pa_dev
