// pa_prefill_tc.cu -- chunked-prefill attention on the 5th-generation tensor
// cores (tcgen05.mma, accumulators in tensor memory) for fp16/bf16 caches
// ("PyTorch LLM Serving Engine", "What is implemented": chunked prefill; "Loading":
// online softmax while walking the block table).
//
// A CTA owns 256 query rows (two tiles of 128) of one sequence's chunk and one
// kv head: row R = c*G + j is query token c, query head kvh*G + j.  The keys the
// rows can see are walked in tiles of 64 (four 16-token blocks), each tile used
// by both query tiles:
//   S_t  = Q K_t^T      tcgen05.mma M=128 N=64  K=head_dim -> TMEM (two buffers)
//   P_t  = exp2(S_t*scale - m)   one softmax thread per row, written to shared
//                                memory as f16/bf16 in the MMA's K-major layout
//   O   += P_t V_t      tcgen05.mma M=128 N=head_dim K=64 -> TMEM
// Warps: 0 = TMA producer (paged K/V tiles into a ring of stages), 1 = MMA
// issuer (the warp runs the schedule, one elected lane issues) and tensor-memory
// owner, 2..5 and 6..9 = softmax for query
// tiles 0 and 1, one TMEM lane (row) per thread; the two softmax warpgroups run
// in parallel, so one tile's exponentials overlap the other tile's MMAs.  The
// running maximum is rescaled lazily: O (in TMEM) and the normaliser are only
// rescaled when a row's maximum grows by more than 2^8, so the exponentials stay
// below 256.  A parity wait only tells a barrier's current phase from the one
// before, so every barrier is waited on at every phase, in order; every wait is
// bounded.
#include <algorithm>

#include "pa_attn_common.cuh"
#include "pa_internal.h"

namespace pa_dev {
namespace tc {

constexpr int kRows = 128;      // query rows per tile (MMA M)
constexpr int kQTiles = 2;      // query tiles per CTA
constexpr int kCtaRows = kQTiles * kRows;
constexpr int kKeys = 64;       // keys per tile (MMA N of S, K of P V)
constexpr int kTileBlocks = kKeys / kBlock;
constexpr int kNS = 3;          // K/V stages
constexpr int kSoftmaxThreads = 128;  // per query tile
constexpr int kThreads = 64 + kQTiles * kSoftmaxThreads;  // 10 warps
constexpr float kLazyRescale = 8.0f;  // log2 of the growth that forces a rescale
constexpr float kNoMax = -1.0e30f;    // running-maximum sentinel: 2^(-inf - kNoMax) = 0

template <int D>
struct Layout {
  static constexpr int kChunks = D / 64;               // 128-byte chunks of a row
  static constexpr int kQBytes = kRows * D * 2;        // per tile: [chunk][128 rows][128 B]
  static constexpr int kKVChunk = kKeys * 128;         // one chunk of a K or V tile
  static constexpr int kKVBytes = kChunks * kKVChunk;  // [chunk][64 rows][128 B]
  static constexpr int kStageBytes = 2 * kKVBytes;     // K then V
  static constexpr int kPBytes = kRows * kKeys * 2;    // [128 rows][128 B]
  static constexpr int kQOff = 0;
  static constexpr int kStageOff = kQOff + kQTiles * kQBytes;
  static constexpr int kPOff = kStageOff + kNS * kStageBytes;  // [tile][buffer]
  static constexpr int kBarOff = kPOff + kQTiles * 2 * kPBytes;
  // barriers: kv_full[NS], kv_free[NS], q_full, then per query tile s_full[2],
  // s_free[2], p_full[2], p_free[2]
  static constexpr int kTileBars = 8;
  static constexpr int kNumBars = 2 * kNS + 1 + kQTiles * kTileBars;
  static constexpr int kFlagOff = kBarOff + kNumBars * 8;  // valid flags [NS][4] ints
  static constexpr int kTmemSlotOff = kFlagOff + kNS * kTileBlocks * 4;
  static constexpr int kUsed = kTmemSlotOff + 16;
  static constexpr int kBytes = kUsed + 1024;  // room to align the base to 1024
  // tensor memory columns per query tile: S buffers 0/1, then O
  static constexpr uint32_t kSCol0 = 0, kSCol1 = kKeys, kOCol = 2 * kKeys;
  static constexpr uint32_t kTileCols = 256;
  static constexpr uint32_t kTmemCols = kQTiles * kTileCols;
  static_assert(kOCol + D <= kTileCols, "tensor memory budget");
  static_assert(kBytes <= 232448, "shared memory budget");
};

struct TileBars {
  uint64_t *s_full, *s_free, *p_full, *p_free;
};

__device__ __forceinline__ TileBars tile_bars(uint64_t* base) {
  TileBars b;
  b.s_full = base;
  b.s_free = base + 2;
  b.p_full = base + 4;
  b.p_free = base + 6;
  return b;
}

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

__device__ __forceinline__ void commit_elect(uint64_t* bar) {
  asm volatile(
      "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(
          smem_u32(bar))
      : "memory");
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

// 32 consecutive fp32 columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
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
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 32; i++) v[i] = __uint_as_float(r[i]);
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

// Byte offset of 16-byte unit u (0..7) of row r in a 128-byte-row swizzled chunk.
__device__ __forceinline__ uint32_t sw_unit(int r, int u) {
  return (uint32_t)(r * 128 + (((u ^ r) & 7) << 4));
}

template <int D, typename QT>
__global__ void __launch_bounds__(kThreads, 1)
    pa_prefill_tc_kernel(const __grid_constant__ AttnParams p,
                         const __grid_constant__ CUtensorMap tmk,
                         const __grid_constant__ CUtensorMap tmv) {
  using LY = Layout<D>;
  constexpr bool BF = std::is_same<QT, __nv_bfloat16>::value;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + LY::kBarOff);
  uint64_t* kv_full = bars;
  uint64_t* kv_free = bars + kNS;
  uint64_t* q_full = bars + 2 * kNS;
  uint64_t* tbar0 = q_full + 1;  // per-tile barriers follow
  int* vflags = reinterpret_cast<int*>(smem + LY::kFlagOff);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + LY::kTmemSlotOff);

  const int n = blockIdx.y;
  const int tile = blockIdx.x % p.q_tiles;
  const int kvh = blockIdx.x / p.q_tiles;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = p.group;
  const bool reporter = threadIdx.x == 0 && blockIdx.x == 0;

  const int q0 = p.cu_q_lens[n], q1 = p.cu_q_lens[n + 1];
  if (q0 < 0 || q1 < q0 || q1 > p.num_q_tokens) {
    if (reporter) set_flag(p.err, PA_FLAG_Q_LEN);
    return;
  }
  int C = q1 - q0;
  if (C > p.max_q_len) {
    if (reporter) set_flag(p.err, PA_FLAG_Q_LEN);
    C = p.max_q_len;
  }
  const int L = clamp_context(p, n, reporter);
  if (C > L && reporter) set_flag(p.err, PA_FLAG_Q_LEN);
  const int R0 = tile * kCtaRows;
  const int nrows = C * G;
  if (R0 >= nrows) return;
  const int c_first = R0 / G;
  const int c_last = (min(R0 + kCtaRows, nrows) - 1) / G;
  const int hi_u = L - C + c_last;
  const int lo_u = p.window > 0 ? max(0, L - C + c_first - p.window + 1) : 0;
  const int first = lo_u / kBlock;
  const int last = hi_u / kBlock;
  const int ntiles = hi_u >= lo_u ? (last - first) / kTileBlocks + 1 : 0;
  QT* out = static_cast<QT*>(p.out);
  if (ntiles == 0) {  // no row sees a key: zeros
    for (int idx = threadIdx.x; idx < kCtaRows * D; idx += kThreads) {
      const int R = R0 + idx / D;
      if (R < nrows)
        out[((long long)(q0 + R / G) * p.num_q_heads + kvh * G + R % G) * D + idx % D] =
            to_out<QT>(0.0f);
    }
    return;
  }

  if (threadIdx.x == 0) {
    for (int i = 0; i < kNS; i++) {
      mbar_init(&kv_full[i], 1);
      mbar_init(&kv_free[i], 1);
    }
    mbar_init(q_full, kQTiles * kSoftmaxThreads);
    for (int q = 0; q < kQTiles; q++) {
      const TileBars tb = tile_bars(tbar0 + q * LY::kTileBars);
      for (int i = 0; i < 2; i++) {
        mbar_init(&tb.s_full[i], 1);
        mbar_init(&tb.s_free[i], kSoftmaxThreads);
        mbar_init(&tb.p_full[i], kSoftmaxThreads);
        mbar_init(&tb.p_free[i], 1);
      }
    }
    fence_mbar_init();
  }
  if (warp == 1) {  // tensor memory: per query tile, S (2 x 64 columns) and O
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(tmem_slot)),
                 "r"(LY::kTmemCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  fence_before();
  __syncthreads();
  fence_after();
  const uint32_t tmem = *tmem_slot;
  bool timed_out = false;

  if (warp == 0) {
    // ---------------- producer: K/V tiles of four blocks each
    const int32_t* table = p.block_tables + (long long)n * p.max_blocks_per_seq + first;
    const int nblk = last - first + 1;
    // block ids, 32 at a time: lane l holds entry 32*k + l of batch k; batch k+1
    // is loaded while batch k is used, so the table's latency stays off the path
    constexpr int kTilesPerBatch = 32 / kTileBlocks;
    auto batch = [&](int k) { return 32 * k + lane < nblk ? table[32 * k + lane] : -1; };
    int ids = batch(0), ids_next = batch(1);
    int issued = 0;
    for (int t = 0; t < ntiles && !timed_out; t++, issued++) {
      const int st = t % kNS;
      if (t > 0 && t % kTilesPerBatch == 0) {
        ids = ids_next;
        ids_next = batch(t / kTilesPerBatch + 1);
      }
      const int from = __shfl_sync(0xffffffffu, ids, (kTileBlocks * t + lane) & 31);
      const bool inside = lane < kTileBlocks && kTileBlocks * t + lane < nblk;
      const int mine = inside ? from : -1;
      const bool ok = inside && mine >= 0 && mine < p.num_blocks;
      if (t >= kNS && !mbar_wait(&kv_free[st], ((t / kNS) - 1) & 1)) {
        timed_out = true;
        break;
      }
      if (lane < kTileBlocks) {
        vflags[st * kTileBlocks + lane] = ok ? 1 : 0;
        if (inside && !ok) set_flag(p.err, PA_FLAG_BLOCK_ID);
      }
      __syncwarp();  // every lane's flag is written before lane 0 arms the stage
      const unsigned okmask = __ballot_sync(0xffffffffu, ok);
      if (lane == 0)
        mbar_arrive_expect_tx(&kv_full[st], __popc(okmask) * 2u * LY::kKVBytes / kTileBlocks);
      __syncwarp();
      if (ok) {
        uint8_t* kbase = smem + LY::kStageOff + st * LY::kStageBytes;
        uint8_t* vbase = kbase + LY::kKVBytes;
        const int row0 = (mine * p.num_kv_heads + kvh) * kBlock;
#pragma unroll
        for (int h = 0; h < LY::kChunks; h++) {
          tma_load_2d(kbase + h * LY::kKVChunk + lane * kBlock * 128, &tmk, 64 * h, row0,
                      &kv_full[st]);
          tma_load_2d(vbase + h * LY::kKVChunk + lane * kBlock * 128, &tmv, 64 * h, row0,
                      &kv_full[st]);
        }
      }
    }
    // no copy may still be landing in shared memory when the CTA exits; the last
    // kNS tiles issued are their stages' current phases
    if (lane == 0)
      for (int t = issued > kNS ? issued - kNS : 0; t < issued; t++)
        if (!mbar_wait(&kv_full[t % kNS], (t / kNS) & 1)) break;
    if (timed_out && lane == 0) set_flag(p.err, PA_FLAG_TIMEOUT);
  } else if (warp == 1) {
    // ---------------- MMA issuer (the whole warp; one elected lane issues)
    {
      const uint32_t idS = idesc<BF>(kRows, kKeys, false);
      const uint32_t idO = idesc<BF>(kRows, D, true);
      auto pv = [&](int q, int t) -> bool {  // O_q += P_{q,t} V_t
        const TileBars tb = tile_bars(tbar0 + q * LY::kTileBars);
        if (!warp_wait(&tb.p_full[t & 1], (t >> 1) & 1)) return false;
        fence_after();
        const uint32_t sP = smem_u32(smem + LY::kPOff + (2 * q + (t & 1)) * LY::kPBytes);
        const uint32_t sV = smem_u32(smem + LY::kStageOff + (t % kNS) * LY::kStageBytes) +
                            LY::kKVBytes;
        const uint32_t dO = tmem + q * LY::kTileCols + LY::kOCol;
#pragma unroll
        for (int s = 0; s < kKeys / 16; s++)
          mma_elect(dO, sw128_desc(sP + 32 * s, 16, 1024),
                    sw128_desc(sV + 2048 * s, LY::kKVChunk, 1024), idO, (t > 0 || s > 0) ? 1u : 0u);
        commit_elect(&tb.p_free[t & 1]);
        return true;
      };
      bool ok = warp_wait(q_full, 0);
      for (int t = 0; t < ntiles && ok; t++) {
        const int st = t % kNS;
        ok = warp_wait(&kv_full[st], (t / kNS) & 1);
        const uint32_t sK = smem_u32(smem + LY::kStageOff + st * LY::kStageBytes);
        for (int q = 0; q < kQTiles && ok; q++) {
          const TileBars tb = tile_bars(tbar0 + q * LY::kTileBars);
          if (t >= 2) ok = warp_wait(&tb.s_free[t & 1], ((t - 2) >> 1) & 1);
          if (!ok) break;
          fence_after();
          const uint32_t sQ = smem_u32(smem + LY::kQOff + q * LY::kQBytes);
          const uint32_t dS = tmem + q * LY::kTileCols + ((t & 1) ? LY::kSCol1 : LY::kSCol0);
#pragma unroll
          for (int s = 0; s < D / 16; s++)
            mma_elect(dS, sw128_desc(sQ + (s / 4) * (kRows * 128) + (s % 4) * 32, 16, 1024),
                      sw128_desc(sK + (s / 4) * LY::kKVChunk + (s % 4) * 32, 16, 1024), idS,
                      s > 0 ? 1u : 0u);
          commit_elect(&tb.s_full[t & 1]);
        }
        if (ok && t >= 1) {
          for (int q = 0; q < kQTiles && ok; q++) ok = pv(q, t - 1);
          if (ok) commit_elect(&kv_free[(t - 1) % kNS]);
        }
      }
      if (ok) {
        for (int q = 0; q < kQTiles && ok; q++) ok = pv(q, ntiles - 1);
        if (ok) commit_elect(&kv_free[(ntiles - 1) % kNS]);
      }
      if (!ok && lane == 0) set_flag(p.err, PA_FLAG_TIMEOUT);
    }
    __syncwarp();
  } else {
    // ---------------- softmax: query tile q, thread <-> row (TMEM lane 32*(warp%4) + lane)
    const int q = (warp - 2) / 4;
    const TileBars tb = tile_bars(tbar0 + q * LY::kTileBars);
    const int stid = threadIdx.x - 64 - q * kSoftmaxThreads;  // 0..127 within the tile
    const int row = 32 * (warp & 3) + lane;
    const int R = R0 + q * kRows + row;
    const bool rvalid = R < nrows;
    const int c = rvalid ? R / G : 0;
    const int pos = L - C + c;
    const int row_hi = rvalid ? pos : -1;
    const int row_lo = p.window > 0 ? max(0, pos - p.window + 1) : 0;
    const long long orow = (long long)(q0 + c) * p.num_q_heads + kvh * G + (rvalid ? R % G : 0);
    const uint32_t lane_base = tmem + q * LY::kTileCols + ((uint32_t)(32 * (warp & 3)) << 16);
    const float sc = p.scale_log2;

    // Q row -> shared memory in the MMA's swizzled K-major layout
    {
      const uint4* src = reinterpret_cast<const uint4*>(static_cast<const QT*>(p.q) + orow * D);
      uint8_t* qt = smem + LY::kQOff + q * LY::kQBytes;
#pragma unroll
      for (int u = 0; u < D / 8; u++) {
        const uint4 v = rvalid ? src[u] : make_uint4(0, 0, 0, 0);
        *reinterpret_cast<uint4*>(qt + (u / 8) * (kRows * 128) + sw_unit(row, u % 8)) = v;
      }
      fence_proxy_async();
      mbar_arrive(q_full);
    }

    // p_free[b] completes when the P V that read P buffer b has finished, and
    // with it every earlier MMA.  Tile t waits on it for the P V of tile t-1
    // (buffer (t-1)&1) before rescaling O, and for the P V of tile t-2 (buffer
    // t&1) before writing P.  Per buffer these are successive phases, and a
    // repeated wait on the same phase is safe: the next one needs this tile's P.
    float m_used = kNoMax, l = 0.0f;
    for (int t = 0; t < ntiles; t++) {
      if (!mbar_wait(&tb.s_full[t & 1], (t >> 1) & 1)) {
        timed_out = true;
        break;
      }
      fence_after();
      const int pos0 = (first + kTileBlocks * t) * kBlock;
      const int* vf = vflags + (t % kNS) * kTileBlocks;
      const bool blocks_ok = vf[0] && vf[1] && vf[2] && vf[3];
      float x[kKeys];
      {
        float v[32];
        const uint32_t scol = (t & 1) ? LY::kSCol1 : LY::kSCol0;
        tmem_ld32(lane_base + scol, v);
#pragma unroll
        for (int i = 0; i < 32; i++) x[i] = v[i];
        tmem_ld32(lane_base + scol + 32, v);
#pragma unroll
        for (int i = 0; i < 32; i++) x[32 + i] = v[i];
      }
      fence_before();
      mbar_arrive(&tb.s_free[t & 1]);  // the MMA may overwrite this S buffer now
      // maximum of the scaled scores this row can see; an inner tile (every key
      // visible to every row of the warp) skips the masks.  Eight partial maxima
      // and sums keep the dependency chains short.
      float part[8];
      const bool inner = __all_sync(0xffffffffu, blocks_ok && pos0 >= row_lo &&
                                                     pos0 + kKeys - 1 <= row_hi) &&
                         sc > 0.0f;
      if (inner) {
#pragma unroll
        for (int j = 0; j < 8; j++) part[j] = x[j];
#pragma unroll
        for (int i = 8; i < kKeys; i++) part[i & 7] = fmaxf(part[i & 7], x[i]);
      } else {
#pragma unroll
        for (int j = 0; j < 8; j++) part[j] = -INFINITY;
#pragma unroll
        for (int i = 0; i < kKeys; i++) {
          const int kp = pos0 + i;
          const bool vis = kp >= row_lo && kp <= row_hi && vf[i / kBlock];
          x[i] = vis ? x[i] * sc : -INFINITY;
          part[i & 7] = fmaxf(part[i & 7], x[i]);
        }
      }
      float mt = fmaxf(fmaxf(fmaxf(part[0], part[1]), fmaxf(part[2], part[3])),
                       fmaxf(fmaxf(part[4], part[5]), fmaxf(part[6], part[7])));
      if (inner) mt *= sc;
      // lazy rescale: only when this row's maximum grew by more than 2^8
      const bool need = mt > m_used + kLazyRescale;
      if (__any_sync(0xffffffffu, need)) {
        const float m_new = need ? mt : m_used;
        const float factor = need ? fast_exp2(m_used - m_new) : 1.0f;
        if (t > 0) {  // O holds tiles < t: wait for the last P V, then scale it in place
          if (!mbar_wait(&tb.p_free[(t - 1) & 1], ((t - 1) >> 1) & 1)) {
            timed_out = true;
            break;
          }
          fence_after();
#pragma unroll
          for (int c0 = 0; c0 < D; c0 += 32) {
            float v[32];
            tmem_ld32(lane_base + LY::kOCol + c0, v);
#pragma unroll
            for (int i = 0; i < 32; i++) v[i] *= factor;
            tmem_st32(lane_base + LY::kOCol + c0, v);
          }
        }
        l *= factor;
        m_used = m_new;
      }
      // inner tiles hold raw scores (the scale is folded into one FFMA), edge
      // tiles already-scaled ones (-inf where masked)
      const float mul = inner ? sc : 1.0f;
      const float sub = -m_used;
#pragma unroll
      for (int j = 0; j < 8; j++) part[j] = 0.0f;
#pragma unroll
      for (int i = 0; i < kKeys; i++) {
        x[i] = fast_exp2(fmaf(x[i], mul, sub));
        part[i & 7] += x[i];
      }
      l += ((part[0] + part[1]) + (part[2] + part[3])) + ((part[4] + part[5]) + (part[6] + part[7]));
      // P buffer t&1 was last read by the P V of tile t-2
      if (t >= 2 && !mbar_wait(&tb.p_free[t & 1], ((t - 2) >> 1) & 1)) {
        timed_out = true;
        break;
      }
      // P row -> shared memory (f16/bf16, K-major swizzled)
      uint8_t* prow = smem + LY::kPOff + (2 * q + (t & 1)) * LY::kPBytes;
#pragma unroll
      for (int u = 0; u < kKeys / 8; u++) {
        uint4 pk;
        pk.x = pack2<BF>(x[8 * u + 0], x[8 * u + 1]);
        pk.y = pack2<BF>(x[8 * u + 2], x[8 * u + 3]);
        pk.z = pack2<BF>(x[8 * u + 4], x[8 * u + 5]);
        pk.w = pack2<BF>(x[8 * u + 6], x[8 * u + 7]);
        *reinterpret_cast<uint4*>(prow + sw_unit(row, u)) = pk;
      }
      // V rows of keys no row can see (before the window, past the context,
      // blocks not in the pool) may hold garbage: zero them so 0 * V stays 0.
      // Both query tiles read the stage; tile 0's warps clear it, and the MMA
      // thread waits for tile 0's P before either tile's P V.
      const bool edge = pos0 < lo_u || pos0 + kKeys - 1 > hi_u || !blocks_ok;
      if (edge && q == 0) {
        uint8_t* vbase = smem + LY::kStageOff + (t % kNS) * LY::kStageBytes + LY::kKVBytes;
        for (int idx = stid; idx < kKeys * LY::kChunks * 8; idx += kSoftmaxThreads) {
          const int key = idx / (LY::kChunks * 8);
          const int rest = idx % (LY::kChunks * 8);
          const int kp = pos0 + key;
          if (kp < lo_u || kp > hi_u || !vf[key / kBlock])
            *reinterpret_cast<uint4*>(vbase + (rest / 8) * LY::kKVChunk + sw_unit(key, rest % 8)) =
                make_uint4(0, 0, 0, 0);
        }
      }
      fence_proxy_async();
      fence_before();
      mbar_arrive(&tb.p_full[t & 1]);
    }
    // epilogue: wait for the last P V
    if (!timed_out && mbar_wait(&tb.p_free[(ntiles - 1) & 1], ((ntiles - 1) >> 1) & 1)) {
      fence_after();
      const float inv = l > 0.0f ? 1.0f / l : 0.0f;
      QT* dst = out + orow * D;
#pragma unroll
      for (int c0 = 0; c0 < D; c0 += 32) {
        float v[32];
        tmem_ld32(lane_base + LY::kOCol + c0, v);
        if (rvalid) {
#pragma unroll
          for (int u = 0; u < 4; u++) {
            uint4 pk;
            pk.x = pack2<BF>(v[8 * u + 0] * inv, v[8 * u + 1] * inv);
            pk.y = pack2<BF>(v[8 * u + 2] * inv, v[8 * u + 3] * inv);
            pk.z = pack2<BF>(v[8 * u + 4] * inv, v[8 * u + 5] * inv);
            pk.w = pack2<BF>(v[8 * u + 6] * inv, v[8 * u + 7] * inv);
            *reinterpret_cast<uint4*>(dst + c0 + 8 * u) = pk;
          }
        }
      }
    } else {
      timed_out = true;
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

template <int D, typename QT>
cudaError_t launch_prefill_tc(const AttnParams& p, const CUtensorMap& tmk,
                              const CUtensorMap& tmv, int num_seqs, cudaStream_t stream) {
  constexpr int smem = tc::Layout<D>::kBytes;
  auto kern = tc::pa_prefill_tc_kernel<D, QT>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  AttnParams pt = p;
  pt.q_tiles = (int)(((long long)p.max_q_len * p.group + tc::kCtaRows - 1) / tc::kCtaRows);
  const dim3 grid((unsigned)(pt.q_tiles * pt.num_kv_heads), (unsigned)num_seqs);
  kern<<<grid, tc::kThreads, smem, stream>>>(pt, tmk, tmv);
  return cudaGetLastError();
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
