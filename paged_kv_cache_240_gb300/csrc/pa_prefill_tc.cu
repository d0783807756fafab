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
#include <cstring>
#include <type_traits>

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
constexpr int kMaxPlan = 512;         // (sequence, tile) pairs the CTA orders by cost
constexpr int kItemCost = 2;          // per-item overhead, in key tiles

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
  // barriers: kv_full[NS], kv_free[NS], q_full, q_free, then per query tile
  // s_full[2], s_free[2], p_full[2], p_free[2]
  static constexpr int kTileBars = 8;
  static constexpr int kNumBars = 2 * kNS + 2 + kQTiles * kTileBars;
  static constexpr int kFlagOff = kBarOff + kNumBars * 8;  // valid flags [NS][4] ints
  static constexpr int kTmemSlotOff = kFlagOff + kNS * kTileBlocks * 4;
  static constexpr int kOrderOff = kTmemSlotOff + 16;  // work order [kMaxPlan] uint16
  static constexpr int kUsed = kOrderOff + kMaxPlan * 2;
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

// One work item: 256 query rows (two tiles) of one sequence's chunk and one kv
// head, and the key range those rows can see.
struct Item {
  bool valid;  // rows exist (a sequence whose chunk is shorter has fewer items)
  int n, kvh, q0, C, L, R0, nrows, lo_u, hi_u, first, ntiles;
};

__device__ __forceinline__ Item item_info(const AttnParams& p, int n, int kvh, int tile,
                                          bool report) {
  Item it;
  it.valid = false;
  it.ntiles = 0;
  it.n = n;
  it.kvh = kvh;
  report = report && kvh == 0 && tile == 0;  // one report per sequence
  const int q0 = p.cu_q_lens[it.n], q1 = p.cu_q_lens[it.n + 1];
  if (q0 < 0 || q1 < q0 || q1 > p.num_q_tokens) {
    if (report) set_flag(p.err, PA_FLAG_Q_LEN);
    return it;
  }
  int C = q1 - q0;
  if (C > p.max_q_len) {
    if (report) set_flag(p.err, PA_FLAG_Q_LEN);
    C = p.max_q_len;
  }
  const int L = clamp_context(p, it.n, report);
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

// The work list: items ordered by cost (key tiles + a fixed overhead), longest
// first, when the CTA could rank the (sequence, tile) pairs (every kv head of a
// pair costs the same); in (sequence, kv head, tile) order otherwise.  Round r
// of the list goes to the CTAs in alternating directions (CTA b takes position
// r*grid + b in even rounds, r*grid + grid-1-b in odd ones), so a CTA that drew
// a long item early draws a short one next.  Returns false past the end.
struct WorkList {
  const uint16_t* order;  // pair index by rank, or nullptr
  int num_pairs, kv_heads, q_tiles;

  __device__ __forceinline__ bool at(int j, int& n, int& kvh, int& tile) const {
    const int grid = gridDim.x, b = blockIdx.x;
    const long long s = (long long)j * grid + ((j & 1) ? grid - 1 - b : b);
    if (s >= (long long)num_pairs * kv_heads) return false;
    if (order) {
      const int pair = order[s / kv_heads];
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
};

// Persistent: each CTA walks its part of the work list.  Every role walks the
// same items; the tile counter g (and the item counter k for Q) runs on across
// items, so each barrier keeps stepping one phase at a time, and the next
// item's Q and first K/V tiles load while the current item's last tiles finish.
template <int D, typename QT>
__global__ void __launch_bounds__(kThreads, 1)
    pa_prefill_tc_kernel(const __grid_constant__ AttnParams p,
                         const __grid_constant__ CUtensorMap tmk,
                         const __grid_constant__ CUtensorMap tmv,
                         const __grid_constant__ CUtensorMap tmq, int num_seqs, int q_tma) {
  using LY = Layout<D>;
  constexpr bool BF = std::is_same<QT, __nv_bfloat16>::value;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + LY::kBarOff);
  uint64_t* kv_full = bars;
  uint64_t* kv_free = bars + kNS;
  uint64_t* q_full = bars + 2 * kNS;
  uint64_t* q_free = q_full + 1;
  uint64_t* tbar0 = q_full + 2;  // per-tile barriers follow
  int* vflags = reinterpret_cast<int*>(smem + LY::kFlagOff);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + LY::kTmemSlotOff);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = p.group;
  const bool reporter = threadIdx.x == 0;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kNS; i++) {
      mbar_init(&kv_full[i], 1);
      mbar_init(&kv_free[i], 1);
    }
    mbar_init(q_full, 32);  // the producer warp's lanes
    mbar_init(q_free, 1);
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
  // the work order (the P buffers serve as scratch: nothing has written them yet)
  WorkList wl;
  wl.num_pairs = num_seqs * p.q_tiles;
  wl.kv_heads = p.num_kv_heads;
  wl.q_tiles = p.q_tiles;
  wl.order = nullptr;
  if (wl.num_pairs <= kMaxPlan) {
    int* cost = reinterpret_cast<int*>(smem + LY::kPOff);
    uint16_t* order = reinterpret_cast<uint16_t*>(smem + LY::kOrderOff);
    for (int j = threadIdx.x; j < wl.num_pairs; j += kThreads) {
      const Item it = item_info(p, j / p.q_tiles, 0, j % p.q_tiles, false);
      cost[j] = it.valid ? it.ntiles + kItemCost : 0;
    }
    __syncthreads();
    for (int j = threadIdx.x; j < wl.num_pairs; j += kThreads) {
      const int cj = cost[j];
      int rank = 0;
      for (int i2 = 0; i2 < wl.num_pairs; i2++) {
        const int ci = cost[i2];
        rank += (ci > cj || (ci == cj && i2 < j)) ? 1 : 0;
      }
      order[rank] = (uint16_t)j;
    }
    wl.order = order;
  }
  fence_before();
  __syncthreads();
  fence_after();
  const uint32_t tmem = *tmem_slot;
  bool timed_out = false;

  if (warp == 0) {
    // ---------------- producer: each item's Q, then its K/V tiles of four blocks
    int g = 0, k = 0;  // tiles and items with tiles so far
    int n, kvh, tile;
    for (int j = 0; !timed_out && wl.at(j, n, kvh, tile); j++) {
      const Item it = item_info(p, n, kvh, tile, reporter);
      if (!it.valid || it.ntiles == 0) continue;
      // Q of this item, once the previous item's S MMAs have finished with it
      if (k > 0 && !warp_wait(q_free, (k - 1) & 1)) {
        timed_out = true;
        break;
      }
      uint8_t* qs = smem + LY::kQOff;
      if (q_tma) {
        // box [128/G tokens][G heads][64 columns] = 128 rows of the tile
        if (lane == 0) mbar_arrive_expect_tx(q_full, kQTiles * LY::kQBytes);
        __syncwarp();
        if (lane < kQTiles * LY::kChunks) {
          const int q = lane / LY::kChunks, h = lane % LY::kChunks;
          tma_load_3d(qs + q * LY::kQBytes + h * (kRows * 128), &tmq, 64 * h, it.kvh * G,
                      it.q0 + (it.R0 + q * kRows) / G, q_full);
        }
        if (lane != 0) mbar_arrive(q_full);
      } else {
        const QT* qg = static_cast<const QT*>(p.q);
        for (int r = lane; r < kCtaRows; r += 32) {
          const int R = it.R0 + r;
          const bool rv = R < it.nrows;
          const long long orow =
              rv ? (long long)(it.q0 + R / G) * p.num_q_heads + it.kvh * G + R % G : 0;
          const uint4* src = reinterpret_cast<const uint4*>(qg + orow * D);
          uint8_t* qt = qs + (r / kRows) * LY::kQBytes;
#pragma unroll
          for (int u = 0; u < D / 8; u++)
            cp_async_16_or_zero(qt + (u / 8) * (kRows * 128) + sw_unit(r % kRows, u % 8), src + u,
                                rv);
        }
        cp_async_wait_all();
        fence_proxy_async();
        mbar_arrive(q_full);
      }
      k++;
      // K/V tiles; block ids 32 at a time (lane l holds entry 32*b + l of batch
      // b), the next batch loaded while this one is used
      const int32_t* table =
          p.block_tables + (long long)it.n * p.max_blocks_per_seq + it.first;
      const int nblk = it.hi_u / kBlock - it.first + 1;
      constexpr int kTilesPerBatch = 32 / kTileBlocks;
      auto batch = [&](int b) { return 32 * b + lane < nblk ? table[32 * b + lane] : -1; };
      int ids = batch(0), ids_next = batch(1);
      for (int t = 0; t < it.ntiles; t++, g++) {
        const int st = g % kNS;
        if (t > 0 && t % kTilesPerBatch == 0) {
          ids = ids_next;
          ids_next = batch(t / kTilesPerBatch + 1);
        }
        const int from = __shfl_sync(0xffffffffu, ids, (kTileBlocks * t + lane) & 31);
        const bool inside = lane < kTileBlocks && kTileBlocks * t + lane < nblk;
        const int mine = inside ? from : -1;
        const bool ok = inside && mine >= 0 && mine < p.num_blocks;
        if (g >= kNS && !warp_wait(&kv_free[st], ((g / kNS) - 1) & 1)) {
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
          const int row0 = (mine * p.num_kv_heads + it.kvh) * kBlock;
#pragma unroll
          for (int h = 0; h < LY::kChunks; h++) {
            tma_load_2d(kbase + h * LY::kKVChunk + lane * kBlock * 128, &tmk, 64 * h, row0,
                        &kv_full[st]);
            tma_load_2d(vbase + h * LY::kKVChunk + lane * kBlock * 128, &tmv, 64 * h, row0,
                        &kv_full[st]);
          }
        }
      }
    }
    // no copy may still be landing in shared memory when the CTA exits; the last
    // kNS tiles issued and the last Q are their barriers' current phases
    if (lane == 0) {
      for (int t = g > kNS ? g - kNS : 0; t < g; t++)
        if (!mbar_wait(&kv_full[t % kNS], (t / kNS) & 1)) break;
      if (k > 0) mbar_wait(q_full, (k - 1) & 1);
    }
    if (timed_out && lane == 0) set_flag(p.err, PA_FLAG_TIMEOUT);
  } else if (warp == 1) {
    // ---------------- MMA issuer (the whole warp; one elected lane issues)
    const uint32_t idS = idesc<BF>(kRows, kKeys, false);
    const uint32_t idO = idesc<BF>(kRows, D, true);
    // O_q (+)= P_{q,g} V_g; `first` starts a new accumulation
    auto pv = [&](int q, int g, bool first) -> bool {
      const TileBars tb = tile_bars(tbar0 + q * LY::kTileBars);
      if (!warp_wait(&tb.p_full[g & 1], (g >> 1) & 1)) return false;
      fence_after();
      const uint32_t sP = smem_u32(smem + LY::kPOff + (2 * q + (g & 1)) * LY::kPBytes);
      const uint32_t sV =
          smem_u32(smem + LY::kStageOff + (g % kNS) * LY::kStageBytes) + LY::kKVBytes;
      const uint32_t dO = tmem + q * LY::kTileCols + LY::kOCol;
#pragma unroll
      for (int s = 0; s < kKeys / 16; s++)
        mma_elect(dO, sw128_desc(sP + 32 * s, 16, 1024),
                  sw128_desc(sV + 2048 * s, LY::kKVChunk, 1024), idO,
                  (!first || s > 0) ? 1u : 0u);
      commit_elect(&tb.p_free[g & 1]);
      return true;
    };
    bool ok = true;
    int g = 0, k = 0;
    int n, kvh, tile;
    for (int j = 0; ok && wl.at(j, n, kvh, tile); j++) {
      const Item it = item_info(p, n, kvh, tile, false);
      if (!it.valid || it.ntiles == 0) continue;
      ok = warp_wait(q_full, k & 1);
      k++;
      for (int t = 0; t < it.ntiles && ok; t++, g++) {
        const int st = g % kNS;
        ok = warp_wait(&kv_full[st], (g / kNS) & 1);
        const uint32_t sK = smem_u32(smem + LY::kStageOff + st * LY::kStageBytes);
        for (int q = 0; q < kQTiles && ok; q++) {
          const TileBars tb = tile_bars(tbar0 + q * LY::kTileBars);
          if (g >= 2) ok = warp_wait(&tb.s_free[g & 1], ((g - 2) >> 1) & 1);
          if (!ok) break;
          fence_after();
          const uint32_t sQ = smem_u32(smem + LY::kQOff + q * LY::kQBytes);
          const uint32_t dS = tmem + q * LY::kTileCols + ((g & 1) ? LY::kSCol1 : LY::kSCol0);
#pragma unroll
          for (int s = 0; s < D / 16; s++)
            mma_elect(dS, sw128_desc(sQ + (s / 4) * (kRows * 128) + (s % 4) * 32, 16, 1024),
                      sw128_desc(sK + (s / 4) * LY::kKVChunk + (s % 4) * 32, 16, 1024), idS,
                      s > 0 ? 1u : 0u);
          commit_elect(&tb.s_full[g & 1]);
        }
        if (ok && t == it.ntiles - 1) commit_elect(q_free);  // Q is no longer read
        if (ok && t >= 1) {
          for (int q = 0; q < kQTiles && ok; q++) ok = pv(q, g - 1, t == 1);
          if (ok) commit_elect(&kv_free[(g - 1) % kNS]);
        }
      }
      if (ok) {
        for (int q = 0; q < kQTiles && ok; q++) ok = pv(q, g - 1, it.ntiles == 1);
        if (ok) commit_elect(&kv_free[(g - 1) % kNS]);
      }
    }
    if (!ok && lane == 0) set_flag(p.err, PA_FLAG_TIMEOUT);
    __syncwarp();
  } else {
    // ---------------- softmax: query tile q, thread <-> row (TMEM lane 32*(warp%4) + lane)
    const int q = (warp - 2) / 4;
    const TileBars tb = tile_bars(tbar0 + q * LY::kTileBars);
    const int stid = threadIdx.x - 64 - q * kSoftmaxThreads;  // 0..127 within the tile
    const int row = 32 * (warp & 3) + lane;
    const uint32_t lane_base = tmem + q * LY::kTileCols + ((uint32_t)(32 * (warp & 3)) << 16);
    const float sc = p.scale_log2;
    QT* out = static_cast<QT*>(p.out);
    int g = 0;
    int n, kvh, tile;
    for (int j = 0; !timed_out && wl.at(j, n, kvh, tile); j++) {
      const Item it = item_info(p, n, kvh, tile, false);
      if (!it.valid) continue;
      const int R = it.R0 + q * kRows + row;
      const bool rvalid = R < it.nrows;
      const int c = rvalid ? R / G : 0;
      const int pos = it.L - it.C + c;
      const int row_hi = rvalid ? pos : -1;
      const int row_lo = p.window > 0 ? max(0, pos - p.window + 1) : 0;
      const long long orow =
          (long long)(it.q0 + c) * p.num_q_heads + it.kvh * G + (rvalid ? R % G : 0);
      QT* dst = out + orow * D;
      if (it.ntiles == 0) {  // no row sees a key: zeros
        if (rvalid)
#pragma unroll
          for (int u = 0; u < D / 8; u++) reinterpret_cast<uint4*>(dst)[u] = make_uint4(0, 0, 0, 0);
        continue;
      }
      // p_free[b] completes when the P V that read P buffer b has finished, and
      // with it every earlier MMA.  Tile g waits on it for the P V of tile g-1
      // (buffer (g-1)&1) before rescaling O, and for the P V of tile g-2 (buffer
      // g&1) before writing P.  Per buffer these are successive phases, and a
      // repeated wait on the same phase is safe: the next one needs this tile's P.
      float m_used = kNoMax, l = 0.0f;
      for (int t = 0; t < it.ntiles; t++, g++) {
        if (!mbar_wait(&tb.s_full[g & 1], (g >> 1) & 1)) {
          timed_out = true;
          break;
        }
        fence_after();
        const int pos0 = (it.first + kTileBlocks * t) * kBlock;
        const int* vf = vflags + (g % kNS) * kTileBlocks;
        const bool blocks_ok = vf[0] && vf[1] && vf[2] && vf[3];
        float x[kKeys];
        {
          float v[32];
          const uint32_t scol = (g & 1) ? LY::kSCol1 : LY::kSCol0;
          tmem_ld32(lane_base + scol, v);
#pragma unroll
          for (int j = 0; j < 32; j++) x[j] = v[j];
          tmem_ld32(lane_base + scol + 32, v);
#pragma unroll
          for (int j = 0; j < 32; j++) x[32 + j] = v[j];
        }
        fence_before();
        mbar_arrive(&tb.s_free[g & 1]);  // the MMA may overwrite this S buffer now
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
          for (int j = 8; j < kKeys; j++) part[j & 7] = fmaxf(part[j & 7], x[j]);
        } else {
#pragma unroll
          for (int j = 0; j < 8; j++) part[j] = -INFINITY;
#pragma unroll
          for (int j = 0; j < kKeys; j++) {
            const int kp = pos0 + j;
            const bool vis = kp >= row_lo && kp <= row_hi && vf[j / kBlock];
            x[j] = vis ? x[j] * sc : -INFINITY;
            part[j & 7] = fmaxf(part[j & 7], x[j]);
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
          if (t > 0) {  // O holds this item's tiles < t: wait for the last P V, scale O
            if (!mbar_wait(&tb.p_free[(g - 1) & 1], ((g - 1) >> 1) & 1)) {
              timed_out = true;
              break;
            }
            fence_after();
#pragma unroll
            for (int c0 = 0; c0 < D; c0 += 32) {
              float v[32];
              tmem_ld32(lane_base + LY::kOCol + c0, v);
#pragma unroll
              for (int j = 0; j < 32; j++) v[j] *= factor;
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
        for (int j = 0; j < kKeys; j++) {
          x[j] = fast_exp2(fmaf(x[j], mul, sub));
          part[j & 7] += x[j];
        }
        l += ((part[0] + part[1]) + (part[2] + part[3])) +
             ((part[4] + part[5]) + (part[6] + part[7]));
        // P buffer g&1 was last read by the P V of tile g-2
        if (g >= 2 && !mbar_wait(&tb.p_free[g & 1], ((g - 2) >> 1) & 1)) {
          timed_out = true;
          break;
        }
        // P row -> shared memory (f16/bf16, K-major swizzled)
        uint8_t* prow = smem + LY::kPOff + (2 * q + (g & 1)) * LY::kPBytes;
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
        // warp waits for tile 0's P before either tile's P V.
        const bool edge = pos0 < it.lo_u || pos0 + kKeys - 1 > it.hi_u || !blocks_ok;
        if (edge && q == 0) {
          uint8_t* vbase = smem + LY::kStageOff + (g % kNS) * LY::kStageBytes + LY::kKVBytes;
          for (int idx = stid; idx < kKeys * LY::kChunks * 8; idx += kSoftmaxThreads) {
            const int key = idx / (LY::kChunks * 8);
            const int rest = idx % (LY::kChunks * 8);
            const int kp = pos0 + key;
            if (kp < it.lo_u || kp > it.hi_u || !vf[key / kBlock])
              *reinterpret_cast<uint4*>(vbase + (rest / 8) * LY::kKVChunk +
                                        sw_unit(key, rest % 8)) = make_uint4(0, 0, 0, 0);
          }
        }
        fence_proxy_async();
        fence_before();
        mbar_arrive(&tb.p_full[g & 1]);
      }
      if (timed_out) break;
      // epilogue: wait for this item's last P V (tile g-1)
      if (!mbar_wait(&tb.p_free[(g - 1) & 1], ((g - 1) >> 1) & 1)) {
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
            uint4 pk;
            pk.x = pack2<BF>(v[8 * u + 0] * inv, v[8 * u + 1] * inv);
            pk.y = pack2<BF>(v[8 * u + 2] * inv, v[8 * u + 3] * inv);
            pk.z = pack2<BF>(v[8 * u + 4] * inv, v[8 * u + 5] * inv);
            pk.w = pack2<BF>(v[8 * u + 6] * inv, v[8 * u + 7] * inv);
            *reinterpret_cast<uint4*>(dst + c0 + 8 * u) = pk;
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

template <int D, typename QT>
cudaError_t launch_prefill_tc(const AttnParams& p, const CUtensorMap& tmk,
                              const CUtensorMap& tmv, int num_seqs, cudaStream_t stream) {
  constexpr int smem = tc::Layout<D>::kBytes;
  auto kern = tc::pa_prefill_tc_kernel<D, QT>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
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
  kern<<<grid, tc::kThreads, smem, stream>>>(pt, tmk, tmv, tmq, num_seqs, q_tma ? 1 : 0);
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
