// pa_decode.cu -- paged decode attention with split-K over the context
// ("PyTorch LLM Serving Engine", "Loading": online softmax while walking the
// block table; "MicroGen", Key Features: GQA via repeat_kv, sliding window).
//
// Grid: x = partition + num_parts * (kv head * row_groups + row group), y = seq.
// A CTA owns one (sequence, kv head, group of up to 8 GQA query heads,
// partition of whole blocks).  Its four consumer warps take the partition's
// blocks round-robin, each keeping its own online-softmax state for the same
// heads; the states are merged in shared memory at the end.  A sequence whose
// visible context fits in one partition writes its output directly.  Longer
// ones are split, and the partitions' states (max, normaliser, unnormalised
// output) are merged as  M = max_p m_p,
//   out = sum_p 2^(m_p - M) o_p / sum_p 2^(m_p - M) l_p   (log2-domain maxima),
// in one of two ways:
//   - cluster merge: the num_parts CTAs of a (sequence, kv head, row group) form
//     one thread-block cluster; each sequence's visible blocks are split evenly
//     into as many partitions as its length warrants (up to num_parts, each of
//     at least min_part_blocks), every CTA leaves its state in its own shared
//     memory, and after a cluster barrier the CTAs merge the output elements
//     between them, reading the others' states over distributed shared memory.
//     One launch, no workspace.
//   - workspace merge: partitions of a fixed part_blocks write their states to
//     a caller-provided workspace and pa_reduce_kernel merges them; used when
//     the batch has too few (sequence, kv head) units for clusters of at most 16
//     CTAs to fill the GPU, or when the caller fixes the partition size.
// Partition boundaries and the merge order depend only on logical positions, so
// the result is bit-identical under any relabelling of physical blocks.
#include <algorithm>
#include <mutex>
#include <type_traits>

#include "pa_attn_common.cuh"
#include "pa_internal.h"

namespace pa_dev {

// Decode MMA orientation: the 16 tokens of a block are the M dimension and up to
// eight GQA query heads of the sequence's one query token are the N dimension:
//   S^T = K Q^T   A = K rows (ldmatrix), B = Q^T held in registers
//   O^T += V^T P^T   A = V^T (ldmatrix.trans), B = P^T (movmatrix of S^T's C tile)
// so a block costs 2*D/16 m16n8k16 MMAs and the O^T accumulator is D/16 tiles.
constexpr int kDecHeads = 8;

// Q^T -> B fragments: thread (g, t) holds head g.  Same d order as the K tile
// fragments: natural for 16-bit caches; for int8 the thread's four codes of
// a k-step are d = 16c+4t..16c+4t+3 (slots 2t,2t+1 -> d+0,1; 2t+8,2t+9 -> d+2,3).
// int8 caches with bf16 q: the head's row is scaled by a power of two into f16
// range (q_prescale_shift); returns that shift (0 otherwise), the same for the
// four lanes that hold a head.
template <int MODE, int D, typename QT>
__device__ __forceinline__ int load_qt(uint32_t (&qb)[D / 16][2], const QT* row, int t) {
  if constexpr (MODE != kI8) {
#pragma unroll
    for (int ks = 0; ks < D / 16; ks++) {
      qb[ks][0] = row ? *reinterpret_cast<const uint32_t*>(row + 16 * ks + 2 * t) : 0u;
      qb[ks][1] = row ? *reinterpret_cast<const uint32_t*>(row + 16 * ks + 8 + 2 * t) : 0u;
    }
    return 0;
  } else {
    uint2 raw[D / 16];
#pragma unroll
    for (int ks = 0; ks < D / 16; ks++)
      raw[ks] = row ? *reinterpret_cast<const uint2*>(row + 16 * ks + 4 * t) : make_uint2(0, 0);
    if constexpr (std::is_same<QT, __half>::value) {
#pragma unroll
      for (int ks = 0; ks < D / 16; ks++) {
        qb[ks][0] = raw[ks].x;
        qb[ks][1] = raw[ks].y;
      }
      return 0;
    } else {
      float amax = 0.0f;
#pragma unroll
      for (int ks = 0; ks < D / 16; ks++) {
        const __nv_bfloat16* e = reinterpret_cast<const __nv_bfloat16*>(&raw[ks]);
#pragma unroll
        for (int j = 0; j < 4; j++) amax = fmaxf(amax, fabsf(__bfloat162float(e[j])));
      }
      amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
      amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
      const int shift = q_prescale_shift(amax);
      const float mul = pow2i(-shift);
#pragma unroll
      for (int ks = 0; ks < D / 16; ks++) {
        const __nv_bfloat16* e = reinterpret_cast<const __nv_bfloat16*>(&raw[ks]);
        qb[ks][0] = pack_f16(__bfloat162float(e[0]) * mul, __bfloat162float(e[1]) * mul);
        qb[ks][1] = pack_f16(__bfloat162float(e[2]) * mul, __bfloat162float(e[3]) * mul);
      }
      return shift;
    }
  }
}

// Output column d of O^T tile mt, C-fragment row r (0: g, 1: g+8) of thread g.
template <int MODE, int D>
__device__ __forceinline__ int ot_col(int mt, int g, int r) {
  if constexpr (MODE == kI8) return 16 * mt + 2 * g + r;
  else return 16 * mt + 8 * r + g;
}

// One 16-token block through one warp: the thread's two heads are 2t, 2t+1.
// Keys at positions outside [lo, hi] are masked; their V rows may hold garbage
// (tail slots, data before the window) and are zeroed before O^T += V^T P^T.
// hsc[c] is head 2t+c's score scale (sm_scale * log2(e), times the query's
// prescale 2^shift for int8 caches with bf16 q).
//
// int8 caches: the MMAs see each code as the exact f16 integer code + 1152, so
// S^T comes out high by 1152 * sum_d q[h][d] (kcorr, per head, subtracted here)
// and O^T high by 1152 * sum_j P'[j][h], where P'[j][h] = 2^(y_j - n_h) is the
// value weight of pa_device.cuh (y_j = s_j + log2 v_scale_j, n the running
// reference) rounded to f16 as the MMA sees it; that sum is kept in lv with the
// same rescaling as O^T and subtracted once at the end.  O^T and lv are
// relative to n, the normaliser l to the softmax maximum m.
template <int MODE, int D>
__device__ __forceinline__ void attend_block_dec(const uint32_t (&qb)[D / 16][2],
                                                 float (&o)[D / 16][4], float (&m)[2],
                                                 float (&l)[2], float (&n)[2], float (&lv)[2],
                                                 const float (&kcorr)[2], const uint8_t* stage,
                                                 const float* scales, int lane, int pos0, int lo,
                                                 int hi, const float (&hsc)[2]) {
  using T = Tile<MODE, D>;
  constexpr bool BF = MODE == kBF16;
  const int g = lane >> 2, t = lane & 3;
  const int mi = lane >> 3, mr = lane & 7;
  const uint32_t kbase = smem_u32(stage);
  const uint32_t vbase = kbase + T::kTileBytes;

  // ---- S^T = K Q^T, two independent accumulation chains
  float sa[4] = {0.0f, 0.0f, 0.0f, 0.0f}, sb[4] = {0.0f, 0.0f, 0.0f, 0.0f};
  const int krow = 8 * (mi & 1) + mr;
  if constexpr (MODE != kI8) {
#pragma unroll
    for (int ks = 0; ks < D / 16; ks++) {
      uint32_t a[4];
      ldsm_x4(a, kbase + T::off(krow, 32 * ks + 16 * (mi >> 1)));
      mma16816<BF>(ks & 1 ? sb : sa, a, qb[ks][0], qb[ks][1]);
    }
  } else {
#pragma unroll
    for (int c = 0; c < D / 16; c += 2) {
      uint32_t r[4], a[4];
      ldsm_x4(r, kbase + T::off(krow, 16 * (c + (mi >> 1))));
      // the cache holds offset-binary bytes (code + 128): no sign fix-up
      biased_i8x4_to_f16_plus1152(r[0], a[0], a[2]);  // tokens g,   step c
      biased_i8x4_to_f16_plus1152(r[1], a[1], a[3]);  // tokens g+8, step c
      mma16816<false>(sa, a, qb[c][0], qb[c][1]);
      biased_i8x4_to_f16_plus1152(r[2], a[0], a[2]);  // step c+1
      biased_i8x4_to_f16_plus1152(r[3], a[1], a[3]);
      mma16816<false>(sb, a, qb[c + 1][0], qb[c + 1][1]);
    }
  }

  // ---- scale, mask, online softmax over tokens (log2 domain); i: token g+8(i>>1), head 2t+(i&1)
  bool kept[2];
#pragma unroll
  for (int r = 0; r < 2; r++) {
    const int pos = pos0 + g + 8 * r;
    kept[r] = pos >= lo && pos <= hi;
  }
  float s[4], mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
  for (int i = 0; i < 4; i++) {
    const int tok = g + 8 * (i >> 1);
    float x;
    if constexpr (MODE == kI8) x = (sa[i] + sb[i] - kcorr[i & 1]) * (hsc[i & 1] * scales[tok]);
    else x = (sa[i] + sb[i]) * hsc[i & 1];
    x = kept[i >> 1] ? x : -INFINITY;
    s[i] = x;
    mx[i & 1] = fmaxf(mx[i & 1], x);
  }
  float ref[2], corr[2];
#pragma unroll
  for (int c = 0; c < 2; c++) {
#pragma unroll
    for (int off = 4; off < 32; off <<= 1)
      mx[c] = fmaxf(mx[c], __shfl_xor_sync(0xffffffffu, mx[c], off));
    const float mn = fmaxf(m[c], mx[c]);
    ref[c] = mn == -INFINITY ? 0.0f : mn;
    corr[c] = fast_exp2(m[c] - ref[c]);
    m[c] = mn;
  }
  float p[4];
#pragma unroll
  for (int i = 0; i < 4; i++) {
    const float e = fast_exp2(s[i] - ref[i & 1]);
    l[i & 1] = (i < 2 ? l[i & 1] * corr[i & 1] : l[i & 1]) + e;
    p[i] = e;
  }
  if constexpr (MODE != kI8) {
    if (!__all_sync(0xffffffffu, corr[0] == 1.0f && corr[1] == 1.0f)) {
#pragma unroll
      for (int mt = 0; mt < D / 16; mt++) {
        o[mt][0] *= corr[0];
        o[mt][1] *= corr[1];
        o[mt][2] *= corr[0];
        o[mt][3] *= corr[1];
      }
    }
  } else {
    // value weights 2^(y - n), y = s + log2 v_scale (-inf for a masked token,
    // whatever its slot holds); n moves up when a weight would pass 2^kLazyV
    float lgv[2], y[4];
#pragma unroll
    for (int r = 0; r < 2; r++)
      lgv[r] = kept[r] ? fast_log2(scales[kBlock + g + 8 * r]) : -INFINITY;
    bool grow = false;
#pragma unroll
    for (int i = 0; i < 4; i++) {
      y[i] = s[i] + lgv[i >> 1];
      grow |= y[i] > n[i & 1] + kLazyV;
    }
    if (__any_sync(0xffffffffu, grow)) {
      float ym[2] = {fmaxf(y[0], y[2]), fmaxf(y[1], y[3])};
#pragma unroll
      for (int c = 0; c < 2; c++) {
#pragma unroll
        for (int off = 4; off < 32; off <<= 1)
          ym[c] = fmaxf(ym[c], __shfl_xor_sync(0xffffffffu, ym[c], off));
        const float nn = fmaxf(n[c], ym[c]);
        const float f = fast_exp2(n[c] - nn);
        n[c] = nn;
        lv[c] *= f;
#pragma unroll
        for (int mt = 0; mt < D / 16; mt++) {
          o[mt][c] *= f;
          o[mt][c + 2] *= f;
        }
      }
    }
#pragma unroll
    for (int i = 0; i < 4; i++) p[i] = fast_exp2(y[i] - n[i & 1]);
  }
  // P^T as the PV B operand: C tile (token g, heads 2t, 2t+1) transposed to
  // (head g, tokens 2t, 2t+1), once for tokens 0..7 and once for 8..15.
  const uint32_t pk0 = pack2<BF>(p[0], p[1]), pk1 = pack2<BF>(p[2], p[3]);
  if constexpr (MODE == kI8) {
    const float2 f0 = __half22float2(*reinterpret_cast<const __half2*>(&pk0));
    const float2 f1 = __half22float2(*reinterpret_cast<const __half2*>(&pk1));
    lv[0] += f0.x + f1.x;
    lv[1] += f0.y + f1.y;
  }
  const uint32_t pb0 = movmatrix_t(pk0);
  const uint32_t pb1 = movmatrix_t(pk1);

  // ---- O^T += V^T P^T
  if constexpr (MODE != kI8) {
    uint32_t mk01 = 0xffffffffu, mk89 = 0xffffffffu;
    if (pos0 < lo || pos0 + kBlock - 1 > hi) {
      auto keep = [&](int tok) {
        const int pos = pos0 + tok;
        return pos >= lo && pos <= hi;
      };
      mk01 = (keep(2 * t) ? 0x0000ffffu : 0u) | (keep(2 * t + 1) ? 0xffff0000u : 0u);
      mk89 = (keep(2 * t + 8) ? 0x0000ffffu : 0u) | (keep(2 * t + 9) ? 0xffff0000u : 0u);
    }
    const int vrow = 8 * (mi >> 1) + mr;
#pragma unroll
    for (int mt = 0; mt < D / 16; mt++) {
      uint32_t a[4];
      ldsm_x4_t(a, vbase + T::off(vrow, 32 * mt + 16 * (mi & 1)));
      a[0] &= mk01;
      a[1] &= mk01;
      a[2] &= mk89;
      a[3] &= mk89;
      mma16816<BF>(o[mt], a, pb0, pb1);
    }
  } else {
    // ldmatrix.trans on 16-bit pairs of codes: matrix (tokens 8j..8j+7, bytes
    // 16mt..16mt+15) gives thread (g, t) tokens 8j+2t, 8j+2t+1 at d = 16mt+2g and
    // +1; one byte permute per f16 pair (code + 1152) makes the A fragment of
    // tile mt, whose rows g and g+8 are d = 16mt+2g and 16mt+2g+1
    const int vrow = 8 * (mi & 1) + mr;
#pragma unroll
    for (int mp = 0; mp < D / 32; mp++) {
      uint32_t r[4];
      ldsm_x4_t(r, vbase + T::off(vrow, 32 * mp + 16 * (mi >> 1)));
#pragma unroll
      for (int h = 0; h < 2; h++) {
        const uint32_t x0 = r[2 * h], x1 = r[2 * h + 1];  // offset-binary code bytes
        uint32_t a[4];
        a[0] = __byte_perm(x0, 0x64646464u, 0x4240);  // row g:   tokens 2t, 2t+1
        a[1] = __byte_perm(x0, 0x64646464u, 0x4341);  // row g+8: tokens 2t, 2t+1
        a[2] = __byte_perm(x1, 0x64646464u, 0x4240);  // row g:   tokens 2t+8, 2t+9
        a[3] = __byte_perm(x1, 0x64646464u, 0x4341);  // row g+8: tokens 2t+8, 2t+9
        mma16816<false>(o[2 * mp + h], a, pb0, pb1);
      }
    }
  }
}

// The step's new K and V rows of (sequence b, kv head kvh) written into slot
// `off` of physical block `phys` by one warp (E = D/32 elements per lane; an
// int8 cache quantises them as the KV write does), then ordered before the TMA
// copy of that block (generic-proxy writes, then an async-proxy read).
template <int MODE, int D, typename QT>
__device__ __forceinline__ void write_new_row(const AttnParams& p, int b, int kvh, int phys,
                                              int off, int lane) {
  constexpr int E = D / 32;
  using R = typename std::conditional<E == 4, uint2, uint32_t>::type;  // E 16-bit values
  const long long src = ((long long)b * p.num_kv_heads + kvh) * D + lane * E;
  const long long dst_row = ((long long)phys * p.num_kv_heads + kvh) * kBlock + off;
#pragma unroll
  for (int which = 0; which < 2; which++) {
    const R raw = *reinterpret_cast<const R*>(static_cast<const QT*>(which ? p.v_new : p.k_new) +
                                              src);
    uint8_t* cache = const_cast<uint8_t*>(which ? p.v_cache : p.k_cache);
    if constexpr (MODE == kI8) {
      float x[E];
      const QT* e = reinterpret_cast<const QT*>(&raw);
#pragma unroll
      for (int i = 0; i < E; i++) x[i] = in_to_f32<QT>(e[i]);
      uint8_t q[E];
      float scale;
      quantize_row<E>(x, q, scale);
      uint8_t* dst = cache + dst_row * D + lane * E;
      if constexpr (E == 4) *reinterpret_cast<uint32_t*>(dst) = *reinterpret_cast<uint32_t*>(q);
      else *reinterpret_cast<uint16_t*>(dst) = *reinterpret_cast<uint16_t*>(q);
      if (lane == 0) const_cast<float*>(which ? p.v_scale : p.k_scale)[dst_row] = scale;
    } else {
      *reinterpret_cast<R*>(cache + (dst_row * D + lane * E) * 2) = raw;
    }
  }
  asm volatile("fence.proxy.async.global;" ::: "memory");
  __syncwarp();
}

// Partitions of a sequence with visible context L, their size in blocks (psz)
// and the visible range (keys from lo, blocks first..last).  L >= 1.
__device__ __forceinline__ int decode_parts(const AttnParams& p, int L, int& lo, int& first,
                                            int& last, int& psz) {
  lo = p.window > 0 ? max(0, L - p.window) : 0;
  first = lo / kBlock;
  last = (L - 1) / kBlock;
  const int nb = last - first + 1;
  if (p.merge_mode == kMergeCluster) {
    const int np = max(1, min(p.num_parts, (nb + p.min_part_blocks - 1) / p.min_part_blocks));
    psz = (nb + np - 1) / np;
  } else {
    psz = p.part_blocks;
  }
  return (nb + psz - 1) / psz;
}

// Decode CTAs have no producer warp: warp w of the four owns blocks w, w+4,
// w+8, ... of its partition and the two stages w and w+4, which hold its next
// two blocks.  It issues the TMA copies for a block itself, and refills a stage
// as soon as it has finished with it, so a stage is only ever waited on, read
// and refilled by one warp and no "stage empty" barrier is needed.
constexpr int kDecWarps = 4;
constexpr int kDecThreads = kDecWarps * 32;
// Cluster merge: at most 16 CTAs per cluster (the non-portable maximum, checked
// on the device).
constexpr int kMaxCluster = 16;
static_assert(kMaxCluster * kDecHeads <= kDecThreads, "one thread per (partition, row)");
static_assert(kStages == 2 * kDecWarps, "two stages per decode warp");

template <int MODE, int D>
struct DecSmem {
  static constexpr int kOS = D + 4;  // fp32 row stride of the warp-merge area
  static constexpr int kMergeBytes = kDecWarps * kDecHeads * (kOS + 2) * 4;
  // after the warp merge, this CTA's partition state for the cluster merge:
  // m[8], l[8], ok, then o[8][D] (fp32)
  static constexpr int kPartOff = (kMergeBytes + 127) / 128 * 128;
  static constexpr int kPartOOff = kPartOff + (2 * kDecHeads + 4) * 4;
  static constexpr int kPartBytes = kPartOOff - kPartOff + kDecHeads * D * 4;
  // then, private to this CTA, the partitions' states gathered for the merge:
  // m (then weights) [16][8], l [16][8], the rows' maxima [8] and 1 / normaliser [8]
  static constexpr int kGatherOff = kPartOff + kPartBytes;
  static constexpr int kGatherBytes = (2 * kMaxCluster * kDecHeads + 2 * kDecHeads) * 4;
  static_assert(kGatherOff + kGatherBytes <= Smem<MODE, D>::kDataBytes,
                "merge areas must fit the stages");
};

// Cluster-wide barrier: every thread of every CTA in the cluster arrives, and
// this CTA's earlier shared-memory writes are visible to the others after it.
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile(
      "barrier.cluster.arrive.release.aligned;\n\t"
      "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// fp32 at the same shared-memory offset as `local` in cluster CTA `rank`.
__device__ __forceinline__ float ld_cluster_f32(const void* local, uint32_t rank) {
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_u32(local)),
               "r"(rank));
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(remote) : "memory");
  return v;
}

// Warp-level copy of one block of kv head kvh into stage `slot`: lane 0 arms
// the stage's barrier and issues the TMA boxes; for int8, lanes 0-7 fetch the
// two 64-byte scale runs with cp.async.  A block id outside the pool is not
// copied: the stage is marked invalid and its barrier completes at once.
template <int MODE, int D>
__device__ __forceinline__ void fetch_block(const AttnParams& p, const void* tmk, const void* tmv,
                                            const SmemPtrs& s, int slot, int phys, int kvh,
                                            int lane) {
  using T = Tile<MODE, D>;
  const bool ok = phys >= 0 && phys < p.num_blocks;
  const long long row0 = ((long long)(ok ? phys : 0) * p.num_kv_heads + kvh) * kBlock;
  if (lane == 0) {
    s.valid[slot] = ok ? 1 : 0;
    if (ok) {
      mbar_arrive_expect_tx(&s.full[slot], T::kTxBytes);
      uint8_t* st = s.stages + slot * T::kStageBytes;
#pragma unroll
      for (int h = 0; h < T::kChunks; h++) {
        tma_load_2d(st + h * T::kBoxBytes, tmk, h * T::kChunkElems, (int)row0, &s.full[slot]);
        tma_load_2d(st + T::kTileBytes + h * T::kBoxBytes, tmv, h * T::kChunkElems, (int)row0,
                    &s.full[slot]);
      }
    } else {
      set_flag(p.err, PA_FLAG_BLOCK_ID);
      mbar_arrive(&s.full[slot]);
    }
  }
  if constexpr (MODE == kI8) {
    if (lane < T::kScaleLanes) {
      if (ok) {
        const float* src = (lane < 4 ? p.k_scale : p.v_scale) + row0 + 4 * (lane & 3);
        cp_async_16(s.scales + slot * 2 * kBlock + (lane < 4 ? 0 : kBlock) + 4 * (lane & 3), src);
        cp_async_arrive_noinc(&s.full[slot]);
      } else {
        mbar_arrive(&s.full[slot]);
      }
    }
  }
}

// WRITE: the launch also writes the step's new rows (p.k_new, p.v_new) at each
// sequence's position L-1 (an instance of its own, so that the plain decode's
// register allocation does not carry the write).
template <int MODE, int D, typename QT, bool WRITE>
__global__ void __launch_bounds__(kDecThreads, MODE == kI8 ? 5 : 3)
    pa_decode_kernel(const __grid_constant__ AttnParams p, const __grid_constant__ CUtensorMap tmk,
                     const __grid_constant__ CUtensorMap tmv) {
  extern __shared__ __align__(128) uint8_t smem[];
  pdl_wait();               // the kernel before (say, the K/V write) is complete
  pdl_launch_dependents();  // the split-K merge may start its launch
  const int b = blockIdx.y;
  const int part = blockIdx.x % p.num_parts;
  const int hx = blockIdx.x / p.num_parts;
  const int kvh = hx / p.row_groups, rg = hx % p.row_groups;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rows = min(kDecHeads, p.group - rg * kDecHeads);  // query heads of this CTA
  const int h0 = kvh * p.group + rg * kDecHeads;              // the first of them
  QT* out = static_cast<QT*>(p.out);

  const int L = clamp_context(p, b, threadIdx.x == 0 && blockIdx.x == 0);
  if (L == 0) {  // nothing visible: zeros
    if (part == 0)
      for (int idx = threadIdx.x; idx < rows * D; idx += kDecThreads)
        out[((long long)b * p.num_q_heads + h0 + idx / D) * D + idx % D] = to_out<QT>(0.0f);
    return;
  }
  int lo, first, last, psz;
  const int nparts = decode_parts(p, L, lo, first, last, psz);
  // a split sequence of the cluster merge: every CTA of the cluster takes part in
  // the merge, including those its length leaves without a partition; otherwise
  // (the decision is the same for the whole cluster) such CTAs have nothing to do
  const bool cluster_merge = p.merge_mode == kMergeCluster && nparts > 1;
  if (part >= nparts && !cluster_merge) return;
  const int blk0 = first + part * psz;
  const int nblk = part < nparts ? min(psz, last + 1 - blk0) : 0;
  const int nmine = nblk > warp ? (nblk - warp + kDecWarps - 1) / kDecWarps : 0;  // this warp's blocks

  const SmemPtrs s = smem_ptrs<MODE, D>(smem);
  init_barriers(s, Tile<MODE, D>::kFullArrivals, 1);
  // block ids of this warp's blocks k = 0..nmine-1 (logical block blk0 + warp + 4k)
  const int32_t* table = p.block_tables + (long long)b * p.max_blocks_per_seq + blk0 + warp;
  int ids = lane < nmine ? table[kDecWarps * lane] : -1;
  // with the step's new rows given, the warp that copies the block holding
  // position L-1 writes them into it first (before its first copy, so that the
  // write's registers are free again in the loop)
  if constexpr (WRITE) {
    const int j = last - blk0;  // the newest block's index in this partition
    if (j >= 0 && j < nblk && j % kDecWarps == warp) {
      const int phys = p.block_tables[(long long)b * p.max_blocks_per_seq + last];
      if (phys >= 0 && phys < p.num_blocks)
        write_new_row<MODE, D, QT>(p, b, kvh, phys, (L - 1) % kBlock, lane);
    }
  }
  auto fetch = [&](int k, int slot, int phys) {
    fetch_block<MODE, D>(p, &tmk, &tmv, s, slot, phys, kvh, lane);
  };
#pragma unroll
  for (int k = 0; k < 2; k++)
    if (k < nmine) fetch(k, warp + kDecWarps * k, __shfl_sync(0xffffffffu, ids, k));

  const int g = lane >> 2, t = lane & 3;
  const QT* q = static_cast<const QT*>(p.q);
  uint32_t qb[D / 16][2];
  const int qshift = load_qt<MODE, D, QT>(
      qb, g < rows ? q + ((long long)b * p.num_q_heads + h0 + g) * D : nullptr, t);
  // score scale of this thread's score columns (heads 2t, 2t+1; lane 8t+4c holds head 2t+c)
  float hsc[2] = {p.scale_log2, p.scale_log2};
  if constexpr (MODE == kI8 && !std::is_same<QT, __half>::value) {
#pragma unroll
    for (int c = 0; c < 2; c++)
      hsc[c] = p.scale_log2 * pow2i(__shfl_sync(0xffffffffu, qshift, 8 * t + 4 * c));
  }
  float o[D / 16][4];
#pragma unroll
  for (int mt = 0; mt < D / 16; mt++)
#pragma unroll
    for (int i = 0; i < 4; i++) o[mt][i] = 0.0f;
  float m[2] = {-INFINITY, -INFINITY}, l[2] = {0.0f, 0.0f}, lv[2] = {0.0f, 0.0f};
  float n[2] = {kNoRef, kNoRef};  // int8: the value weights' reference
  float kcorr[2] = {0.0f, 0.0f};
  if constexpr (MODE == kI8) {
    // 1152 * sum_d q[h][d] (the f16 q the MMA sees) for this thread's score columns h = 2t, 2t+1
    float qs = 0.0f;
#pragma unroll
    for (int ks = 0; ks < D / 16; ks++)
#pragma unroll
      for (int j = 0; j < 2; j++) {
        const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&qb[ks][j]));
        qs += f.x + f.y;
      }
    qs += __shfl_xor_sync(0xffffffffu, qs, 1);
    qs += __shfl_xor_sync(0xffffffffu, qs, 2);  // all of head g's row
    kcorr[0] = 1152.0f * __shfl_sync(0xffffffffu, qs, 8 * t);
    kcorr[1] = 1152.0f * __shfl_sync(0xffffffffu, qs, 8 * t + 4);
  }

  int kfail = -1;  // the block whose wait ran out
  for (int k = 0; k < nmine; k++) {
    const int slot = warp + kDecWarps * (k & 1);
    if (!mbar_wait(&s.full[slot], (k >> 1) & 1)) {
      if (lane == 0) set_flag(p.err, PA_FLAG_TIMEOUT);
      kfail = k;
      break;
    }
    if (s.valid[slot])
      attend_block_dec<MODE, D>(qb, o, m, l, n, lv, kcorr,
                                s.stages + slot * Tile<MODE, D>::kStageBytes,
                                s.scales + slot * 2 * kBlock, lane,
                                (blk0 + warp + kDecWarps * k) * kBlock, lo, L - 1, hsc);
    __syncwarp();
    if (k + 2 < nmine) {
      if (((k + 2) & 31) == 0)  // next 32 of this warp's block ids
        ids = (k + 2 + lane) < nmine ? table[kDecWarps * (k + 2 + lane)] : -1;
      fetch(k + 2, slot, __shfl_sync(0xffffffffu, ids, (k + 2) & 31));
    }
  }
  if (kfail >= 0) {  // no copy may still be landing in shared memory when the CTA exits
    // only blocks kfail and kfail+1 can be in flight, and they are their stages'
    // current phases (a parity wait cannot tell an older phase from the current one)
    for (int k = kfail; k < nmine && k < kfail + 2; k++)
      if (!mbar_wait(&s.full[warp + kDecWarps * (k & 1)], (k >> 1) & 1)) break;
    if (lane == 0) *s.abort_flag = 1;
  }
  // the normalisers were summed per thread over its two tokens: add up the tokens
#pragma unroll
  for (int c = 0; c < 2; c++)
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      l[c] += __shfl_xor_sync(0xffffffffu, l[c], off);
      if constexpr (MODE == kI8) lv[c] += __shfl_xor_sync(0xffffffffu, lv[c], off);
    }
  if constexpr (MODE == kI8) {
    // remove the 1152 carried by every V code, then move O^T from the value
    // weights' reference n to the softmax's m (fp32; no key seen: m = -inf, O^T = 0)
    float f[2];
#pragma unroll
    for (int c = 0; c < 2; c++) f[c] = m[c] == -INFINITY ? 0.0f : exp2f(n[c] - m[c]);
#pragma unroll
    for (int mt = 0; mt < D / 16; mt++)
#pragma unroll
      for (int i = 0; i < 4; i++) o[mt][i] = (o[mt][i] - 1152.0f * lv[i & 1]) * f[i & 1];
  }
  __syncthreads();  // every stage consumed: reuse them for the merge
  const bool aborted = *s.abort_flag != 0;
  if (aborted && !cluster_merge) return;

  constexpr int OS = DecSmem<MODE, D>::kOS;
  float* mw = reinterpret_cast<float*>(s.stages);  // [warp][head]
  float* lw = mw + kDecWarps * kDecHeads;          // [warp][head]
  float* ow = lw + kDecWarps * kDecHeads;          // [warp][head][OS]
  if (g == 0) {
    mw[warp * kDecHeads + 2 * t] = m[0];
    mw[warp * kDecHeads + 2 * t + 1] = m[1];
    lw[warp * kDecHeads + 2 * t] = l[0];
    lw[warp * kDecHeads + 2 * t + 1] = l[1];
  }
#pragma unroll
  for (int mt = 0; mt < D / 16; mt++)
#pragma unroll
    for (int i = 0; i < 4; i++) {
      const int h = 2 * t + (i & 1);
      if (h < rows) ow[(warp * kDecHeads + h) * OS + ot_col<MODE, D>(mt, g, i >> 1)] = o[mt][i];
    }
  __syncthreads();

  if (cluster_merge) {
    // this CTA's partition state, then the cluster merge of every output element
    using DS = DecSmem<MODE, D>;
    float* pm = reinterpret_cast<float*>(s.stages + DS::kPartOff);  // [head]
    float* pl = pm + kDecHeads;                                      // [head]
    int* pok = reinterpret_cast<int*>(pl + kDecHeads);
    float* po = reinterpret_cast<float*>(s.stages + DS::kPartOOff);  // [head][D]
    for (int idx = threadIdx.x; idx < rows * D; idx += kDecThreads) {
      const int r = idx / D, d = idx % D;
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < kDecWarps; w++) M = fmaxf(M, mw[w * kDecHeads + r]);
      float num = 0.0f, den = 0.0f;
      if (M != -INFINITY) {
#pragma unroll
        for (int w = 0; w < kDecWarps; w++) {
          const float e = exp2f(mw[w * kDecHeads + r] - M);
          num += e * ow[(w * kDecHeads + r) * OS + d];
          den += e * lw[w * kDecHeads + r];
        }
      }
      po[r * D + d] = num;
      if (d == 0) {
        pm[r] = M;
        pl[r] = den;
      }
    }
    // the cluster rank is the partition (grid x = partition + num_parts * ...)
    if (threadIdx.x == 0) *pok = (!aborted && cluster_ctarank() == (uint32_t)part) ? 1 : 0;
    cluster_sync_all();  // every partition's state is in place
    // No remote read below waits for another: each partition's (m, l) of every
    // row and its flag, one thread per (partition, row), into this CTA's shared
    // memory; the rows' maxima, normalisers and the partitions' weights there;
    // then each output element's partition outputs, all issued at once.
    float* gm = reinterpret_cast<float*>(s.stages + DS::kGatherOff);  // [q][8]: m, then weight
    float* gl = gm + kMaxCluster * kDecHeads;                          // [q][8]: l
    float* rmax = gl + kMaxCluster * kDecHeads;                        // [8]
    float* rinv = rmax + kDecHeads;                                    // [8]: 1 / normaliser
    bool ok_q = true;
    if (threadIdx.x < nparts * kDecHeads) {
      const int q = threadIdx.x / kDecHeads, r = threadIdx.x % kDecHeads;
      gm[threadIdx.x] = r < rows ? ld_cluster_f32(pm + r, q) : -INFINITY;
      gl[threadIdx.x] = r < rows ? ld_cluster_f32(pl + r, q) : 0.0f;
      if (r == 0) ok_q = __float_as_int(ld_cluster_f32(pok, q)) == 1;
    }
    const bool all_ok = __syncthreads_and(ok_q) != 0;
    if (threadIdx.x < rows) {
      const int r = threadIdx.x;
      float M = -INFINITY;
      for (int q = 0; q < nparts; q++) M = fmaxf(M, gm[q * kDecHeads + r]);
      float den = 0.0f;
      if (M != -INFINITY)
        for (int q = 0; q < nparts; q++)
          den += exp2f(gm[q * kDecHeads + r] - M) * gl[q * kDecHeads + r];
      rmax[r] = M;
      rinv[r] = den > 0.0f ? 1.0f / den : 0.0f;
    }
    __syncthreads();
    if (threadIdx.x < nparts * kDecHeads) {  // weight 2^(m_q - M); 0 without a key
      const float M = rmax[threadIdx.x % kDecHeads];
      gm[threadIdx.x] = M != -INFINITY ? exp2f(gm[threadIdx.x] - M) : 0.0f;
    }
    __syncthreads();
    if (all_ok) {
      for (int idx = part * kDecThreads + threadIdx.x; idx < rows * D;
           idx += p.num_parts * kDecThreads) {
        const int r = idx / D, d = idx % D;
        float v[kMaxCluster];
#pragma unroll
        for (int q = 0; q < kMaxCluster; q++)
          v[q] = q < nparts ? ld_cluster_f32(po + r * D + d, q) : 0.0f;
        float num = 0.0f;
#pragma unroll
        for (int q = 0; q < kMaxCluster; q++)
          if (q < nparts) num += gm[q * kDecHeads + r] * v[q];
        out[((long long)b * p.num_q_heads + h0 + r) * D + d] = to_out<QT>(num * rinv[r]);
      }
    }
    cluster_sync_all();  // no CTA leaves while another still reads its state
    return;
  }

  const bool direct = nparts == 1;
  for (int idx = threadIdx.x; idx < rows * D; idx += kDecThreads) {
    const int r = idx / D, d = idx % D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kDecWarps; w++) M = fmaxf(M, mw[w * kDecHeads + r]);
    float num = 0.0f, den = 0.0f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < kDecWarps; w++) {
        const float e = exp2f(mw[w * kDecHeads + r] - M);
        num += e * ow[(w * kDecHeads + r) * OS + d];
        den += e * lw[w * kDecHeads + r];
      }
    }
    const long long hrow = (long long)b * p.num_q_heads + h0 + r;
    if (direct) {
      out[hrow * D + d] = to_out<QT>(den > 0.0f ? num / den : 0.0f);
    } else {
      const long long pi = hrow * p.num_parts + part;
      p.ws_o[pi * D + d] = num;
      if (d == 0) {
        p.ws_m[pi] = M;
        p.ws_l[pi] = den;
      }
    }
  }
}

// One 128-thread CTA per (sequence, query head) merges that head's partition
// states: the maximum and the normaliser over all partitions are reduced by the
// whole CTA, then each warp accumulates the weighted partial outputs of every
// fourth partition (lanes across head_dim, several rows in flight) and the four
// sums are added in shared memory.
constexpr int kRedThreads = 128;

template <int D, typename QT>
__global__ void __launch_bounds__(kRedThreads) pa_reduce_kernel(const AttnParams p) {
  pdl_wait();  // the partitions' states are written
  pdl_launch_dependents();
  __shared__ float red[kRedThreads / 32];
  __shared__ float4 part_sum[kRedThreads / 32][D / 4];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const long long hrow = blockIdx.x;  // b * num_q_heads + h
  const int b = (int)(hrow / p.num_q_heads);
  const int L = clamp_context(p, b, false);
  if (L == 0) return;
  int lo, first, last, psz;
  const int nparts = decode_parts(p, L, lo, first, last, psz);
  if (nparts <= 1) return;  // written directly by the attention kernel
  const long long base = hrow * p.num_parts;

  float M = -INFINITY;
  for (int q = threadIdx.x; q < nparts; q += kRedThreads) M = fmaxf(M, p.ws_m[base + q]);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
  if (lane == 0) red[warp] = M;
  __syncthreads();
  M = fmaxf(fmaxf(red[0], red[1]), fmaxf(red[2], red[3]));
  __syncthreads();
  QT* out = static_cast<QT*>(p.out) + hrow * D;
  if (M == -INFINITY) {  // no partition saw a key
    for (int d = threadIdx.x; d < D; d += kRedThreads) out[d] = to_out<QT>(0.0f);
    return;
  }
  float den = 0.0f;
  for (int q = threadIdx.x; q < nparts; q += kRedThreads)
    den += exp2f(p.ws_m[base + q] - M) * p.ws_l[base + q];
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) den += __shfl_xor_sync(0xffffffffu, den, off);
  if (lane == 0) red[warp] = den;

  // lanes across head_dim: D/32 floats each (a float4 for D = 128, a float2 for 64)
  constexpr int E = D / 32;
  float acc[E];
#pragma unroll
  for (int e = 0; e < E; e++) acc[e] = 0.0f;
#pragma unroll 4
  for (int q = warp; q < nparts; q += kRedThreads / 32) {
    const float w = exp2f(p.ws_m[base + q] - M);  // 0 for a partition with no visible key
    const float* src = p.ws_o + (base + q) * D + lane * E;
    if constexpr (E == 4) {
      const float4 v = *reinterpret_cast<const float4*>(src);
      acc[0] += w * v.x;
      acc[1] += w * v.y;
      acc[2] += w * v.z;
      acc[3] += w * v.w;
    } else {
      const float2 v = *reinterpret_cast<const float2*>(src);
      acc[0] += w * v.x;
      acc[1] += w * v.y;
    }
  }
  float* mine = reinterpret_cast<float*>(&part_sum[warp][0]) + lane * E;
#pragma unroll
  for (int e = 0; e < E; e++) mine[e] = acc[e];
  __syncthreads();
  const float total = red[0] + red[1] + red[2] + red[3];
  for (int d = threadIdx.x; d < D; d += kRedThreads) {
    float v = 0.0f;
#pragma unroll
    for (int w = 0; w < kRedThreads / 32; w++) v += reinterpret_cast<const float*>(&part_sum[w][0])[d];
    out[d] = to_out<QT>(total > 0.0f ? v / total : 0.0f);
  }
}

}  // namespace pa_dev

using namespace pa_dev;

namespace {

int current_sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return n;
}

// Most blocks one sequence's visible context can touch.
int max_blocks_touched(int max_blocks_per_seq, int window) {
  if (window <= 0) return max_blocks_per_seq;
  return std::min(max_blocks_per_seq, (window + 2 * kBlock - 2) / kBlock);
}


// Whether a cluster of `size` decode CTAs with the largest shared-memory
// footprint (16-bit cache, head_dim 128) can be resident on the current device;
// asked of the occupancy calculator once per device and size.
bool cluster_fits(int size) {
  if (size <= 1) return true;
  if (size > kMaxCluster) return false;
  static std::mutex mu;
  static signed char known[64][kMaxCluster + 1];  // 0 unknown, 1 fits, 2 does not
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
  std::lock_guard<std::mutex> lock(mu);
  if (known[dev][size] == 0) {
    auto kern = pa_decode_kernel<kF16, 128, __half, false>;
    constexpr int smem = Smem<kF16, 128>::kBytes;
    bool ok = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) ==
                  cudaSuccess &&
              (size <= 8 || cudaFuncSetAttribute(kern,
                                                 cudaFuncAttributeNonPortableClusterSizeAllowed,
                                                 1) == cudaSuccess);
    int n = 0;
    if (ok) {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3((unsigned)size, 1, 1);
      cfg.blockDim = dim3(kDecThreads, 1, 1);
      cfg.dynamicSmemBytes = smem;
      cudaLaunchAttribute at[1];
      at[0].id = cudaLaunchAttributeClusterDimension;
      at[0].val.clusterDim.x = (unsigned)size;
      at[0].val.clusterDim.y = 1;
      at[0].val.clusterDim.z = 1;
      cfg.attrs = at;
      cfg.numAttrs = 1;
      ok = cudaOccupancyMaxActiveClusters(&n, kern, &cfg) == cudaSuccess && n >= 1;
    }
    cudaGetLastError();  // a refusal here only means "no"
    known[dev][size] = ok ? 1 : 2;
  }
  return known[dev][size] == 1;
}

struct Split {
  int mode;             // kMergeWorkspace or kMergeCluster
  int part_blocks;      // workspace: blocks per partition
  int num_parts;        // partitions per (sequence, kv head, row group) at most
  int min_part_blocks;  // cluster: smallest partition
};

// The workspace split: partitions of 64 blocks (1024 tokens) unless the batch is
// too small to give every SM two CTAs, in which case halve them (down to 4).
Split workspace_split(long long units, int maxb, int partition_blocks, int sms) {
  int pb = partition_blocks;
  if (pb <= 0) {
    const long long target = 2LL * sms;
    pb = 64;
    while (pb > 4 && units * ((maxb + pb - 1) / pb) < target) pb /= 2;
  }
  Split s;
  s.mode = kMergeWorkspace;
  s.part_blocks = std::max(1, std::min(pb, maxb));
  s.num_parts = (maxb + s.part_blocks - 1) / s.part_blocks;
  s.min_part_blocks = 1;
  return s;
}

// partition_blocks > 0: fixed partitions, workspace merge.  partition_blocks < 0:
// each sequence split evenly into up to -partition_blocks partitions (at most 16),
// cluster merge (a cluster the device cannot hold falls back to the workspace
// merge).  0, the automatic choice: the workspace merge with 64-block partitions
// while the batch gives every SM two CTAs that way; a smaller batch whose
// sequences span at most 256 blocks and whose (sequence, kv head, row group)
// units fill the SMs at 16 CTAs each takes 16-CTA clusters (each CTA at most
// 16 blocks, no merge launch); a smaller one still halves the workspace
// partitions (down to 4 blocks).  Measured on GB300 (decode call, graph
// replays, L2 flushed): the Qwen2.5-1.5B batch 15.2 us with 16-CTA clusters
// against 17.0 us with the merge kernel; the 7B MHA, INT8 and mixed batches
// keep the workspace merge (clusters of 2-16 measured 1 % faster to 2x slower).
Split choose_split(int num_seqs, int num_kv_heads, int row_groups, int max_blocks_per_seq,
                   int window, int partition_blocks) {
  const int maxb = max_blocks_touched(max_blocks_per_seq, window);
  const long long units = (long long)num_seqs * num_kv_heads * row_groups;
  const int sms = std::max(current_sm_count(), 1);
  if (partition_blocks > 0) return workspace_split(units, maxb, partition_blocks, sms);
  if (partition_blocks == 0) {
    const bool small = units * ((maxb + 63) / 64) < 2LL * sms;
    if (small && maxb > kMaxCluster && maxb <= kMaxCluster * kMaxCluster &&
        units * kMaxCluster >= sms && cluster_fits(kMaxCluster)) {
      Split s;
      s.mode = kMergeCluster;
      s.part_blocks = 0;
      s.num_parts = kMaxCluster;
      s.min_part_blocks = 1;
      return s;
    }
    return workspace_split(units, maxb, 0, sms);
  }
  int P = std::min(std::min(-partition_blocks, kMaxCluster), maxb);
  const int min_part = 1;
  P = std::max(P, 1);
  if (!cluster_fits(P))
    return workspace_split(units, maxb, partition_blocks < 0 ? (maxb + P - 1) / P : 0, sms);
  Split s;
  s.mode = kMergeCluster;
  s.part_blocks = 0;
  s.num_parts = P;
  s.min_part_blocks = min_part;
  return s;
}

size_t workspace_for(int num_seqs, int num_q_heads, int head_dim, const Split& s) {
  if (s.mode != kMergeWorkspace || s.num_parts <= 1) return 0;
  const size_t n = (size_t)num_seqs * num_q_heads * s.num_parts;
  return n * head_dim * 4 + 2 * n * 4 + 16;
}

template <int MODE, int D, typename QT>
cudaError_t launch_decode(const AttnParams& p, const CUtensorMap& tmk, const CUtensorMap& tmv,
                          int num_seqs, cudaStream_t stream) {
  constexpr int smem = Smem<MODE, D>::kBytes;
  auto kern = p.k_new ? pa_decode_kernel<MODE, D, QT, true> : pa_decode_kernel<MODE, D, QT, false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const dim3 grid((unsigned)(p.num_parts * p.num_kv_heads * p.row_groups), (unsigned)num_seqs);
  // the partitions of a (sequence, kv head, row group) are one cluster when
  // they merge in the launch
  const bool cluster = p.merge_mode == kMergeCluster && p.num_parts > 1;
  if (cluster && p.num_parts > 8) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
  }
  e = pa_internal::launch_dependent(kern, grid, dim3(kDecThreads), smem, stream,
                                    cluster ? (unsigned)p.num_parts : 1u, p, tmk, tmv);
  if (e != cudaSuccess || cluster || p.num_parts <= 1) return e;
  const long long heads = (long long)num_seqs * p.num_q_heads;
  return pa_internal::launch_dependent(pa_reduce_kernel<D, QT>, dim3((unsigned)heads),
                                       dim3(kRedThreads), 0, stream, 1u, p);
}

template <int MODE, typename QT>
cudaError_t launch_decode_d(const AttnParams& p, const CUtensorMap& tmk, const CUtensorMap& tmv,
                           int head_dim, int num_seqs, cudaStream_t s) {
  return head_dim == 128 ? launch_decode<MODE, 128, QT>(p, tmk, tmv, num_seqs, s)
                         : launch_decode<MODE, 64, QT>(p, tmk, tmv, num_seqs, s);
}

}  // namespace

extern "C" size_t pa_decode_workspace_bytes(int num_seqs, int num_q_heads, int num_kv_heads,
                                            int head_dim, int max_blocks_per_seq, int window,
                                            int partition_blocks) {
  if (num_seqs < 0 || num_q_heads < 1 || num_kv_heads < 1 || num_q_heads % num_kv_heads ||
      (head_dim != 64 && head_dim != 128) || max_blocks_per_seq < 1 || window < 0)
    return (size_t)-1;
  const int G = num_q_heads / num_kv_heads;
  const int row_groups = (G + kDecHeads - 1) / kDecHeads;
  const Split s = choose_split(num_seqs, num_kv_heads, row_groups, max_blocks_per_seq, window,
                               partition_blocks);
  return workspace_for(num_seqs, num_q_heads, head_dim, s);
}

namespace {

// pa_decode_partitioned, and with k_new / v_new (of kv_dtype) the write of the
// step's new rows in the same launch (pa_decode_append).
pa_status decode_call(const pa_cache* cache, void* out, const void* q, pa_dtype q_dtype,
                      int num_seqs, int num_q_heads, const int32_t* block_tables,
                      int max_blocks_per_seq, const int32_t* context_lens, float sm_scale,
                      int window, int partition_blocks, void* workspace, size_t workspace_bytes,
                      int32_t* err_flag, void* stream, const void* k_new, const void* v_new,
                      pa_dtype kv_dtype) {
  using pa_internal::aligned16;
  pa_status st = pa_internal::check_cache(cache);
  if (st != PA_OK) return st;
  if (num_seqs < 0 || num_q_heads < 1 || num_q_heads % cache->num_kv_heads ||
      max_blocks_per_seq < 1 || window < 0 || !err_flag ||
      !(sm_scale == sm_scale) || sm_scale > 3.0e38f || sm_scale < -3.0e38f)
    return PA_ERR_INVALID_ARG;
  if (num_seqs == 0) return PA_OK;
  if (!out || !q || !block_tables || !context_lens) return PA_ERR_INVALID_ARG;
  if (!aligned16(out) || !aligned16(q) || !aligned16(block_tables) || !aligned16(context_lens) ||
      !aligned16(err_flag))
    return PA_ERR_INVALID_ARG;
  if (cache->dtype == PA_I8) {
    if (q_dtype != PA_F16 && q_dtype != PA_BF16) return PA_ERR_UNSUPPORTED;
  } else if (q_dtype != cache->dtype) {
    return PA_ERR_UNSUPPORTED;
  }
  if (k_new || v_new) {  // the step's new rows: q's 16-bit type, 16-byte aligned
    if (!k_new || !v_new || !aligned16(k_new) || !aligned16(v_new)) return PA_ERR_INVALID_ARG;
    if (kv_dtype != q_dtype) return PA_ERR_UNSUPPORTED;
  }
  if (num_seqs > 65535 || !pa_internal::cache_rows_fit(cache)) return PA_ERR_UNSUPPORTED;
  if ((long long)max_blocks_per_seq * kBlock > 0x7fffffffLL) return PA_ERR_UNSUPPORTED;

  const int G = num_q_heads / cache->num_kv_heads;
  const int row_groups = (G + kDecHeads - 1) / kDecHeads;
  const Split sp = choose_split(num_seqs, cache->num_kv_heads, row_groups, max_blocks_per_seq,
                                window, partition_blocks);
  const size_t need = workspace_for(num_seqs, num_q_heads, cache->head_dim, sp);
  if (need > 0 && (!workspace || !aligned16(workspace) || workspace_bytes < need))
    return PA_ERR_INVALID_ARG;
  if ((long long)sp.num_parts * cache->num_kv_heads * row_groups > 0x7fffffffLL)
    return PA_ERR_UNSUPPORTED;

  AttnParams p = {};
  p.q = q;
  p.out = out;
  p.k_cache = static_cast<const uint8_t*>(cache->k_cache);
  p.v_cache = static_cast<const uint8_t*>(cache->v_cache);
  p.k_scale = cache->k_scale;
  p.v_scale = cache->v_scale;
  p.block_tables = block_tables;
  p.context_lens = context_lens;
  p.err = err_flag;
  p.num_blocks = cache->num_blocks;
  p.num_kv_heads = cache->num_kv_heads;
  p.num_q_heads = num_q_heads;
  p.group = G;
  p.row_groups = row_groups;
  p.max_blocks_per_seq = max_blocks_per_seq;
  p.window = window;
  p.part_blocks = sp.part_blocks;
  p.num_parts = sp.num_parts;
  p.merge_mode = sp.mode;
  p.min_part_blocks = sp.min_part_blocks;
  p.scale_log2 = sm_scale * 1.4426950408889634f;
  p.k_new = k_new;
  p.v_new = v_new;
  if (need > 0) {
    const size_t n = (size_t)num_seqs * num_q_heads * sp.num_parts;
    p.ws_o = static_cast<float*>(workspace);
    p.ws_m = p.ws_o + n * cache->head_dim;
    p.ws_l = p.ws_m + n;
  }

  CUtensorMap tmk, tmv;
  if (!pa_internal::encode_cache_map(&tmk, cache, cache->k_cache) ||
      !pa_internal::encode_cache_map(&tmv, cache, cache->v_cache))
    return pa_internal::cuda_status(cudaErrorInvalidValue);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  const int D = cache->head_dim;
  if (cache->dtype == PA_F16) e = launch_decode_d<kF16, __half>(p, tmk, tmv, D, num_seqs, s);
  else if (cache->dtype == PA_BF16) e = launch_decode_d<kBF16, __nv_bfloat16>(p, tmk, tmv, D, num_seqs, s);
  else if (q_dtype == PA_F16) e = launch_decode_d<kI8, __half>(p, tmk, tmv, D, num_seqs, s);
  else e = launch_decode_d<kI8, __nv_bfloat16>(p, tmk, tmv, D, num_seqs, s);
  return pa_internal::cuda_status(e);
}

}  // namespace

extern "C" pa_status pa_decode_partitioned(const pa_cache* cache, void* out, const void* q,
                                           pa_dtype q_dtype, int num_seqs, int num_q_heads,
                                           const int32_t* block_tables, int max_blocks_per_seq,
                                           const int32_t* context_lens, float sm_scale, int window,
                                           int partition_blocks, void* workspace,
                                           size_t workspace_bytes, int32_t* err_flag,
                                           void* stream) {
  return decode_call(cache, out, q, q_dtype, num_seqs, num_q_heads, block_tables,
                     max_blocks_per_seq, context_lens, sm_scale, window, partition_blocks,
                     workspace, workspace_bytes, err_flag, stream, nullptr, nullptr, q_dtype);
}

extern "C" pa_status pa_decode_append(const pa_cache* cache, const void* k_new,
                                      const void* v_new, pa_dtype kv_dtype, void* out,
                                      const void* q, pa_dtype q_dtype, int num_seqs,
                                      int num_q_heads, const int32_t* block_tables,
                                      int max_blocks_per_seq, const int32_t* context_lens,
                                      float sm_scale, int window, void* workspace,
                                      size_t workspace_bytes, int32_t* err_flag, void* stream) {
  if (num_seqs > 0 && (!k_new || !v_new)) return PA_ERR_INVALID_ARG;
  return decode_call(cache, out, q, q_dtype, num_seqs, num_q_heads, block_tables,
                     max_blocks_per_seq, context_lens, sm_scale, window, 0, workspace,
                     workspace_bytes, err_flag, stream, k_new, v_new, kv_dtype);
}

extern "C" pa_status pa_decode(const pa_cache* cache, void* out, const void* q, pa_dtype q_dtype,
                               int num_seqs, int num_q_heads, const int32_t* block_tables,
                               int max_blocks_per_seq, const int32_t* context_lens, float sm_scale,
                               int window, void* workspace, size_t workspace_bytes,
                               int32_t* err_flag, void* stream) {
  return pa_decode_partitioned(cache, out, q, q_dtype, num_seqs, num_q_heads, block_tables,
                               max_blocks_per_seq, context_lens, sm_scale, window, 0, workspace,
                               workspace_bytes, err_flag, stream);
}

// ---------------------------------------------------------------------------
// pa_decode_noalloc: pa_decode for callers that cannot allocate device memory.
//
// The split-K partials go to a fixed scratch array compiled into this library
// (PA_NOALLOC_SCRATCH_BYTES per device, held from the moment a device loads the
// library until the process exits) instead of a workspace the caller passes.
// Its device address is looked up once per device, on that device's first call,
// with the device current; host code never hands the array's name itself to a
// kernel, because on the host that name only stands in for the device symbol.
// Nothing in the scratch has to start at zero: every partial a merge reads was
// written earlier in the same call.  All calls on a device share the one array,
// so calls whose kernels can overlap on the GPU (different streams, or host
// threads without ordering between them) corrupt each other's partials.
namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[PA_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mu;
void* g_noalloc_addr[kMaxDevices];                // device address of the scratch, per device
unsigned long long g_noalloc_ctx[kMaxDevices];    // id of the context it was looked up in

// Unique id of the calling thread's current context (0 if the driver cannot say).
// A device reset ends the context the cached address belongs to; the next call
// sees a new id and looks the address up again.
unsigned long long current_context_id() {
  typedef CUresult (*GetCurrentFn)(CUcontext*);
  typedef CUresult (*GetIdFn)(CUcontext, unsigned long long*);
  static GetCurrentFn get_current = []() -> GetCurrentFn {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) !=
            cudaSuccess || q != cudaDriverEntryPointSuccess)
      return nullptr;
    return reinterpret_cast<GetCurrentFn>(f);
  }();
  static GetIdFn get_id = []() -> GetIdFn {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) !=
            cudaSuccess || q != cudaDriverEntryPointSuccess)
      return nullptr;
    return reinterpret_cast<GetIdFn>(f);
  }();
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || !ctx ||
      get_id(ctx, &id) != CUDA_SUCCESS)
    return 0;
  return id;
}

pa_status noalloc_scratch(void** addr) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return pa_internal::cuda_status(e);
  if (dev < 0 || dev >= kMaxDevices) return PA_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (!g_noalloc_addr[dev]) {  // first call on this device: the runtime makes its context
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || p == nullptr)
      return pa_internal::cuda_status(e != cudaSuccess ? e : cudaErrorInvalidSymbol);
    g_noalloc_addr[dev] = p;
    g_noalloc_ctx[dev] = current_context_id();
  } else {
    const unsigned long long id = current_context_id();
    if (id != g_noalloc_ctx[dev]) {  // the device was reset since: look it up again
      void* p = nullptr;
      e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
      if (e != cudaSuccess || p == nullptr)
        return pa_internal::cuda_status(e != cudaSuccess ? e : cudaErrorInvalidSymbol);
      g_noalloc_addr[dev] = p;
      g_noalloc_ctx[dev] = current_context_id();  // the lookup may have made the context
    }
  }
  *addr = g_noalloc_addr[dev];
  return PA_OK;
}

}  // namespace

extern "C" pa_status pa_decode_noalloc(const pa_cache* cache, void* out, const void* q,
                                       pa_dtype q_dtype, int num_seqs, int num_q_heads,
                                       const int32_t* block_tables, int max_blocks_per_seq,
                                       const int32_t* context_lens, float sm_scale, int window,
                                       int32_t* err_flag, void* stream) {
  pa_status st = pa_internal::check_cache(cache);
  if (st != PA_OK) return st;
  if (num_seqs < 0) return PA_ERR_INVALID_ARG;
  if (num_seqs == 0) return PA_OK;
  const size_t need =
      pa_decode_workspace_bytes(num_seqs, num_q_heads, cache->num_kv_heads, cache->head_dim,
                                max_blocks_per_seq, window, 0);
  if (need == (size_t)-1) return PA_ERR_INVALID_ARG;
  if (need > (size_t)PA_NOALLOC_SCRATCH_BYTES) return PA_ERR_UNSUPPORTED;
  void* scratch = nullptr;
  if (need > 0) {
    st = noalloc_scratch(&scratch);
    if (st != PA_OK) return st;
  }
  return pa_decode_partitioned(cache, out, q, q_dtype, num_seqs, num_q_heads, block_tables,
                               max_blocks_per_seq, context_lens, sm_scale, window, 0, scratch,
                               need, err_flag, stream);
}
