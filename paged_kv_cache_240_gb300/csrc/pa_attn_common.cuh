// pa_attn_common.cuh -- pieces shared by the decode and chunked-prefill
// attention kernels.
//
// CTA layout: warps 0..3 are consumers, warp 4 is the producer.  The producer
// walks the sequence's block table (32 entries per coalesced load) and, for each
// logical block, has one thread issue TMA tensor copies of the (block, kv head)
// K and V tiles -- 16 rows x head_dim of the cache viewed as a 2-D tensor
// [num_blocks*num_kv_heads*16, head_dim] -- plus bulk copies of the int8
// scales, into a ring of shared-memory stages; the copies complete on a
// per-stage mbarrier.  Consumers wait on that barrier, run the block through
// tensor-core MMAs and an online-softmax update, and release the stage.  Block
// ids outside the pool are never copied: the stage is marked invalid and its
// keys are left out.
//
// Per-warp math (m16n8k16 MMA, fp32 accumulate).  A warp owns 16 query rows
// (GQA heads of one token for decode, (token, head) pairs for prefill):
//   S  = Q K^T    A = Q rows (registers), B = the block's 16 K rows (ldmatrix)
//   online softmax on S in the log2 domain, per row
//   O += P V      A = P (f16/bf16), B = the block's 16 V rows (ldmatrix.trans)
// For int8 caches the codes are turned into exact f16 integers in registers, the
// K scale multiplies the scores and the V scale goes into P as a value weight with
// its own running reference (pa_device.cuh), so dequantised values are never
// materialised.
#pragma once

#include <type_traits>

#include "pa_device.cuh"

namespace pa_dev {

constexpr int kConsumerWarps = 4;
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr int kStages = 8;
constexpr int kRowsPerWarp = 16;

struct AttnParams {
  const void* q;
  void* out;
  const uint8_t* k_cache;
  const uint8_t* v_cache;
  const float* k_scale;
  const float* v_scale;
  const int32_t* block_tables;
  const int32_t* context_lens;
  const int32_t* cu_q_lens;  // prefill only
  float* ws_o;               // decode split-K partials
  float* ws_m;
  float* ws_l;
  int32_t* err;
  int num_blocks, num_kv_heads, num_q_heads, group, row_groups;
  int max_blocks_per_seq, window;
  int part_blocks, num_parts;        // decode: blocks per partition, partitions per (seq, head)
  int num_q_tokens, max_q_len, q_tiles;  // prefill
  float scale_log2;                  // sm_scale * log2(e)
  // decode: how partitions are formed and merged (kMergeWorkspace: fixed
  // part_blocks per partition, partials merged by a second kernel;
  // kMergeCluster: each sequence's blocks split evenly into at most num_parts
  // partitions of at least min_part_blocks, merged inside the launch)
  int merge_mode, min_part_blocks;
  // decode: the step's new rows [num_seqs][num_kv_heads][D] (q's type) to write
  // at each sequence's position L-1 before attending, or null
  const void* k_new;
  const void* v_new;
};
constexpr int kMergeWorkspace = 0, kMergeCluster = 1;

// Shared-memory layout of one CTA (from a base aligned to the swizzle atom):
// stages, int8 scales, barriers and per-stage flags.  After the pipeline drains,
// the decode kernel reuses the stage area to merge its warps' states.
template <int MODE, int D>
struct Smem {
  using T = Tile<MODE, D>;
  static constexpr int kMergeStride = D + 4;  // fp32 row stride of the warp-merge area
  static constexpr int kMergeBytes = kConsumerWarps * kRowsPerWarp * (kMergeStride + 2) * 4;
  static constexpr int kStagesBytes = kStages * T::kStageBytes;
  static constexpr int kDataBytes = kStagesBytes > kMergeBytes ? kStagesBytes : kMergeBytes;
  static constexpr int kScaleOff = (kDataBytes + 127) / 128 * 128;
  static constexpr int kBarOff = kScaleOff + kStages * T::kScaleBytes;
  static constexpr int kUsed = kBarOff + 2 * kStages * 8 + kStages * 4 + 16;
  static constexpr int kBytes = kUsed + T::kAlign;  // room to align the base
};

struct SmemPtrs {
  uint8_t* stages;
  float* scales;  // [stage][K 16 | V 16]
  uint64_t* full;
  uint64_t* empty;
  int* valid;
  int* abort_flag;
};

template <int MODE, int D>
__device__ __forceinline__ SmemPtrs smem_ptrs(uint8_t* raw) {
  using S = Smem<MODE, D>;
  const uint32_t a = smem_u32(raw);
  uint8_t* smem = raw + ((Tile<MODE, D>::kAlign - (a & (Tile<MODE, D>::kAlign - 1))) &
                         (Tile<MODE, D>::kAlign - 1));
  SmemPtrs s;
  s.stages = smem;
  s.scales = reinterpret_cast<float*>(smem + S::kScaleOff);
  s.full = reinterpret_cast<uint64_t*>(smem + S::kBarOff);
  s.empty = s.full + kStages;
  s.valid = reinterpret_cast<int*>(s.empty + kStages);
  s.abort_flag = s.valid + kStages;
  return s;
}

__device__ __forceinline__ void init_barriers(const SmemPtrs& s, int full_count,
                                              int empty_count) {
  if (threadIdx.x == 0) {
#pragma unroll
    for (int i = 0; i < kStages; i++) {
      mbar_init(&s.full[i], full_count);
      mbar_init(&s.empty[i], empty_count);
    }
    *s.abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
}

// Producer warp: fill stages for logical blocks table[0 .. nblk-1] of kv head
// kvh.  The warp loads 32 table entries at a time; lane 0 issues the copies.
template <int MODE, int D>
__device__ __forceinline__ void produce(const AttnParams& p, const void* tmk, const void* tmv,
                                        const SmemPtrs& s, const int32_t* table, int kvh,
                                        int nblk, int lane) {
  using T = Tile<MODE, D>;
  int issued = 0;
  bool stop = false;
  for (int base = 0; base < nblk && !stop; base += 32) {
    const int mine = base + lane < nblk ? table[base + lane] : -1;
    const int cnt = min(32, nblk - base);
    for (int j = 0; j < cnt; j++) {
      const int i = base + j;
      const int slot = i % kStages;
      if (i >= kStages && !mbar_wait(&s.empty[slot], ((i / kStages) - 1) & 1)) {
        if (lane == 0) set_flag(p.err, PA_FLAG_TIMEOUT);
        stop = true;
        break;
      }
      const int phys = __shfl_sync(0xffffffffu, mine, j);
      if (lane == 0) {
        const bool ok = phys >= 0 && phys < p.num_blocks;
        s.valid[slot] = ok ? 1 : 0;
        if (ok) {
          mbar_arrive_expect_tx(&s.full[slot], T::kTxBytes);
          uint8_t* st = s.stages + slot * T::kStageBytes;
          const int row0 = (phys * p.num_kv_heads + kvh) * kBlock;
#pragma unroll
          for (int h = 0; h < T::kChunks; h++) {
            tma_load_2d(st + h * T::kBoxBytes, tmk, h * T::kChunkElems, row0, &s.full[slot]);
            tma_load_2d(st + T::kTileBytes + h * T::kBoxBytes, tmv, h * T::kChunkElems, row0,
                        &s.full[slot]);
          }
        } else {
          set_flag(p.err, PA_FLAG_BLOCK_ID);
          mbar_arrive(&s.full[slot]);
        }
      }
      if constexpr (MODE == kI8) {
        // the two 64-byte scale runs: lanes 0-3 K, lanes 4-7 V, 16 bytes each
        if (lane < T::kScaleLanes) {
          if (phys >= 0 && phys < p.num_blocks) {
            const long long row0 = ((long long)phys * p.num_kv_heads + kvh) * kBlock;
            const float* src = (lane < 4 ? p.k_scale : p.v_scale) + row0 + 4 * (lane & 3);
            cp_async_16(s.scales + slot * 2 * kBlock + (lane < 4 ? 0 : kBlock) + 4 * (lane & 3),
                        src);
            cp_async_arrive_noinc(&s.full[slot]);
          } else {
            mbar_arrive(&s.full[slot]);
          }
        }
      }
      __syncwarp();
      issued = i + 1;
    }
  }
  // No copy may still be landing in shared memory when the CTA exits.
  if (lane == 0)
    for (int i = issued > kStages ? issued - kStages : 0; i < issued; i++)
      if (!mbar_wait(&s.full[i % kStages], (i / kStages) & 1)) {
        set_flag(p.err, PA_FLAG_TIMEOUT);
        break;
      }
}

// Q rows -> A fragments.  f16/bf16 caches: k-step ks covers d = 16ks..16ks+15 in
// the natural order.  int8 caches: the K tile is read with ldmatrix on bytes, so
// a thread holds the four codes d = 16c+4t..16c+4t+3 of a row; the k-slots of
// step c are mapped to those d (slots 2t,2t+1 -> d+0,1; slots 2t+8,2t+9 -> d+2,3)
// and Q is laid out the same way (a dot product does not depend on the order).
// int8 caches with bf16 q: each row is scaled by a power of two into f16 range
// (q_prescale_shift); shift[r] receives that shift (0 otherwise).
template <int MODE, int D, typename QT>
__device__ __forceinline__ void load_q(uint32_t (&qa)[D / 16][4], const QT* row0, const QT* row1,
                                       int t, int (&shift)[2]) {
  const QT* rows[2] = {row0, row1};
  shift[0] = shift[1] = 0;
  if constexpr (MODE != kI8) {
#pragma unroll
    for (int ks = 0; ks < D / 16; ks++)
#pragma unroll
      for (int r = 0; r < 2; r++) {
        qa[ks][r] = rows[r] ? *reinterpret_cast<const uint32_t*>(rows[r] + 16 * ks + 2 * t) : 0u;
        qa[ks][2 + r] =
            rows[r] ? *reinterpret_cast<const uint32_t*>(rows[r] + 16 * ks + 8 + 2 * t) : 0u;
      }
  } else {
    constexpr bool kBf16Q = !std::is_same<QT, __half>::value;
    float mul[2] = {1.0f, 1.0f};
    if constexpr (kBf16Q) {
#pragma unroll
      for (int r = 0; r < 2; r++) {
        float amax = 0.0f;
        if (rows[r]) {
#pragma unroll
          for (int ks = 0; ks < D / 16; ks++) {
            const uint2 raw = *reinterpret_cast<const uint2*>(rows[r] + 16 * ks + 4 * t);
            const __nv_bfloat16* e = reinterpret_cast<const __nv_bfloat16*>(&raw);
#pragma unroll
            for (int j = 0; j < 4; j++) amax = fmaxf(amax, fabsf(__bfloat162float(e[j])));
          }
        }
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
        shift[r] = q_prescale_shift(amax);
        mul[r] = pow2i(-shift[r]);
      }
    }
#pragma unroll
    for (int ks = 0; ks < D / 16; ks++) {
#pragma unroll
      for (int r = 0; r < 2; r++) {
        uint32_t lo = 0, hi = 0;
        if (rows[r]) {
          const uint2 raw = *reinterpret_cast<const uint2*>(rows[r] + 16 * ks + 4 * t);
          if constexpr (!kBf16Q) {
            lo = raw.x;
            hi = raw.y;
          } else {
            const __nv_bfloat16* e = reinterpret_cast<const __nv_bfloat16*>(&raw);
            lo = pack_f16(__bfloat162float(e[0]) * mul[r], __bfloat162float(e[1]) * mul[r]);
            hi = pack_f16(__bfloat162float(e[2]) * mul[r], __bfloat162float(e[3]) * mul[r]);
          }
        }
        qa[ks][r] = lo;      // a0a1 / a2a3: rows gid / gid+8, first k pair
        qa[ks][2 + r] = hi;  // a4a5 / a6a7: rows gid / gid+8, second k pair
      }
    }
  }
}

// Output column d held by C-fragment column n of PV n-tile nt.
template <int MODE, int D>
__device__ __forceinline__ int o_col(int nt, int n) {
  if constexpr (MODE == kI8) return (D / 8) * n + nt;
  else return 8 * nt + n;
}

// One 16-token block through one warp's 16 rows.  pos0 is the logical position
// of the block's first token; row r of this thread (gid, gid+8) sees keys in
// [row_lo[r], row_hi[r]] and its scores are scaled by rsc[r] (sm_scale * log2(e),
// times the row's query prescale for int8 caches with bf16 q).  Tokens outside
// [keep_lo, keep_hi] may hold garbage (tail slots, data before the window) and
// their V rows are zeroed before PV (int8: their weight is 0 and codes are finite).
// int8 caches: P is the value weight 2^(s + log2 v_scale - n[r]) of pa_device.cuh,
// O is relative to the running reference n[r] and l to the softmax maximum m[r].
template <int MODE, int D>
__device__ __forceinline__ void attend_block(const uint32_t (&qa)[D / 16][4], float (&o)[D / 8][4],
                                             float (&m)[2], float (&l)[2], float (&n)[2],
                                             const uint8_t* stage, const float* scales, int lane,
                                             int pos0, const int (&row_lo)[2],
                                             const int (&row_hi)[2], int keep_lo, int keep_hi,
                                             const float (&rsc)[2]) {
  using T = Tile<MODE, D>;
  constexpr bool BF = MODE == kBF16;
  const int t = lane & 3;
  const int mi = lane >> 3, mr = lane & 7;
  const uint32_t kbase = smem_u32(stage);
  const uint32_t vbase = kbase + T::kTileBytes;

  // ---- S = Q K^T: two n-tiles of 8 tokens
  float s[2][4];
#pragma unroll
  for (int nt = 0; nt < 2; nt++)
#pragma unroll
    for (int i = 0; i < 4; i++) s[nt][i] = 0.0f;
  const int krow = 8 * (mi >> 1) + mr;  // token row this lane addresses for ldmatrix
  if constexpr (MODE != kI8) {
#pragma unroll
    for (int ks = 0; ks < D / 16; ks++) {
      uint32_t b[4];
      ldsm_x4(b, kbase + T::off(krow, 32 * ks + 16 * (mi & 1)));
      mma16816<BF>(s[0], qa[ks], b[0], b[1]);
      mma16816<BF>(s[1], qa[ks], b[2], b[3]);
    }
  } else {
#pragma unroll
    for (int c = 0; c < D / 16; c += 2) {
      uint32_t r[4], lo, hi;
      ldsm_x4(r, kbase + T::off(krow, 16 * (c + (mi & 1))));
      biased_i8x4_to_f16(r[0], lo, hi);
      mma16816<false>(s[0], qa[c], lo, hi);
      biased_i8x4_to_f16(r[1], lo, hi);
      mma16816<false>(s[0], qa[c + 1], lo, hi);
      biased_i8x4_to_f16(r[2], lo, hi);
      mma16816<false>(s[1], qa[c], lo, hi);
      biased_i8x4_to_f16(r[3], lo, hi);
      mma16816<false>(s[1], qa[c + 1], lo, hi);
    }
  }

  // ---- scale, mask, online softmax (log2 domain)
  float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
  for (int nt = 0; nt < 2; nt++)
#pragma unroll
    for (int i = 0; i < 4; i++) {
      const int tok = 8 * nt + 2 * t + (i & 1);
      const int r = i >> 1;
      const int pos = pos0 + tok;
      float x = s[nt][i] * rsc[r];
      if constexpr (MODE == kI8) x *= scales[tok];
      x = (pos >= row_lo[r] && pos <= row_hi[r]) ? x : -INFINITY;
      s[nt][i] = x;
      mx[r] = fmaxf(mx[r], x);
    }
  float ref[2], corr[2];
#pragma unroll
  for (int r = 0; r < 2; r++) {
    mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 1));
    mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 2));
    const float mn = fmaxf(m[r], mx[r]);
    ref[r] = mn == -INFINITY ? 0.0f : mn;
    corr[r] = exp2f(m[r] - ref[r]);
    m[r] = mn;
  }
  float ls[2] = {0.0f, 0.0f};
  if constexpr (MODE != kI8) {
#pragma unroll
    for (int nt = 0; nt < 2; nt++)
#pragma unroll
      for (int i = 0; i < 4; i++) {
        const float e = exp2f(s[nt][i] - ref[i >> 1]);
        ls[i >> 1] += e;
        s[nt][i] = e;
      }
#pragma unroll
    for (int r = 0; r < 2; r++) l[r] = l[r] * corr[r] + ls[r];
    // The running maximum rarely moves once a few blocks are in: skip the
    // rescale when no row of the warp needs it.
    if (!__all_sync(0xffffffffu, corr[0] == 1.0f && corr[1] == 1.0f)) {
#pragma unroll
      for (int nt = 0; nt < D / 8; nt++) {
        o[nt][0] *= corr[0];
        o[nt][1] *= corr[0];
        o[nt][2] *= corr[1];
        o[nt][3] *= corr[1];
      }
    }
  } else {
    // value weights: y = s + log2 v_scale (-inf where the row does not see the
    // key, whatever its slot holds), relative to n, which moves up when a weight
    // would pass 2^kLazyV
    float lgv[2][2];
#pragma unroll
    for (int nt = 0; nt < 2; nt++)
#pragma unroll
      for (int j = 0; j < 2; j++) {
        const int pos = pos0 + 8 * nt + 2 * t + j;
        lgv[nt][j] = pos >= keep_lo && pos <= keep_hi
                         ? fast_log2(scales[kBlock + 8 * nt + 2 * t + j])
                         : -INFINITY;
      }
    float y[2][4];
    bool grow = false;
#pragma unroll
    for (int nt = 0; nt < 2; nt++)
#pragma unroll
      for (int i = 0; i < 4; i++) {
        const float e = exp2f(s[nt][i] - ref[i >> 1]);
        ls[i >> 1] += e;
        y[nt][i] = s[nt][i] + lgv[nt][i & 1];
        grow |= y[nt][i] > n[i >> 1] + kLazyV;
      }
#pragma unroll
    for (int r = 0; r < 2; r++) l[r] = l[r] * corr[r] + ls[r];
    if (__any_sync(0xffffffffu, grow)) {
#pragma unroll
      for (int r = 0; r < 2; r++) {
        float ym = fmaxf(fmaxf(y[0][2 * r], y[0][2 * r + 1]), fmaxf(y[1][2 * r], y[1][2 * r + 1]));
        ym = fmaxf(ym, __shfl_xor_sync(0xffffffffu, ym, 1));
        ym = fmaxf(ym, __shfl_xor_sync(0xffffffffu, ym, 2));
        const float nn = fmaxf(n[r], ym);
        const float f = fast_exp2(n[r] - nn);
        n[r] = nn;
#pragma unroll
        for (int nt = 0; nt < D / 8; nt++) {
          o[nt][2 * r] *= f;
          o[nt][2 * r + 1] *= f;
        }
      }
    }
#pragma unroll
    for (int nt = 0; nt < 2; nt++)
#pragma unroll
      for (int i = 0; i < 4; i++) s[nt][i] = fast_exp2(y[nt][i] - n[i >> 1]);
  }
  uint32_t pa[4];
  pa[0] = pack2<BF>(s[0][0], s[0][1]);  // row gid,   tokens 2t, 2t+1
  pa[1] = pack2<BF>(s[0][2], s[0][3]);  // row gid+8, tokens 2t, 2t+1
  pa[2] = pack2<BF>(s[1][0], s[1][1]);  // row gid,   tokens 2t+8, 2t+9
  pa[3] = pack2<BF>(s[1][2], s[1][3]);  // row gid+8, tokens 2t+8, 2t+9

  // ---- O += P V
  if constexpr (MODE != kI8) {
    const int vrow = 8 * (mi & 1) + mr;
    if (pos0 >= keep_lo && pos0 + kBlock - 1 <= keep_hi) {
#pragma unroll
      for (int n2 = 0; n2 < D / 16; n2++) {
        uint32_t b[4];
        ldsm_x4_t(b, vbase + T::off(vrow, 16 * (2 * n2 + (mi >> 1))));
        mma16816<BF>(o[2 * n2], pa, b[0], b[1]);
        mma16816<BF>(o[2 * n2 + 1], pa, b[2], b[3]);
      }
    } else {
      auto keep = [&](int tok) {
        const int pos = pos0 + tok;
        return pos >= keep_lo && pos <= keep_hi;
      };
      const uint32_t mk01 = (keep(2 * t) ? 0x0000ffffu : 0u) | (keep(2 * t + 1) ? 0xffff0000u : 0u);
      const uint32_t mk89 =
          (keep(2 * t + 8) ? 0x0000ffffu : 0u) | (keep(2 * t + 9) ? 0xffff0000u : 0u);
#pragma unroll
      for (int n2 = 0; n2 < D / 16; n2++) {
        uint32_t b[4];
        ldsm_x4_t(b, vbase + T::off(vrow, 16 * (2 * n2 + (mi >> 1))));
        mma16816<BF>(o[2 * n2], pa, b[0] & mk01, b[1] & mk89);
        mma16816<BF>(o[2 * n2 + 1], pa, b[2] & mk01, b[3] & mk89);
      }
    }
  } else {
    // Thread (gid, t) reads bytes [W*4*gid, W*4*gid + W*4) of V rows 2t, 2t+1,
    // 2t+8, 2t+9; n-tile nt then holds column d = (D/8)*gid + nt.
    constexpr int W = D / 32;
    const int gid = lane >> 2;
    const uint8_t* vt = stage + T::kTileBytes;
    uint32_t R[4][W];
    const int toks[4] = {2 * t, 2 * t + 1, 2 * t + 8, 2 * t + 9};
#pragma unroll
    for (int j = 0; j < 4; j++) {
      if constexpr (W == 4) {
        const uint4 v4 = *reinterpret_cast<const uint4*>(vt + T::off(toks[j], 16 * gid));
        R[j][0] = v4.x;
        R[j][1] = v4.y;
        R[j][2] = v4.z;
        R[j][3] = v4.w;
      } else {
        const uint2 v2 = *reinterpret_cast<const uint2*>(vt + T::off(toks[j], 8 * gid));
        R[j][0] = v2.x;
        R[j][1] = v2.y;
      }
    }
#pragma unroll
    for (int w = 0; w < W; w++) {
      uint32_t p0, p1, q0, q1;
      biased_i8_pairs<0>(R[0][w], R[1][w], p0, p1);
      biased_i8_pairs<0>(R[2][w], R[3][w], q0, q1);
      mma16816<false>(o[4 * w + 0], pa, p0, q0);
      mma16816<false>(o[4 * w + 1], pa, p1, q1);
      biased_i8_pairs<2>(R[0][w], R[1][w], p0, p1);
      biased_i8_pairs<2>(R[2][w], R[3][w], q0, q1);
      mma16816<false>(o[4 * w + 2], pa, p0, q0);
      mma16816<false>(o[4 * w + 3], pa, p1, q1);
    }
  }
}

__device__ __forceinline__ int clamp_context(const AttnParams& p, int seq, bool report) {
  const int cap = p.max_blocks_per_seq * kBlock;
  int L = p.context_lens[seq];
  if (L < 0 || L > cap) {
    if (report) set_flag(p.err, PA_FLAG_CONTEXT_LEN);
    L = L < 0 ? 0 : cap;
  }
  return L;
}

}  // namespace pa_dev
