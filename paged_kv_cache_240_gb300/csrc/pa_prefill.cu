// pa_prefill.cu -- chunked-prefill attention over the paged cache ("PyTorch LLM
// Serving Engine", "What is implemented": configurable prefill chunks share the
// step with decode; "Loading": online softmax while walking the block table).
//
// The queries of one sequence's chunk and one kv head form C*G rows, row
// R = c*G + j being query token c and query head kvh*G + j (GQA).  A CTA takes 64
// consecutive rows (16 per consumer warp) and walks every block its rows can see
// (the union of their causal/window ranges).  All four warps read each stage;
// each masks per row (key position <= its query position, and > position - W
// when windowed) and skips blocks that none of its rows sees.
#include <algorithm>

#include "pa_attn_common.cuh"
#include "pa_internal.h"

namespace pa_dev {

constexpr int kTileRows = kConsumerWarps * kRowsPerWarp;

template <int MODE, int D, typename QT>
__global__ void __launch_bounds__(kThreads)
    pa_prefill_kernel(const __grid_constant__ AttnParams p, const __grid_constant__ CUtensorMap tmk,
                     const __grid_constant__ CUtensorMap tmv) {
  extern __shared__ __align__(128) uint8_t smem[];
  pdl_wait();  // the kernel before (say, the K/V write) is complete
  pdl_launch_dependents();
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
  if (C > L && reporter) set_flag(p.err, PA_FLAG_Q_LEN);  // early queries see nothing
  const int R0 = tile * kTileRows;
  const int nrows = C * G;
  if (R0 >= nrows) return;

  // Keys any row of this tile can see.
  const int c_first = R0 / G;
  const int c_last = (min(R0 + kTileRows, nrows) - 1) / G;
  const int pos_first = L - C + c_first, pos_last = L - C + c_last;
  const int hi_u = pos_last;
  const int lo_u = p.window > 0 ? max(0, pos_first - p.window + 1) : 0;
  const int first = lo_u / kBlock;
  const int nblk = hi_u >= lo_u ? hi_u / kBlock - first + 1 : 0;

  const SmemPtrs s = smem_ptrs<MODE, D>(smem);
  init_barriers(s, Tile<MODE, D>::kFullArrivals, kConsumerWarps);
  const int32_t* table = p.block_tables + (long long)n * p.max_blocks_per_seq + first;

  if (warp == kConsumerWarps) {
    produce<MODE, D>(p, &tmk, &tmv, s, table, kvh, nblk, lane);
    return;
  }

  // ---------------- consumer warps: rows R0 + 16*warp + gid (+8)
  const int gid = lane >> 2, t = lane & 3;
  const QT* q = static_cast<const QT*>(p.q);
  const QT* qrow[2];
  int row_lo[2], row_hi[2];
  long long orow[2];
#pragma unroll
  for (int r = 0; r < 2; r++) {
    const int R = R0 + kRowsPerWarp * warp + gid + 8 * r;
    qrow[r] = nullptr;
    row_lo[r] = 0;
    row_hi[r] = -1;  // sees nothing
    orow[r] = -1;
    if (R < nrows) {
      const int c = R / G, j = R % G;
      const int pos = L - C + c;
      orow[r] = (long long)(q0 + c) * p.num_q_heads + kvh * G + j;
      qrow[r] = q + orow[r] * D;
      row_hi[r] = pos;
      row_lo[r] = p.window > 0 ? max(0, pos - p.window + 1) : 0;
    }
  }
  // Union of this warp's row ranges: blocks outside it are skipped.
  int wlo = row_hi[0] >= row_lo[0] ? row_lo[0] : 0x7fffffff;
  int whi = row_hi[0];
  if (row_hi[1] >= row_lo[1]) {
    wlo = min(wlo, row_lo[1]);
    whi = max(whi, row_hi[1]);
  }
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    wlo = min(wlo, __shfl_xor_sync(0xffffffffu, wlo, off));
    whi = max(whi, __shfl_xor_sync(0xffffffffu, whi, off));
  }

  uint32_t qa[D / 16][4];
  int qshift[2];
  load_q<MODE, D, QT>(qa, qrow[0], qrow[1], t, qshift);
  const float rsc[2] = {p.scale_log2 * pow2i(qshift[0]), p.scale_log2 * pow2i(qshift[1])};
  float o[D / 8][4];
#pragma unroll
  for (int nt = 0; nt < D / 8; nt++)
#pragma unroll
    for (int i = 0; i < 4; i++) o[nt][i] = 0.0f;
  float m[2] = {-INFINITY, -INFINITY}, l[2] = {0.0f, 0.0f};
  float nref[2] = {kNoRef, kNoRef};  // int8: the value weights' reference

  bool timed_out = false;
  for (int i = 0; i < nblk; i++) {
    const int slot = i % kStages;
    if (!mbar_wait(&s.full[slot], (i / kStages) & 1)) {
      if (lane == 0) set_flag(p.err, PA_FLAG_TIMEOUT);
      timed_out = true;
      break;
    }
    const int pos0 = (first + i) * kBlock;
    if (s.valid[slot] && pos0 <= whi && pos0 + kBlock - 1 >= wlo)
      attend_block<MODE, D>(qa, o, m, l, nref, s.stages + slot * Tile<MODE, D>::kStageBytes,
                            s.scales + slot * 2 * kBlock, lane, pos0,
                            row_lo, row_hi, lo_u, hi_u, rsc);
    __syncwarp();
    if (lane == 0) mbar_arrive(&s.empty[slot]);
  }
  if (timed_out) return;
#pragma unroll
  for (int r = 0; r < 2; r++) {
    l[r] += __shfl_xor_sync(0xffffffffu, l[r], 1);
    l[r] += __shfl_xor_sync(0xffffffffu, l[r], 2);
  }
  QT* out = static_cast<QT*>(p.out);
#pragma unroll
  for (int r = 0; r < 2; r++) {
    if (orow[r] < 0) continue;
    // int8: O is relative to the value weights' reference, l to m
    float inv = l[r] > 0.0f ? 1.0f / l[r] : 0.0f;
    if constexpr (MODE == kI8) inv = l[r] > 0.0f ? exp2f(nref[r] - m[r]) / l[r] : 0.0f;
    QT* dst = out + orow[r] * D;
#pragma unroll
    for (int nt = 0; nt < D / 8; nt++) {
      dst[o_col<MODE, D>(nt, 2 * t)] = to_out<QT>(o[nt][2 * r] * inv);
      dst[o_col<MODE, D>(nt, 2 * t + 1)] = to_out<QT>(o[nt][2 * r + 1] * inv);
    }
  }
}

// The tensor-memory kernel for 16-bit caches (pa_prefill_tc.cu).
template <int D, typename QT>
cudaError_t launch_prefill_tc(const AttnParams& p, const CUtensorMap& tmk, const CUtensorMap& tmv,
                              int num_seqs, cudaStream_t stream);

}  // namespace pa_dev

using namespace pa_dev;

namespace {

template <int MODE, int D, typename QT>
cudaError_t launch_prefill(const AttnParams& p, const CUtensorMap& tmk, const CUtensorMap& tmv,
                           int num_seqs, cudaStream_t stream) {
  constexpr int smem = Smem<MODE, D>::kBytes;
  auto kern = pa_prefill_kernel<MODE, D, QT>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const dim3 grid((unsigned)(p.q_tiles * p.num_kv_heads), (unsigned)num_seqs);
  return pa_internal::launch_dependent(kern, grid, dim3(kThreads), smem, stream, 1u, p, tmk, tmv);
}

template <int MODE, typename QT>
cudaError_t launch_prefill_d(const AttnParams& p, const CUtensorMap& tmk, const CUtensorMap& tmv,
                           int head_dim, int num_seqs, cudaStream_t s) {
  return head_dim == 128 ? launch_prefill<MODE, 128, QT>(p, tmk, tmv, num_seqs, s)
                         : launch_prefill<MODE, 64, QT>(p, tmk, tmv, num_seqs, s);
}

}  // namespace

extern "C" pa_status pa_prefill_chunk(const pa_cache* cache, void* out, const void* q,
                                      pa_dtype q_dtype, int num_q_tokens, int num_seqs,
                                      int num_q_heads, const int32_t* cu_q_lens, int max_q_len,
                                      const int32_t* block_tables, int max_blocks_per_seq,
                                      const int32_t* context_lens, float sm_scale, int window,
                                      void* workspace, size_t workspace_bytes, int32_t* err_flag,
                                      void* stream) {
  (void)workspace;
  (void)workspace_bytes;
  using pa_internal::aligned16;
  pa_status st = pa_internal::check_cache(cache);
  if (st != PA_OK) return st;
  if (num_q_tokens < 0 || num_seqs < 0 || num_q_heads < 1 ||
      num_q_heads % cache->num_kv_heads || max_q_len < 0 || max_blocks_per_seq < 1 ||
      window < 0 || !err_flag || !(sm_scale == sm_scale) || sm_scale > 3.0e38f ||
      sm_scale < -3.0e38f)
    return PA_ERR_INVALID_ARG;
  if (num_seqs == 0 || num_q_tokens == 0 || max_q_len == 0) return PA_OK;
  if (!out || !q || !cu_q_lens || !block_tables || !context_lens) return PA_ERR_INVALID_ARG;
  if (!aligned16(out) || !aligned16(q) || !aligned16(cu_q_lens) || !aligned16(block_tables) ||
      !aligned16(context_lens) || !aligned16(err_flag))
    return PA_ERR_INVALID_ARG;
  if (cache->dtype == PA_I8) {
    if (q_dtype != PA_F16 && q_dtype != PA_BF16) return PA_ERR_UNSUPPORTED;
  } else if (q_dtype != cache->dtype) {
    return PA_ERR_UNSUPPORTED;
  }
  if (num_seqs > 65535 || !pa_internal::cache_rows_fit(cache)) return PA_ERR_UNSUPPORTED;
  if ((long long)max_blocks_per_seq * kBlock > 0x7fffffffLL) return PA_ERR_UNSUPPORTED;
  const int G = num_q_heads / cache->num_kv_heads;
  const long long tiles = ((long long)max_q_len * G + kTileRows - 1) / kTileRows;
  if (tiles * cache->num_kv_heads > 0x7fffffffLL || (long long)max_q_len * G > 0x7fffffffLL)
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
  p.cu_q_lens = cu_q_lens;
  p.err = err_flag;
  p.num_blocks = cache->num_blocks;
  p.num_kv_heads = cache->num_kv_heads;
  p.num_q_heads = num_q_heads;
  p.group = G;
  p.row_groups = 1;
  p.max_blocks_per_seq = max_blocks_per_seq;
  p.window = window;
  p.num_q_tokens = num_q_tokens;
  p.max_q_len = max_q_len;
  p.q_tiles = (int)tiles;
  p.scale_log2 = sm_scale * 1.4426950408889634f;

  CUtensorMap tmk, tmv;
  if (!pa_internal::encode_cache_map(&tmk, cache, cache->k_cache) ||
      !pa_internal::encode_cache_map(&tmv, cache, cache->v_cache))
    return pa_internal::cuda_status(cudaErrorInvalidValue);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  const int D = cache->head_dim;
  if (cache->dtype != PA_I8) {
    // 16-bit caches: tcgen05 kernel (sizes its own grid)
    const bool bf = cache->dtype == PA_BF16;
    if (D == 128)
      e = bf ? launch_prefill_tc<128, __nv_bfloat16>(p, tmk, tmv, num_seqs, s)
             : launch_prefill_tc<128, __half>(p, tmk, tmv, num_seqs, s);
    else
      e = bf ? launch_prefill_tc<64, __nv_bfloat16>(p, tmk, tmv, num_seqs, s)
             : launch_prefill_tc<64, __half>(p, tmk, tmv, num_seqs, s);
  } else if (q_dtype == PA_F16) {
    e = launch_prefill_d<kI8, __half>(p, tmk, tmv, D, num_seqs, s);
  } else {
    e = launch_prefill_d<kI8, __nv_bfloat16>(p, tmk, tmv, D, num_seqs, s);
  }
  return pa_internal::cuda_status(e);
}
