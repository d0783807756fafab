// pa_linear.cu -- weight-only INT8 linear for decode-sized batches
// ("PyTorch LLM Serving Engine", What is implemented: symmetric per-output-
// channel INT8 weights and a fused backend that reads the quantized weight tiles
// directly; "MicroGen", Key Features: static per-channel INT8 weights).
//
// y[m][n] = scale[n] * sum_k x[m][k] * code[n][k] (+ bias[n]).  The weights
// dominate the bytes (n*k codes against (m+n)*... activations), so the kernel
// streams the codes from HBM once and is bound by bandwidth.  A CTA owns 16 or
// 32 output channels (one or two MMA row tiles of M=16; the launch's plan picks)
// and up to 16 tokens (two N=8 MMAs); its 8 warps
// take interleaved 64-wide k blocks and add their partial sums in shared memory.
// Codes become exact f16 integers in registers (byte permute under 0x64, then
// subtract 1152) and meet the activations in mma.sync m16n8k16 with fp32
// accumulation.  Within a 64-wide k block the products are summed in a permuted
// order -- thread t of a quad reads 16 consecutive codes and activations, so
// every load is 16 contiguous bytes -- which changes only the rounding order.
//
// Up to four matrices that read the same activations (a layer's q, k and v
// projections, or gate and up) run as one launch: the grid's channel tiles are
// the matrices' tiles one after the other.  When the channel tiles are too few
// to fill the GPU, the k blocks are split across CTAs; up to 8 splits of a
// channel tile form one thread-block cluster and the first CTA adds the others'
// partial sums over distributed shared memory (in split order, as a separate
// reduce kernel would), so no workspace and no second launch are needed.  More
// splits (tiny matrices with a long k) go through the workspace and a reduce
// kernel.
#include <algorithm>
#include <mutex>

#include "pa_device.cuh"
#include "pa_internal.h"
#include "pa_linear.h"

namespace pa_dev {
namespace lin {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kCh = 16;   // output channels per CTA
constexpr int kKB = 64;   // k per block

constexpr int kMaxGroup = 4;     // matrices per launch
constexpr int kMaxClusterSplits = 8;

struct LinParams {
  const int8_t* codes[kMaxGroup];
  const float* scales[kMaxGroup];
  const void* bias[kMaxGroup];
  void* y[kMaxGroup];
  int n[kMaxGroup];
  int tile0[kMaxGroup];  // first channel tile of each matrix in the grid
  int count;             // matrices in this launch
  const void* x;
  float* ws;     // workspace merge: [splits][m][n] partial sums (one matrix), or nullptr
  int m, k, splits;
  int cluster;   // splits > 1 merged in the launch (cluster along z)
};

__device__ __forceinline__ void cluster_sync_all() {
  asm volatile(
      "barrier.cluster.arrive.release.aligned;\n\t"
      "barrier.cluster.wait.acquire.aligned;" ::: "memory");
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

// 16 bytes of codes, read once: not kept in L1, and the whole 256-byte L2 line
// fetched (the warps next to this one read its other 64-byte blocks next).
__device__ __forceinline__ uint4 ld_stream(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.L2::256B.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// Two activations (one 32-bit word of fp16 or bf16) as an f16x2 MMA operand.
template <typename XT>
__device__ __forceinline__ uint32_t to_f16x2(uint32_t v) {
  if constexpr (std::is_same<XT, __half>::value) {
    return v;
  } else {
    const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&v));
    return pack_f16(f.x, f.y);
  }
}

template <typename XT>
__device__ __forceinline__ float ld_act(const XT* p) {
  if constexpr (std::is_same<XT, __half>::value) return __half2float(*p);
  else return __bfloat162float(*p);
}

// The matrix whose channel tiles hold this CTA's.
__device__ __forceinline__ int tile_matrix(const LinParams& p) {
  int mat = 0;
#pragma unroll
  for (int i = 1; i < kMaxGroup; i++)
    if (i < p.count && (int)blockIdx.x >= p.tile0[i]) mat = i;
  return mat;
}

// NT token groups of 8 (1 or 2), RT channel tiles of 16 (1 or 2: a CTA owns
// 16 * RT channels).  Grid: x = channel group, y = 16-token group, z = split of
// the k blocks.  The loads are only in flight while their warps are resident,
// so for up to 8 tokens and one channel tile the registers are held to five
// CTAs per SM (40 warps; no spill).  Two channel tiles double the bytes each
// warp keeps in flight (codes of four rows) and halve the CTAs: a launch whose
// 16-channel tiles would need a short second wave runs in one (see plan_linear).
template <typename XT, int NT, int RT>
__global__ void __launch_bounds__(kThreads, NT == 1 ? (RT == 1 ? 5 : 3) : (RT == 1 ? 4 : 2))
    int8_linear_kernel(const LinParams p) {
  constexpr int kCtaCh = kCh * RT;
  __shared__ float red[kWarps][NT * 8][kCtaCh];
  __shared__ float part[NT * 8][kCtaCh];  // this split's sums, for the cluster merge
  pdl_wait();  // the kernel before (say, the one that wrote x) is complete
  pdl_launch_dependents();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  const int m0 = blockIdx.y * 16;
  const int8_t* wg[RT];  // row g of channel tile r (row g + 8 is 8 rows further)
  {
    const int mat = tile_matrix(p);
#pragma unroll
    for (int r = 0; r < RT; r++)
      wg[r] = p.codes[mat] +
              (size_t)(((int)blockIdx.x - p.tile0[mat]) * kCtaCh + r * kCh + g) * p.k;
  }
  const size_t row8 = (size_t)8 * p.k;
  const XT* xs = static_cast<const XT*>(p.x);
  const XT* xrow[NT];
  bool xvalid[NT];
#pragma unroll
  for (int tg = 0; tg < NT; tg++) {
    const int m = m0 + 8 * tg + g;
    xvalid[tg] = m < p.m;
    xrow[tg] = xs + (size_t)(xvalid[tg] ? m : 0) * p.k;
  }
  float acc[NT][RT][4];
#pragma unroll
  for (int tg = 0; tg < NT; tg++)
#pragma unroll
    for (int r = 0; r < RT; r++)
#pragma unroll
      for (int i = 0; i < 4; i++) acc[tg][r][i] = 0.0f;

  const int nblocks = p.k / kKB;
  const int stride = p.splits * kWarps;
  int b = blockIdx.z * kWarps + warp;
  // one block ahead: codes of rows g and g+8 of each channel tile, 16 bytes each
  uint4 wa[RT], wb[RT];
#pragma unroll
  for (int r = 0; r < RT; r++) {
    wa[r] = make_uint4(0, 0, 0, 0);
    wb[r] = wa[r];
    if (b < nblocks) {
      wa[r] = ld_stream(wg[r] + (size_t)b * kKB + 16 * t);
      wb[r] = ld_stream(wg[r] + row8 + (size_t)b * kKB + 16 * t);
    }
  }
  for (; b < nblocks; b += stride) {
    uint4 ca[RT], cb[RT];
#pragma unroll
    for (int r = 0; r < RT; r++) {
      ca[r] = wa[r];
      cb[r] = wb[r];
    }
    const int bn = b + stride;
    if (bn < nblocks) {
#pragma unroll
      for (int r = 0; r < RT; r++) {
        wa[r] = ld_stream(wg[r] + (size_t)bn * kKB + 16 * t);
        wb[r] = ld_stream(wg[r] + row8 + (size_t)bn * kKB + 16 * t);
      }
    }
    uint4 xa[NT], xb[NT];
#pragma unroll
    for (int tg = 0; tg < NT; tg++) {
      const uint4* px = reinterpret_cast<const uint4*>(xrow[tg] + (size_t)b * kKB + 16 * t);
      xa[tg] = xvalid[tg] ? px[0] : make_uint4(0, 0, 0, 0);
      xb[tg] = xvalid[tg] ? px[1] : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int r = 0; r < RT; r++) {
      const uint32_t wra[4] = {ca[r].x, ca[r].y, ca[r].z, ca[r].w};
      const uint32_t wrb[4] = {cb[r].x, cb[r].y, cb[r].z, cb[r].w};
#pragma unroll
      for (int j = 0; j < 4; j++) {
        // k-step j: this thread's codes k + 16t + 4j .. +3 of rows g and g+8, in
        // the A slots (2t, 2t+1) and (2t+8, 2t+9); the activations the same.
        uint32_t a[4];
        biased_i8x4_to_f16(wra[j] ^ 0x80808080u, a[0], a[2]);
        biased_i8x4_to_f16(wrb[j] ^ 0x80808080u, a[1], a[3]);
#pragma unroll
        for (int tg = 0; tg < NT; tg++) {
          const uint32_t xw[8] = {xa[tg].x, xa[tg].y, xa[tg].z, xa[tg].w,
                                  xb[tg].x, xb[tg].y, xb[tg].z, xb[tg].w};
          mma16816<false>(acc[tg][r], a, to_f16x2<XT>(xw[2 * j]), to_f16x2<XT>(xw[2 * j + 1]));
        }
      }
    }
  }
  // C fragment: acc[tg][r][0..1] = channel g of tile r, tokens 2t, 2t+1; [2..3] = channel g+8
#pragma unroll
  for (int tg = 0; tg < NT; tg++)
#pragma unroll
    for (int r = 0; r < RT; r++) {
      red[warp][8 * tg + 2 * t][r * kCh + g] = acc[tg][r][0];
      red[warp][8 * tg + 2 * t + 1][r * kCh + g] = acc[tg][r][1];
      red[warp][8 * tg + 2 * t][r * kCh + g + 8] = acc[tg][r][2];
      red[warp][8 * tg + 2 * t + 1][r * kCh + g + 8] = acc[tg][r][3];
    }
  __syncthreads();
  const int mat = tile_matrix(p);
  const int n0 = ((int)blockIdx.x - p.tile0[mat]) * kCtaCh;
  const int N = p.n[mat];
  const float* scales = p.scales[mat];
  const XT* bias = static_cast<const XT*>(p.bias[mat]);
  XT* y = static_cast<XT*>(p.y[mat]);
  for (int idx = threadIdx.x; idx < NT * 8 * kCtaCh; idx += kThreads) {
    const int mi = idx / kCtaCh, c = idx % kCtaCh;
    const int m = m0 + mi, n = n0 + c;
    if (m >= p.m) continue;
    float s = 0.0f;
#pragma unroll
    for (int w = 0; w < kWarps; w++) s += red[w][mi][c];
    if (p.cluster) {
      part[mi][c] = s;
    } else if (p.splits > 1) {
      p.ws[((size_t)blockIdx.z * p.m + m) * N + n] = s;
    } else {
      float v = scales[n] * s;
      if (bias) v += ld_act<XT>(bias + n);
      y[(size_t)m * N + n] = to_out<XT>(v);
    }
  }
  if (p.cluster) {
    // the splits of this channel tile are one cluster (rank = split): the first
    // adds the others' sums in split order, then scale, bias and the cast
    cluster_sync_all();
    if (blockIdx.z == 0) {
      for (int idx = threadIdx.x; idx < NT * 8 * kCtaCh; idx += kThreads) {
        const int mi = idx / kCtaCh, c = idx % kCtaCh;
        const int m = m0 + mi, n = n0 + c;
        if (m >= p.m) continue;
        float s = 0.0f;
        for (int z = 0; z < p.splits; z++) s += ld_cluster_f32(&part[mi][c], (uint32_t)z);
        float v = scales[n] * s;
        if (bias) v += ld_act<XT>(bias + n);
        y[(size_t)m * N + n] = to_out<XT>(v);
      }
    }
    cluster_sync_all();  // no CTA leaves while the first still reads its sums
  }
}

// Sum of the splits' partial sums, then scale, bias and the cast.
template <typename XT>
__global__ void int8_linear_reduce(const LinParams p) {
  pdl_wait();  // the partial sums are written
  pdl_launch_dependents();
  const size_t idx = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int N = p.n[0];
  if (idx >= (size_t)p.m * N) return;
  const int n = (int)(idx % N);
  float s = 0.0f;
  for (int z = 0; z < p.splits; z++) s += p.ws[(size_t)z * p.m * N + idx];
  float v = p.scales[0][n] * s;
  if (p.bias[0]) v += ld_act<XT>(static_cast<const XT*>(p.bias[0]) + n);
  static_cast<XT*>(p.y[0])[idx] = to_out<XT>(v);
}

// One warp per output channel: amax, scale = amax / 127, codes rounded half to
// even (IEEE division and conversion, as the INT8 KV quantiser).
template <typename WT>
__global__ void int8_quantize_kernel(const WT* w, int n, int k, int8_t* codes, float* scales) {
  const int row = blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= n) return;
  const WT* src = w + (size_t)row * k;
  float amax = 0.0f;
  for (int i = lane; i < k; i += 32) amax = fmaxf(amax, fabsf(ld_act<WT>(src + i)));
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
  const float scale = __fdiv_rn(amax, 127.0f);
  int8_t* dst = codes + (size_t)row * k;
  for (int i = lane; i < k; i += 32) {
    int c = 0;
    if (scale > 0.0f) {
      c = __float2int_rn(__fdiv_rn(ld_act<WT>(src + i), scale));
      c = min(127, max(-127, c));
    }
    dst[i] = (int8_t)c;
  }
  if (lane == 0) scales[row] = scale;
}

}  // namespace lin
}  // namespace pa_dev

namespace {

using pa_internal::aligned16;

int sm_count_linear() {
  int dev = 0, count = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return count;
}

// Splits of the k blocks: enough thread blocks for two per SM, at most one
// k block per warp.  Up to kMaxClusterSplits merge inside the launch; beyond
// that, only as many as the workspace holds.
int choose_splits(long long tiles, int m, int n, int k, size_t ws_bytes, int sms) {
  const long long ctas = tiles * ((m + 15) / 16);
  const int nblocks = k / pa_dev::lin::kKB;
  int splits = 1;
  if (sms > 0 && ctas < 2LL * sms)
    splits = (int)std::min<long long>((2LL * sms + ctas - 1) / ctas,
                                      std::max(1, nblocks / pa_dev::lin::kWarps));
  if (splits <= pa_dev::lin::kMaxClusterSplits) return splits;
  while (splits > pa_dev::lin::kMaxClusterSplits &&
         (size_t)splits * m * n * sizeof(float) > ws_bytes)
    splits--;
  return std::max(1, splits);
}

// Resident CTAs per SM of one kernel instance on the current device (asked of
// the occupancy calculator once per device and instance).
template <typename XT, int NT, int RT>
int resident_per_sm() {
  static std::mutex mu;
  static int known[64];  // 0 unknown
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 1;
  std::lock_guard<std::mutex> lock(mu);
  if (known[dev] == 0) {
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(
            &n, pa_dev::lin::int8_linear_kernel<XT, NT, RT>, pa_dev::lin::kThreads, 0) !=
            cudaSuccess ||
        n < 1)
      n = 1;
    cudaGetLastError();
    known[dev] = n;
  }
  return known[dev];
}

template <typename XT>
int resident_per_sm(int m, int rt) {
  if (m <= 8) return rt == 1 ? resident_per_sm<XT, 1, 1>() : resident_per_sm<XT, 1, 2>();
  return rt == 1 ? resident_per_sm<XT, 2, 1>() : resident_per_sm<XT, 2, 2>();
}

// Channel tiles of 16 or 32 per CTA (rt = 1, 2) and k splits merged over a
// cluster, chosen by a model of the launch: a warp streams its k blocks one
// memory round trip at a time (one block ahead), so a CTA takes about as many
// round trips as its warp has blocks, whatever its channel count; the launch
// takes that times its waves of resident CTAs, but no less than its bytes at
// the HBM rate, plus a little per wave (CTA start-up) and for a merge.  A
// 32-channel tile keeps twice the bytes in flight per warp with half the CTAs:
// it takes a launch whose 16-channel tiles would need a second, nearly empty
// wave (768 tiles of a q/k/v projection group against 760 resident CTAs) into
// one wave.
struct LinPlan {
  int rt, splits;
};

// The plan is made for launches of up to 8 tokens (one N=8 MMA per k step),
// where it was measured (a LLaMA-7B layer stack: 3,616 -> 4,137 GB/s); with
// more tokens the kernel does twice the MMAs per byte and keeps the 16-channel
// tiles and the SM-filling split of choose_splits (the same model picked 32-
// channel tiles there and measured 12 % slower).
template <typename XT>
LinPlan plan_linear(long long tiles16, bool rt2_ok, int m, int k, long long bytes, int sms) {
  using namespace pa_dev::lin;
  if (m > 8) return {1, std::min(choose_splits(tiles16, m, 0, k, 0, sms), kMaxClusterSplits)};
  constexpr double kRoundTripUs = 1.0, kHbmBytesPerUs = 6.5e6, kWaveUs = 0.5, kMergeUs = 0.3;
  const int nblocks = k / kKB;
  const long long mtiles = (m + 15) / 16;
  LinPlan best = {1, 1};
  double best_t = 1e30;
  for (int rt = 1; rt <= (rt2_ok ? 2 : 1); rt++) {
    const long long slots = (long long)std::max(sms, 1) * resident_per_sm<XT>(m, rt);
    const int max_splits = std::max(1, std::min(kMaxClusterSplits, nblocks / kWarps));
    for (int sp = 1; sp <= max_splits; sp++) {
      const long long ctas = tiles16 / rt * mtiles * sp;
      const long long waves = (ctas + slots - 1) / slots;
      const int per_warp = (nblocks + sp * kWarps - 1) / (sp * kWarps);
      const double t = std::max((double)(waves * per_warp) * kRoundTripUs,
                                (double)bytes / kHbmBytesPerUs) +
                       waves * kWaveUs + (sp > 1 ? kMergeUs : 0.0);
      if (t < best_t - 1e-9) {
        best_t = t;
        best = {rt, sp};
      }
    }
  }
  return best;
}

template <typename XT, int RT>
cudaError_t launch_linear_rt(const pa_dev::lin::LinParams& p, long long tiles, cudaStream_t s) {
  using namespace pa_dev::lin;
  const dim3 grid((unsigned)tiles, (unsigned)((p.m + 15) / 16), (unsigned)p.splits);
  // the splits of a channel tile form one cluster (along z) when they merge in
  // the launch; launched as a dependent of the kernel before it in the stream
  cudaError_t e;
  if (p.cluster) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute at[2];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = 1;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = (unsigned)p.splits;
    at[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 2;
    e = p.m <= 8 ? cudaLaunchKernelEx(&cfg, int8_linear_kernel<XT, 1, RT>, p)
                 : cudaLaunchKernelEx(&cfg, int8_linear_kernel<XT, 2, RT>, p);
    return e != cudaSuccess ? e : cudaGetLastError();
  }
  e = p.m <= 8 ? pa_internal::launch_dependent(int8_linear_kernel<XT, 1, RT>, grid,
                                               dim3(kThreads), 0, s, 1u, p)
               : pa_internal::launch_dependent(int8_linear_kernel<XT, 2, RT>, grid,
                                               dim3(kThreads), 0, s, 1u, p);
  if (e != cudaSuccess || p.splits == 1) return e;
  const size_t total = (size_t)p.m * p.n[0];
  return pa_internal::launch_dependent(int8_linear_reduce<XT>,
                                       dim3((unsigned)((total + 255) / 256)), dim3(256), 0, s, 1u,
                                       p);
}

// tiles: CTA channel tiles (16 * rt channels each)
template <typename XT>
cudaError_t launch_linear(const pa_dev::lin::LinParams& p, long long tiles, int rt,
                          cudaStream_t s) {
  return rt == 2 ? launch_linear_rt<XT, 2>(p, tiles, s) : launch_linear_rt<XT, 1>(p, tiles, s);
}

bool misaligned(const void* ptr, uintptr_t mask) {
  return (reinterpret_cast<uintptr_t>(ptr) & mask) != 0;
}

}  // namespace

extern "C" pa_status pa_linear_int8_quantize(const void* w, pa_dtype w_dtype, int n, int k,
                                             int8_t* codes, float* scales, void* stream) {
  if (!w || !codes || !scales || n < 1 || k < 1) return PA_ERR_INVALID_ARG;
  if (w_dtype != PA_F16 && w_dtype != PA_BF16) return PA_ERR_UNSUPPORTED;
  const int rows_per_block = 8;
  const unsigned blocks = (unsigned)((n + rows_per_block - 1) / rows_per_block);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (w_dtype == PA_F16)
    pa_dev::lin::int8_quantize_kernel<__half><<<blocks, 32 * rows_per_block, 0, s>>>(
        static_cast<const __half*>(w), n, k, codes, scales);
  else
    pa_dev::lin::int8_quantize_kernel<__nv_bfloat16><<<blocks, 32 * rows_per_block, 0, s>>>(
        static_cast<const __nv_bfloat16*>(w), n, k, codes, scales);
  return pa_internal::cuda_status(cudaGetLastError());
}

extern "C" size_t pa_linear_int8_workspace_bytes(int m, int n, int k) {
  if (m < 1 || n < pa_dev::lin::kCh || k < pa_dev::lin::kKB) return 0;
  const int splits = choose_splits(n / pa_dev::lin::kCh, m, n, k, (size_t)-1, sm_count_linear());
  return splits > pa_dev::lin::kMaxClusterSplits ? (size_t)splits * m * n * sizeof(float) : 0;
}

extern "C" pa_status pa_linear_int8_grouped(int count, const int8_t* const* codes,
                                            const float* const* scales,
                                            const void* const* bias, const int* n,
                                            const void* x, pa_dtype x_dtype, int m, int k,
                                            void* const* y, void* stream) {
  using namespace pa_dev::lin;
  if (count < 1 || count > kMaxGroup || !codes || !scales || !n || !x || !y || m < 1 || k < 1)
    return PA_ERR_INVALID_ARG;
  if (x_dtype != PA_F16 && x_dtype != PA_BF16) return PA_ERR_UNSUPPORTED;
  if (k % kKB != 0 || k > 65536) return PA_ERR_UNSUPPORTED;
  if (!aligned16(x)) return PA_ERR_INVALID_ARG;
  LinParams p = {};
  long long tiles16 = 0, bytes = 2LL * m * k;
  bool rt2_ok = true;
  for (int i = 0; i < count; i++) {
    const void* b = bias ? bias[i] : nullptr;
    if (!codes[i] || !scales[i] || !y[i] || n[i] < 1) return PA_ERR_INVALID_ARG;
    if (n[i] % kCh != 0) return PA_ERR_UNSUPPORTED;
    if (!aligned16(codes[i]) || misaligned(scales[i], 3) || misaligned(y[i], 1) ||
        misaligned(b, 1))
      return PA_ERR_INVALID_ARG;
    p.codes[i] = codes[i];
    p.scales[i] = scales[i];
    p.bias[i] = b;
    p.y[i] = y[i];
    p.n[i] = n[i];
    tiles16 += n[i] / kCh;
    rt2_ok = rt2_ok && n[i] % (2 * kCh) == 0;
    bytes += (long long)n[i] * k + 4LL * n[i] + 2LL * m * n[i];
  }
  if (tiles16 > 0x7fffffffLL || (m + 15) / 16 > 65535) return PA_ERR_UNSUPPORTED;
  const LinPlan plan = x_dtype == PA_F16
                           ? plan_linear<__half>(tiles16, rt2_ok, m, k, bytes, sm_count_linear())
                           : plan_linear<__nv_bfloat16>(tiles16, rt2_ok, m, k, bytes,
                                                        sm_count_linear());
  long long tiles = 0;  // CTA channel tiles (16 * rt channels)
  for (int i = 0; i < count; i++) {
    p.tile0[i] = (int)tiles;
    tiles += n[i] / (kCh * plan.rt);
  }
  p.count = count;
  p.x = x;
  p.m = m;
  p.k = k;
  p.splits = plan.splits;
  p.cluster = p.splits > 1 ? 1 : 0;
  p.ws = nullptr;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const cudaError_t e = x_dtype == PA_F16 ? launch_linear<__half>(p, tiles, plan.rt, s)
                                          : launch_linear<__nv_bfloat16>(p, tiles, plan.rt, s);
  return pa_internal::cuda_status(e);
}

extern "C" pa_status pa_linear_int8(const int8_t* codes, const float* scales, const void* bias,
                                    const void* x, pa_dtype x_dtype, int m, int n, int k, void* y,
                                    void* workspace, size_t workspace_bytes, void* stream) {
  using namespace pa_dev::lin;
  if (!codes || !scales || !x || !y || m < 1 || n < 1 || k < 1) return PA_ERR_INVALID_ARG;
  if (x_dtype != PA_F16 && x_dtype != PA_BF16) return PA_ERR_UNSUPPORTED;
  if (n % kCh != 0 || k % kKB != 0 || k > 65536) return PA_ERR_UNSUPPORTED;
  if (!aligned16(codes) || !aligned16(x) || misaligned(scales, 3) || misaligned(y, 1) ||
      misaligned(bias, 1) || misaligned(workspace, 3))
    return PA_ERR_INVALID_ARG;
  if ((m + 15) / 16 > 65535) return PA_ERR_UNSUPPORTED;
  LinParams p = {};
  p.codes[0] = codes;
  p.scales[0] = scales;
  p.bias[0] = bias;
  p.y[0] = y;
  p.n[0] = n;
  p.tile0[0] = 0;
  p.count = 1;
  p.x = x;
  p.m = m;
  p.k = k;
  p.splits = choose_splits(n / kCh, m, n, k, workspace ? workspace_bytes : 0, sm_count_linear());
  int rt = 1;
  if (p.splits <= kMaxClusterSplits) {  // the launch's own plan (more splits: the workspace's)
    const long long bytes = (long long)n * k + 4LL * n + 2LL * m * n + 2LL * m * k;
    const LinPlan plan = x_dtype == PA_F16
                             ? plan_linear<__half>(n / kCh, n % (2 * kCh) == 0, m, k, bytes,
                                                   sm_count_linear())
                             : plan_linear<__nv_bfloat16>(n / kCh, n % (2 * kCh) == 0, m, k, bytes,
                                                          sm_count_linear());
    rt = plan.rt;
    p.splits = plan.splits;
  }
  p.cluster = p.splits > 1 && p.splits <= kMaxClusterSplits ? 1 : 0;
  p.ws = static_cast<float*>(workspace);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const long long tiles = n / (kCh * rt);
  const cudaError_t e = x_dtype == PA_F16 ? launch_linear<__half>(p, tiles, rt, s)
                                          : launch_linear<__nv_bfloat16>(p, tiles, rt, s);
  return pa_internal::cuda_status(e);
}
