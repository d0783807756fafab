// pa_linear.cu -- weight-only INT8 linear for decode-sized batches
// ("PyTorch LLM Serving Engine", What is implemented: symmetric per-output-
// channel INT8 weights and a fused backend that reads the quantized weight tiles
// directly; "MicroGen", Key Features: static per-channel INT8 weights).
//
// y[m][n] = scale[n] * sum_k x[m][k] * code[n][k] (+ bias[n]).  The weights
// dominate the bytes (n*k codes against (m+n)*... activations), so the kernel
// streams the codes from HBM once and is bound by bandwidth.  A CTA owns 16
// output channels (the MMA's M) and up to 16 tokens (two N=8 MMAs); its 8 warps
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

// NT token groups of 8 (1 or 2).  Grid: x = channel group, y = 16-token group,
// z = split of the k blocks.  The loads are only in flight while their warps
// are resident, so for up to 8 tokens the registers are held to five CTAs per
// SM (40 warps; no spill): a 688-CTA grid, the 11008-channel projections, then
// runs in one wave instead of a full wave and a short second one.
// The matrix whose channel tiles hold this CTA's.
__device__ __forceinline__ int tile_matrix(const LinParams& p) {
  int mat = 0;
#pragma unroll
  for (int i = 1; i < kMaxGroup; i++)
    if (i < p.count && (int)blockIdx.x >= p.tile0[i]) mat = i;
  return mat;
}

template <typename XT, int NT>
__global__ void __launch_bounds__(kThreads, NT == 1 ? 5 : 4) int8_linear_kernel(const LinParams p) {
  __shared__ float red[kWarps][NT * 8][kCh];
  __shared__ float part[NT * 8][kCh];  // this split's sums, for the cluster merge
  pdl_wait();  // the kernel before (say, the one that wrote x) is complete
  pdl_launch_dependents();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  const int m0 = blockIdx.y * 16;
  const int8_t* wg;
  {
    const int mat = tile_matrix(p);
    wg = p.codes[mat] + (size_t)(((int)blockIdx.x - p.tile0[mat]) * kCh + g) * p.k;
  }
  const int8_t* wg8 = wg + (size_t)8 * p.k;
  const XT* xs = static_cast<const XT*>(p.x);
  const XT* xrow[NT];
  bool xvalid[NT];
#pragma unroll
  for (int tg = 0; tg < NT; tg++) {
    const int m = m0 + 8 * tg + g;
    xvalid[tg] = m < p.m;
    xrow[tg] = xs + (size_t)(xvalid[tg] ? m : 0) * p.k;
  }
  float acc[NT][4];
#pragma unroll
  for (int tg = 0; tg < NT; tg++)
#pragma unroll
    for (int i = 0; i < 4; i++) acc[tg][i] = 0.0f;

  const int nblocks = p.k / kKB;
  const int stride = p.splits * kWarps;
  int b = blockIdx.z * kWarps + warp;
  // one block ahead: codes of rows g and g+8, 16 bytes each
  uint4 wa = make_uint4(0, 0, 0, 0), wb = wa;
  if (b < nblocks) {
    wa = ld_stream(wg + (size_t)b * kKB + 16 * t);
    wb = ld_stream(wg8 + (size_t)b * kKB + 16 * t);
  }
  for (; b < nblocks; b += stride) {
    const uint4 ca = wa, cb = wb;
    const int bn = b + stride;
    if (bn < nblocks) {
      wa = ld_stream(wg + (size_t)bn * kKB + 16 * t);
      wb = ld_stream(wg8 + (size_t)bn * kKB + 16 * t);
    }
    uint4 xa[NT], xb[NT];
#pragma unroll
    for (int tg = 0; tg < NT; tg++) {
      const uint4* px = reinterpret_cast<const uint4*>(xrow[tg] + (size_t)b * kKB + 16 * t);
      xa[tg] = xvalid[tg] ? px[0] : make_uint4(0, 0, 0, 0);
      xb[tg] = xvalid[tg] ? px[1] : make_uint4(0, 0, 0, 0);
    }
    const uint32_t wra[4] = {ca.x, ca.y, ca.z, ca.w}, wrb[4] = {cb.x, cb.y, cb.z, cb.w};
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
        mma16816<false>(acc[tg], a, to_f16x2<XT>(xw[2 * j]), to_f16x2<XT>(xw[2 * j + 1]));
      }
    }
  }
  // C fragment: acc[tg][0..1] = channel g, tokens 2t, 2t+1; [2..3] = channel g+8
#pragma unroll
  for (int tg = 0; tg < NT; tg++) {
    red[warp][8 * tg + 2 * t][g] = acc[tg][0];
    red[warp][8 * tg + 2 * t + 1][g] = acc[tg][1];
    red[warp][8 * tg + 2 * t][g + 8] = acc[tg][2];
    red[warp][8 * tg + 2 * t + 1][g + 8] = acc[tg][3];
  }
  __syncthreads();
  const int mat = tile_matrix(p);
  const int n0 = ((int)blockIdx.x - p.tile0[mat]) * kCh;
  const int N = p.n[mat];
  const float* scales = p.scales[mat];
  const XT* bias = static_cast<const XT*>(p.bias[mat]);
  XT* y = static_cast<XT*>(p.y[mat]);
  for (int idx = threadIdx.x; idx < NT * 8 * kCh; idx += kThreads) {
    const int mi = idx / kCh, c = idx % kCh;
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
      for (int idx = threadIdx.x; idx < NT * 8 * kCh; idx += kThreads) {
        const int mi = idx / kCh, c = idx % kCh;
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

template <typename XT>
cudaError_t launch_linear(const pa_dev::lin::LinParams& p, long long tiles, cudaStream_t s) {
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
    e = p.m <= 8 ? cudaLaunchKernelEx(&cfg, int8_linear_kernel<XT, 1>, p)
                 : cudaLaunchKernelEx(&cfg, int8_linear_kernel<XT, 2>, p);
    return e != cudaSuccess ? e : cudaGetLastError();
  }
  e = p.m <= 8 ? pa_internal::launch_dependent(int8_linear_kernel<XT, 1>, grid, dim3(kThreads),
                                               0, s, 1u, p)
               : pa_internal::launch_dependent(int8_linear_kernel<XT, 2>, grid, dim3(kThreads),
                                               0, s, 1u, p);
  if (e != cudaSuccess || p.splits == 1) return e;
  const size_t total = (size_t)p.m * p.n[0];
  return pa_internal::launch_dependent(int8_linear_reduce<XT>,
                                       dim3((unsigned)((total + 255) / 256)), dim3(256), 0, s, 1u,
                                       p);
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
  long long tiles = 0;
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
    p.tile0[i] = (int)tiles;
    tiles += n[i] / kCh;
  }
  if (tiles > 0x7fffffffLL || (m + 15) / 16 > 65535) return PA_ERR_UNSUPPORTED;
  p.count = count;
  p.x = x;
  p.m = m;
  p.k = k;
  p.splits = std::min(choose_splits(tiles, m, 0, k, 0, sm_count_linear()), kMaxClusterSplits);
  p.cluster = p.splits > 1 ? 1 : 0;
  p.ws = nullptr;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const cudaError_t e = x_dtype == PA_F16 ? launch_linear<__half>(p, tiles, s)
                                          : launch_linear<__nv_bfloat16>(p, tiles, s);
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
  p.cluster = p.splits > 1 && p.splits <= kMaxClusterSplits ? 1 : 0;
  p.ws = static_cast<float*>(workspace);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const cudaError_t e = x_dtype == PA_F16 ? launch_linear<__half>(p, n / kCh, s)
                                          : launch_linear<__nv_bfloat16>(p, n / kCh, s);
  return pa_internal::cuda_status(e);
}
