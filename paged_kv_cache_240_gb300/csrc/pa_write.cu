// pa_write.cu -- KV write: scatter new tokens' K/V rows into their physical
// cache slots, optionally quantising them to int8 with one fp32 scale per
// (token, kv head) row ("PyTorch LLM Serving Engine", "Loading"; "MicroGen",
// Key Features, "Dynamic INT8 KV Quantization: Vector scale").
//
// One warp owns one (token, kv head) row and handles both its K and its V.  The
// row is read and written with coalesced per-lane vectors; for int8 the warp
// finds amax with a butterfly of shuffles, then every lane divides its own
// elements.  Bit-exactness with the CPU oracle rests on three facts: 16-bit ->
// fp32 conversion is exact, fmaxf/fabsf are exact, and __fdiv_rn and
// __float2int_rn are the IEEE round-to-nearest(-even) operations the oracle uses.
// An int8 code c is stored as the byte c + 128 (offset binary), the form the
// attention kernels turn into exact f16 operands without a sign fix-up.
#include <type_traits>

#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa_dev {

struct WriteParams {
  const uint8_t* k;
  const uint8_t* v;
  const int32_t* slot_mapping;
  uint8_t* k_cache;
  uint8_t* v_cache;
  float* k_scale;
  float* v_scale;
  int32_t* err;
  int num_tokens, num_kv_heads, num_blocks;
};

constexpr int kWriteWarps = 8;

// 16-bit cache: copy the row's bits.  D * 2 bytes per row = D/16 bytes per lane.
template <int D>
__global__ void __launch_bounds__(kWriteWarps * 32) write_copy_kernel(WriteParams p) {
  pdl_launch_dependents();  // the attention call after it may start its launch now
  const int lane = threadIdx.x & 31;
  const long long row = (long long)blockIdx.x * kWriteWarps + (threadIdx.x >> 5);
  if (row >= (long long)p.num_tokens * p.num_kv_heads) return;
  const int t = (int)(row / p.num_kv_heads), h = (int)(row % p.num_kv_heads);
  // the row's bits are read together with its slot (neither waits for the other)
  constexpr int kBytes = D * 2;
  using V = typename std::conditional<kBytes / 32 == 8, uint2, uint32_t>::type;  // 8 or 4 B a lane
  const V kv = reinterpret_cast<const V*>(p.k + row * kBytes)[lane];
  const V vv = reinterpret_cast<const V*>(p.v + row * kBytes)[lane];
  const int32_t slot = p.slot_mapping[t];
  if (slot < 0) return;
  if ((long long)slot >= (long long)p.num_blocks * kBlock) {
    if (lane == 0 && h == 0) set_flag(p.err, PA_FLAG_SLOT_RANGE);
    return;
  }
  const long long dst_row = ((long long)(slot / kBlock) * p.num_kv_heads + h) * kBlock + slot % kBlock;
  reinterpret_cast<V*>(p.k_cache + dst_row * kBytes)[lane] = kv;
  reinterpret_cast<V*>(p.v_cache + dst_row * kBytes)[lane] = vv;
}

template <typename IT, int D>
__global__ void __launch_bounds__(kWriteWarps * 32) write_quant_kernel(WriteParams p) {
  pdl_launch_dependents();  // the attention call after it may start its launch now
  constexpr int E = D / 32;  // elements per lane
  const int lane = threadIdx.x & 31;
  const long long row = (long long)blockIdx.x * kWriteWarps + (threadIdx.x >> 5);
  if (row >= (long long)p.num_tokens * p.num_kv_heads) return;
  const int t = (int)(row / p.num_kv_heads), h = (int)(row % p.num_kv_heads);
  // the K and V rows are read together with the slot (neither waits for the other)
  using R = typename std::conditional<E == 4, uint2, uint32_t>::type;
  R raw[2];
#pragma unroll
  for (int which = 0; which < 2; which++)
    raw[which] =
        *reinterpret_cast<const R*>(reinterpret_cast<const IT*>(which ? p.v : p.k) + row * D + lane * E);
  const int32_t slot = p.slot_mapping[t];
  if (slot < 0) return;
  if ((long long)slot >= (long long)p.num_blocks * kBlock) {
    if (lane == 0 && h == 0) set_flag(p.err, PA_FLAG_SLOT_RANGE);
    return;
  }
  const long long dst_row = ((long long)(slot / kBlock) * p.num_kv_heads + h) * kBlock + slot % kBlock;
#pragma unroll
  for (int which = 0; which < 2; which++) {
    float x[E];
    const IT* e = reinterpret_cast<const IT*>(&raw[which]);
#pragma unroll
    for (int i = 0; i < E; i++) x[i] = in_to_f32<IT>(e[i]);
    uint8_t q[E];
    float scale;
    quantize_row<E>(x, q, scale);
    uint8_t* dst = (which ? p.v_cache : p.k_cache) + dst_row * D + lane * E;
    if constexpr (E == 4) {
      *reinterpret_cast<uint32_t*>(dst) = *reinterpret_cast<uint32_t*>(q);
    } else {
      *reinterpret_cast<uint16_t*>(dst) = *reinterpret_cast<uint16_t*>(q);
    }
    if (lane == 0) (which ? p.v_scale : p.k_scale)[dst_row] = scale;
  }
}

}  // namespace pa_dev

using namespace pa_dev;

extern "C" pa_status pa_write_kv(const pa_cache* cache, const void* k, const void* v,
                                 pa_dtype in_dtype, const int32_t* slot_mapping, int num_tokens,
                                 int32_t* err_flag, void* stream) {
  pa_status st = pa_internal::check_cache(cache);
  if (st != PA_OK) return st;
  if (num_tokens < 0 || !err_flag) return PA_ERR_INVALID_ARG;
  if (num_tokens == 0) return PA_OK;
  if (!k || !v || !slot_mapping) return PA_ERR_INVALID_ARG;
  if (!pa_internal::aligned16(k) || !pa_internal::aligned16(v) ||
      !pa_internal::aligned16(slot_mapping) || !pa_internal::aligned16(err_flag))
    return PA_ERR_INVALID_ARG;
  if (in_dtype != PA_F16 && in_dtype != PA_BF16) return PA_ERR_UNSUPPORTED;
  if (cache->dtype != PA_I8 && cache->dtype != in_dtype) return PA_ERR_UNSUPPORTED;

  WriteParams p;
  p.k = static_cast<const uint8_t*>(k);
  p.v = static_cast<const uint8_t*>(v);
  p.slot_mapping = slot_mapping;
  p.k_cache = static_cast<uint8_t*>(cache->k_cache);
  p.v_cache = static_cast<uint8_t*>(cache->v_cache);
  p.k_scale = cache->k_scale;
  p.v_scale = cache->v_scale;
  p.err = err_flag;
  p.num_tokens = num_tokens;
  p.num_kv_heads = cache->num_kv_heads;
  p.num_blocks = cache->num_blocks;

  const long long rows = (long long)num_tokens * cache->num_kv_heads;
  const long long grid = (rows + kWriteWarps - 1) / kWriteWarps;
  if (grid > 0x7fffffffLL) return PA_ERR_UNSUPPORTED;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const dim3 g((unsigned)grid), b(kWriteWarps * 32);
  const bool d128 = cache->head_dim == 128;
  if (cache->dtype != PA_I8) {
    if (d128) write_copy_kernel<128><<<g, b, 0, s>>>(p);
    else write_copy_kernel<64><<<g, b, 0, s>>>(p);
  } else if (in_dtype == PA_F16) {
    if (d128) write_quant_kernel<__half, 128><<<g, b, 0, s>>>(p);
    else write_quant_kernel<__half, 64><<<g, b, 0, s>>>(p);
  } else {
    if (d128) write_quant_kernel<__nv_bfloat16, 128><<<g, b, 0, s>>>(p);
    else write_quant_kernel<__nv_bfloat16, 64><<<g, b, 0, s>>>(p);
  }
  return pa_internal::cuda_status(cudaGetLastError());
}
