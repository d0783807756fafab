// pa_internal.h -- host-side argument checks shared by the entry points.
#pragma once

#include <cuda.h>  // CUtensorMap and its enums (types only; no libcuda link)
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "pa.h"

namespace pa_internal {

// Records the CUDA error behind a PA_ERR_CUDA for pa_last_cuda_error (per
// calling thread) and returns the status to hand back.
void record_cuda_error(cudaError_t e);
inline pa_status cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return PA_OK;
  record_cuda_error(e);
  return PA_ERR_CUDA;
}

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Checks every field of the cache description; nothing is dereferenced on the
// device side here.
inline pa_status check_cache(const pa_cache* c) {
  if (!c) return PA_ERR_INVALID_ARG;
  if (c->block_size != 16) return PA_ERR_UNSUPPORTED;
  if (c->head_dim != 64 && c->head_dim != 128) return PA_ERR_UNSUPPORTED;
  if (c->dtype != PA_F16 && c->dtype != PA_BF16 && c->dtype != PA_I8) return PA_ERR_UNSUPPORTED;
  if (c->num_blocks < 1 || c->num_kv_heads < 1) return PA_ERR_INVALID_ARG;
  if (!c->k_cache || !c->v_cache) return PA_ERR_INVALID_ARG;
  if (!aligned16(c->k_cache) || !aligned16(c->v_cache)) return PA_ERR_INVALID_ARG;
  if (c->dtype == PA_I8) {
    if (!c->k_scale || !c->v_scale) return PA_ERR_INVALID_ARG;
    if (!aligned16(c->k_scale) || !aligned16(c->v_scale)) return PA_ERR_INVALID_ARG;
  }
  return PA_OK;
}

// The driver's tensor-map encoder, fetched once through the runtime so the
// library does not link libcuda directly.
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

inline EncodeTiledFn encode_tiled_fn() {
  static EncodeTiledFn fn = []() -> EncodeTiledFn {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    return reinterpret_cast<EncodeTiledFn>(p);
  }();
  return fn;
}

// 2-D TMA map over one cache tensor seen as [num_blocks*num_kv_heads*16 rows,
// head_dim]: boxes of 16 rows x min(128, row bytes), swizzled to match the
// kernels' shared-memory addressing (128-byte rows: 128B swizzle; 64-byte rows:
// 64B swizzle).
inline bool encode_cache_map(CUtensorMap* m, const pa_cache* c, void* base) {
  EncodeTiledFn fn = encode_tiled_fn();
  if (!fn) return false;
  const int elt = c->dtype == PA_I8 ? 1 : 2;
  const int row_bytes = c->head_dim * elt;
  const int chunk = row_bytes < 128 ? row_bytes : 128;
  const cuuint64_t dims[2] = {(cuuint64_t)c->head_dim,
                              (cuuint64_t)c->num_blocks * c->num_kv_heads * 16};
  const cuuint64_t strides[1] = {(cuuint64_t)row_bytes};
  const cuuint32_t box[2] = {(cuuint32_t)(chunk / elt), 16};
  const cuuint32_t estr[2] = {1, 1};
  const CUtensorMapDataType dt = c->dtype == PA_I8    ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                 : c->dtype == PA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                       : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  const CUtensorMapSwizzle sw = chunk == 128 ? CU_TENSOR_MAP_SWIZZLE_128B
                                             : CU_TENSOR_MAP_SWIZZLE_64B;
  return fn(m, dt, 2, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Launch `kern` on `stream` with the programmatic stream-serialization attribute
// (the kernel may start while the one before it finishes; it waits in-kernel
// before reading its inputs), plus a cluster shape when cluster_x > 1.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_dependent(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                                    cudaStream_t stream, unsigned cluster_x, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute at[2];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  unsigned n = 1;
  if (cluster_x > 1) {
    at[1].id = cudaLaunchAttributeClusterDimension;
    at[1].val.clusterDim.x = cluster_x;
    at[1].val.clusterDim.y = 1;
    at[1].val.clusterDim.z = 1;
    n = 2;
  }
  cfg.attrs = at;
  cfg.numAttrs = n;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
  return e != cudaSuccess ? e : cudaGetLastError();
}

// Rows of the 2-D view must fit the kernels' 32-bit row arithmetic.
inline bool cache_rows_fit(const pa_cache* c) {
  return (long long)c->num_blocks * c->num_kv_heads * 16 < 0x7fffffffLL;
}

}  // namespace pa_internal
