// pa_internal.h -- host-side argument checks shared by the entry points.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "pa.h"

namespace pa_internal {

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

}  // namespace pa_internal
