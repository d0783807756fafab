// pa_device.cuh -- device building blocks for the sm_103a paged-KV kernels:
// mbarrier waits with a time limit, bulk global->shared copies, warp-level
// tensor-core MMA (m16n8k16) and exact int8 -> f16 conversion.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "pa.h"

namespace pa_dev {

constexpr int kBlock = 16;  // tokens per physical block (the pages' 16-token page)

// A bounded wait gives up after this many SM clock cycles (about 2 s at 2 GHz)
// and reports PA_FLAG_TIMEOUT instead of hanging.
constexpr long long kWaitLimitCycles = 4000000000LL;

enum Mode { kF16 = 0, kBF16 = 1, kI8 = 2 };

template <int MODE>
struct ModeTraits {
  static constexpr int kElt = MODE == kI8 ? 1 : 2;
};

// One pipeline stage holds one (block, kv head) tile of K and one of V, each 16
// rows of D elements.  A tile arrives by TMA as kChunks boxes of 16 rows x
// kChunkBytes (128 bytes, or 64 for int8 with D = 64), each box written with the
// hardware swizzle that XORs the 16-byte chunk index of a row with bits of the
// row index (128-byte rows: row & 7; 64-byte rows: (row >> 1) & 3).  Reading
// eight rows at the same logical column then touches eight different bank
// groups, so ldmatrix is conflict-free.
template <int MODE, int D>
struct Tile {
  static constexpr int kElt = ModeTraits<MODE>::kElt;
  static constexpr int kRowBytes = D * kElt;
  static constexpr int kChunkBytes = kRowBytes < 128 ? kRowBytes : 128;
  static constexpr int kChunkElems = kChunkBytes / kElt;
  static constexpr int kChunks = kRowBytes / kChunkBytes;
  static constexpr int kBoxBytes = kBlock * kChunkBytes;
  static constexpr int kTileBytes = kBlock * kRowBytes;
  static constexpr int kStageBytes = 2 * kTileBytes;  // K tile, then V tile
  static constexpr int kScaleBytes = MODE == kI8 ? 2 * kBlock * 4 : 0;  // K, V scales
  static constexpr uint32_t kTxBytes = 2 * kTileBytes;  // TMA bytes per stage
  // Arrivals that complete a stage: the producer's expect-tx arrival, plus one
  // per lane that copies int8 scales with cp.async (4 lanes x 16 bytes each).
  static constexpr int kScaleLanes = MODE == kI8 ? 8 : 0;
  static constexpr int kFullArrivals = 1 + kScaleLanes;
  static constexpr int kAlign = kChunkBytes == 128 ? 1024 : 512;  // swizzle atom

  // Byte offset inside a tile of byte `b` of row `r` (b a multiple of 16 for
  // ldmatrix addresses; the low 4 bits pass through).
  static __device__ __forceinline__ uint32_t off(int r, int b) {
    const int h = b / kChunkBytes, w = b % kChunkBytes;
    const int key = kChunkBytes == 128 ? (r & 7) : ((r >> 1) & 3);
    return h * kBoxBytes + r * kChunkBytes + ((((w >> 4) ^ key) << 4) | (w & 15));
  }
};

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ------------------------------------------------------------------ mbarrier

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return done != 0;
}

// Wait for the phase with the given parity to complete; false if the time
// limit (SM clock cycles) ran out first.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity,
                                          long long limit = kWaitLimitCycles) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (clock64() - t0 > limit) return false;
  }
  return true;
}

// TMA tiled copy of the box at element coordinates (x, y) of a 2-D tensor map
// into shared memory (dst aligned to the map's swizzle atom).  x * element size
// is a multiple of 16 at every call site.
__device__ __forceinline__ void tma_load_2d(void* dst, const void* tmap, int x, int y,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, "
      "{%2, %3}], [%4];" ::"r"(smem_u32(dst)),
      "l"(tmap), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

// As tma_load_2d for a 3-D tensor map (coordinates x, y, z; x * element size a
// multiple of 16).
__device__ __forceinline__ void tma_load_3d(void* dst, const void* tmap, int x, int y, int z,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, "
      "{%2, %3, %4}], [%5];" ::"r"(smem_u32(dst)),
      "l"(tmap), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
      : "memory");
}

// 16-byte asynchronous copy global -> shared through the load/store unit (not
// the TMA unit), and an arrival on `bar` once this thread's earlier cp.async
// copies have landed; the arrival is one of the barrier's expected arrivals.
__device__ __forceinline__ void cp_async_16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src)
               : "memory");
}

// As cp_async_16, but writes 16 zero bytes (reading nothing) when !valid.
__device__ __forceinline__ void cp_async_16_or_zero(void* dst, const void* src, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(dst)), "l"(src),
               "r"(valid ? 16 : 0)
               : "memory");
}

// Wait for every cp.async this thread issued.
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.wait_all;" ::: "memory");
}

__device__ __forceinline__ void cp_async_arrive_noinc(uint64_t* bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

// Named barrier over the first `threads` threads of the CTA (id 1; id 0 is
// __syncthreads).
__device__ __forceinline__ void named_sync(int id, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// ------------------------------------------------------------------ tensor cores

__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

// Transpose of an 8x8 b16 matrix held one row pair per thread (the layout
// ldmatrix and the MMA C fragment use): thread (g, t) gives row g, columns 2t,
// 2t+1 and receives row g, columns 2t, 2t+1 of the transpose.
__device__ __forceinline__ uint32_t movmatrix_t(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}

// D = A(16x16, row) * B(16x8, col) + D, fp32 accumulate.  BF16 selects bf16
// operands, otherwise f16 (both operands always have the same type).
template <bool BF16>
__device__ __forceinline__ void mma16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
  if constexpr (BF16) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  } else {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  }
}

__device__ __forceinline__ uint32_t pack_f16(float lo, float hi) {
  __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

template <bool BF16>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  if constexpr (BF16) return pack_bf16(lo, hi);
  else return pack_f16(lo, hi);
}

// ------------------------------------------------------------------ int8 -> f16

// The f16 with bit pattern 0x64XX is 1024 + XX exactly, so a code c in
// [-128, 127] turned into the byte c + 128 (flip the top bit: the form an int8
// KV cache stores, while the weight codes of the linear layer are flipped as
// they are loaded) and placed under 0x64 is 1024 + 128 + c; subtracting 1152
// leaves c exactly.  This is the
// published "magic number" integer-to-float conversion used by mixed-input
// GEMMs (Kim et al., "Who Says Elephants Can't Run: Bringing Large Scale MoE
// Models into Cloud Scale Production", 2022, Sec. 4), restated here.
__device__ __forceinline__ uint32_t f16x2_minus_1152(uint32_t biased) {
  const __half2 bias = __halves2half2(__ushort_as_half(0x6480), __ushort_as_half(0x6480));
  __half2 h = __hsub2(*reinterpret_cast<__half2*>(&biased), bias);
  return *reinterpret_cast<uint32_t*>(&h);
}

// Four codes (bytes 0..3 of w, each code + 128) -> f16x2 pairs
// (c0, c1) and (c2, c3).
__device__ __forceinline__ void biased_i8x4_to_f16(uint32_t u, uint32_t& lo, uint32_t& hi) {
  lo = f16x2_minus_1152(__byte_perm(u, 0x64646464u, 0x4140));
  hi = f16x2_minus_1152(__byte_perm(u, 0x64646464u, 0x4342));
}

// Bytes k and k+1 of two words (already biased) -> f16x2 pairs
// (a.k, b.k) and (a.k+1, b.k+1); k is 0 or 2.
template <int K>
__device__ __forceinline__ void biased_i8_pairs(uint32_t a, uint32_t b, uint32_t& p0,
                                                uint32_t& p1) {
  constexpr uint32_t sel = K == 0 ? 0x5140u : 0x7362u;
  const uint32_t x = __byte_perm(a, b, sel);  // [a.k, b.k, a.k+1, b.k+1]
  p0 = f16x2_minus_1152(__byte_perm(x, 0x64646464u, 0x4140));
  p1 = f16x2_minus_1152(__byte_perm(x, 0x64646464u, 0x4342));
}

// The same conversions without the final subtraction: each f16 holds the code
// plus 1152 exactly.  A dot product with such values is the true one plus 1152
// times the sum of the other operand, which the caller subtracts once.
__device__ __forceinline__ void biased_i8x4_to_f16_plus1152(uint32_t u, uint32_t& lo,
                                                            uint32_t& hi) {
  lo = __byte_perm(u, 0x64646464u, 0x4140);
  hi = __byte_perm(u, 0x64646464u, 0x4342);
}

// 2^x with the hardware approximation (relative error below 2^-22; -inf -> 0).
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// log2(x) with the hardware approximation (absolute error near 2^-22; 0 -> -inf;
// subnormal inputs are not flushed).
__device__ __forceinline__ float fast_log2(float x) {
  float y;
  asm("lg2.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// ------------------------------------------------------------------ int8 value weights
//
// An int8 cache row's values are code * v_scale, with v_scale = amax / 127 of
// that row ("MicroGen", Key Features: dynamic INT8 KV quantisation with a vector
// scale), so rows of very different magnitudes share one sequence.  The P V
// product takes the softmax weight and the row's scale together as one 16-bit
// MMA operand, w_j = 2^(s_j - m) * v_scale_j.  Folding v_scale into a weight
// that is at most 1 underflows f16 (below 2^-14 it loses bits, below 2^-24 it is
// 0) once the rows are small, so the weights are taken relative to their own
// running reference instead: with y_j = s_j + log2(v_scale_j) and a per-row
// reference n (the largest y_j seen when it was last moved), the operand is
// 2^(y_j - n), at most 2^kLazyV, and the largest term of the sum is at least 1.
// The accumulated O therefore carries the factor 2^-n; it is rescaled only when
// some y_j exceeds n by more than kLazyV, and converted to the softmax's
// reference m once, in fp32, at the end (O * 2^(n - m)).  The error of every
// term is then relative to the largest term, whatever the rows' magnitudes.
constexpr float kLazyV = 8.0f;
constexpr float kNoRef = -3.402823466e38f;  // n before any weight: y - n stays -inf for y = -inf

// bf16 query values reach 3.4e38, f16 operands only 65504.  A query row whose
// largest |q| is 2^E (E >= 15) is multiplied by 2^-(E - 14) before it is
// narrowed to f16 (a power of two: every bit of the bf16 values that matters to
// the fp32 dot product survives) and the score by 2^(E - 14) after the MMA.
// Returns that exponent shift (0 when the row already fits).
__device__ __forceinline__ int q_prescale_shift(float amax) {
  const int e = (int)((__float_as_uint(amax) >> 23) & 0xFF) - 127;
  return e > 14 ? e - 14 : 0;
}
__device__ __forceinline__ float pow2i(int k) {  // 2^k for -126 <= k <= 127
  return __uint_as_float((uint32_t)(k + 127) << 23);
}

// ------------------------------------------------------------------ KV row write
//
// A new token's K or V row, one warp per row, E = D/32 consecutive elements per
// lane: 16-bit inputs convert to fp32 exactly; the int8 quantiser finds amax by
// a butterfly of shuffles (fmaxf/fabsf are exact) and rounds with the IEEE
// operations __fdiv_rn and __float2int_rn, bit for bit the CPU oracle's rule.
// The KV write kernel and the decode kernel that writes its step's token both
// use these.
template <typename IT>
__device__ __forceinline__ float in_to_f32(IT x);
template <>
__device__ __forceinline__ float in_to_f32<__half>(__half x) {
  return __half2float(x);
}
template <>
__device__ __forceinline__ float in_to_f32<__nv_bfloat16>(__nv_bfloat16 x) {
  return __bfloat162float(x);
}

// Quantise one row held as E = D/32 consecutive elements per lane.
template <int E>
__device__ __forceinline__ void quantize_row(const float (&x)[E], uint8_t (&q)[E], float& scale) {
  float amax = 0.0f;
#pragma unroll
  for (int e = 0; e < E; e++) amax = fmaxf(amax, fabsf(x[e]));
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
  scale = __fdiv_rn(amax, 127.0f);
#pragma unroll
  for (int e = 0; e < E; e++) {
    int c = 0;
    if (scale != 0.0f) {
      c = __float2int_rn(__fdiv_rn(x[e], scale));
      c = c > 127 ? 127 : (c < -127 ? -127 : c);
    }
    q[e] = (uint8_t)(c + 128);  // stored offset binary
  }
}


// ------------------------------------------------------------------ dependent launch
//
// Programmatic dependent launch: a kernel launched with the programmatic
// stream-serialization attribute may start while the kernel before it in the
// stream is still running, once every CTA of that kernel has signalled
// (pdl_launch_dependents) or exited; it must pdl_wait() -- which returns when
// the kernel before it has completed and its writes are visible -- before it
// reads anything that kernel may have written.  Launched without the
// attribute, pdl_wait returns at once.  The library's kernels signal at their
// start and wait before their first read of an input, so only launch latency
// and set-up overlap, never data.
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// ------------------------------------------------------------------ misc

__device__ __forceinline__ void set_flag(int32_t* err, int bits) {
  if (err) atomicOr(err, bits);
}

template <typename T>
__device__ __forceinline__ T to_out(float x);
template <>
__device__ __forceinline__ __half to_out<__half>(float x) {
  return __float2half_rn(x);
}
template <>
__device__ __forceinline__ __nv_bfloat16 to_out<__nv_bfloat16>(float x) {
  return __float2bfloat16_rn(x);
}

}  // namespace pa_dev
