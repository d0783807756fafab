/*
 * pa_linear.h -- weight-only INT8 linear layer for decode-sized batches.
 *
 * "PyTorch LLM Serving Engine", "What is implemented": weight-only
 * quantization, symmetric per-output-channel INT8, with a fused backend that
 * reads the quantized weight tiles directly (rather than dequantizing the
 * weights before a floating-point GEMM); "MicroGen", "Key Features": static
 * per-channel INT8 weight quantization.
 *
 *   quantize: per output channel n, amax = max_k |w[n][k]| (fp32), scale[n] =
 *             amax / 127 (one IEEE fp32 division), code[n][k] = w[n][k] / scale
 *             (one IEEE fp32 division) rounded half to even, clamped to
 *             [-127, 127]; amax = 0 gives scale 0 and zero codes (the rule of
 *             the INT8 KV cache in pa.h).
 *   linear:   y[m][n] = scale[n] * sum_k x[m][k] * code[n][k]  (+ bias[n]),
 *             accumulated in fp32, rounded once to the activations' type.
 *
 * Layouts (row-major, contiguous): w, codes [n][k]; scales [n] fp32; x [m][k];
 * y [m][n]; bias [n] (optional).  x, y and bias share one type (PA_F16 or
 * PA_BF16).  Every buffer is the caller's device memory; calls are asynchronous
 * on the caller's stream (NULL: the default stream).
 *
 * Errors (host checks, nothing launched): PA_ERR_INVALID_ARG for NULL or
 * misaligned pointers (codes, w and x 16-byte aligned; y, bias and scales
 * aligned to their element) or non-positive sizes; PA_ERR_UNSUPPORTED when
 * n % 16 != 0 or k % 64 != 0, or k > 65536.  A failed launch returns PA_ERR_CUDA.
 * The MMA takes the activations as fp16: bf16 activations beyond the fp16 range
 * (|x| > 65504) overflow.
 */
#ifndef PA_LINEAR_H
#define PA_LINEAR_H

#include <stddef.h>
#include <stdint.h>

#include "pa.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Quantize w [n][k] (fp16 or bf16) into codes [n][k] and scales [n]. */
pa_status pa_linear_int8_quantize(const void *w, pa_dtype w_dtype, int n, int k, int8_t *codes,
                                  float *scales, void *stream);

/*
 * Workspace for pa_linear_int8 (bytes).  When the output channels are too few
 * to fill the GPU, the call splits the k range across thread blocks; up to 8
 * splits add their partial sums inside the launch (a thread-block cluster, no
 * workspace), more -- only for very few channels over a long k -- go through
 * this workspace and a second kernel.  A smaller workspace (even none) is
 * accepted; the call then splits less.
 */
size_t pa_linear_int8_workspace_bytes(int m, int n, int k);

/* y = x * dequant(codes, scales)^T (+ bias); m tokens, any m >= 1. */
pa_status pa_linear_int8(const int8_t *codes, const float *scales, const void *bias, const void *x,
                         pa_dtype x_dtype, int m, int n, int k, void *y, void *workspace,
                         size_t workspace_bytes, void *stream);

/*
 * pa_linear_int8_grouped -- count (1..4) weight-only INT8 linears that read the
 * same activations x [m][k], in one launch: y[i] = x * dequant(codes[i],
 * scales[i])^T (+ bias[i]), y[i] [m][n[i]].  A decoder layer's q, k and v
 * projections, or its gate and up projections, share x ("PyTorch LLM Serving
 * Engine", "What is implemented": the fused INT8 backend serves every
 * projection).  codes, scales, bias (NULL, or an array whose entries may be
 * NULL), n and y are HOST arrays of count entries; the pointers in them are
 * device pointers with the alignment and type rules of pa_linear_int8, every
 * n[i] a multiple of 16.  Each matrix's result is pa_linear_int8's on it alone
 * up to the order of the fp32 additions: the k range may be split differently
 * (at most 8 splits, merged in the launch; no workspace).
 */
pa_status pa_linear_int8_grouped(int count, const int8_t *const *codes,
                                 const float *const *scales, const void *const *bias,
                                 const int *n, const void *x, pa_dtype x_dtype, int m, int k,
                                 void *const *y, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* PA_LINEAR_H */
