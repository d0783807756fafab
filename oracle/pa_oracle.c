/*
 * pa_oracle.c -- plain CPU oracle for attention over a paged KV cache.
 *
 * TEST INFRASTRUCTURE ONLY.  This is the slow, obviously-correct reference the
 * CUDA library is checked against.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg load it.  It shares no code, header, table or
 * helper with the CUDA library, and neither side includes or links the other.
 *
 * What it computes, from the pages:
 *   - "PyTorch LLM Serving Engine", section "Loading": every layer writes the new
 *     token's K/V to a physical cache slot, then runs a numerically stable online
 *     softmax while it walks the sequence's block table.
 *   - same page, "What is implemented": fixed-size physical blocks, per-sequence
 *     block tables; chunked prefill (a chunk of queries attends to the paged
 *     context before it and causally to itself).
 *   - "MicroGen: Modular, Hardware-Aware LLM Inference Engine", Key Features,
 *     "Paged & Quantized INT8 KV Cache": paged allocator with logical-to-physical
 *     block mapping, sliding-window length, GQA by repeat_kv head repetition,
 *     dynamic INT8 KV quantization with a vector scale.
 *   - "llminfer: A GPU-efficient LLM inference engine", section "Paged KV Cache
 *     And Continuous Batching": page size of 16 tokens.
 *
 * The pages give no formulas, layouts or rounding rules.  The readings used
 * here (each is the plainest one the pages support):
 *   - cache layout [num_blocks][num_kv_heads][block_size][head_dim], scales
 *     [num_blocks][num_kv_heads][block_size]; slot = physical_block*S + offset;
 *     slot < 0 means "no slot" (padding token).
 *   - INT8: per (token, kv head) and separately for K and V, amax = max|x| in
 *     fp32, scale = amax/127 (one fp32 division), code = round-half-even of
 *     x/scale (one fp32 division) clamped to [-127, 127]; amax = 0 gives scale 0
 *     and all-zero codes.  Dequantised value = code*scale.
 *   - GQA: query head h reads kv head h / (Hq/Hkv) (repeat_kv repeats each kv
 *     head Hq/Hkv times in a row).
 *   - a query at position i sees keys j with lo <= j <= i, lo = max(0, i-W+1)
 *     when the window W > 0, else 0.  The chunk of C queries of a sequence with
 *     context length L (counted after the write) sits at positions L-C .. L-1.
 *   - a query that sees no key returns zeros.
 *   - a key whose block-table entry is outside [0, num_blocks) is left out, and
 *     a context length above max_blocks_per_seq*S is cut to that value (this is
 *     how bad device data is handled on both sides).
 *   - attention arithmetic is fp64 throughout: scores, a two-pass softmax
 *     (max, exponentials, normalising sum) and the weighted sum of V rows.
 *
 * Inputs must be finite.  16-bit inputs are passed as raw bit patterns.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { PAO_F16 = 0, PAO_BF16 = 1, PAO_I8 = 2 };

/* IEEE 754 binary16 bit pattern -> value.  Normal: (1024 + m) * 2^(e - 25);
 * subnormal: m * 2^-24. */
double pao_f16_to_double(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int m = h & 0x3ff;
    double v;
    if (e == 0)
        v = ldexp((double)m, -24);
    else if (e == 31)
        v = m ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + m), e - 25);
    return sign ? -v : v;
}

/* bfloat16 bit pattern -> value: the top half of an IEEE binary32. */
double pao_bf16_to_double(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static double elem16(int dtype, uint16_t bits)
{
    return dtype == PAO_BF16 ? pao_bf16_to_double(bits) : pao_f16_to_double(bits);
}

/*
 * Dynamic INT8 quantisation of one row of D values ("MicroGen", Key Features,
 * "Dynamic INT8 KV Quantization: Vector scale"): one scale for the row, chosen
 * from the row's largest magnitude.  Every step is a single fp32 operation.
 */
void pao_quantize_row(const float *x, int D, int8_t *codes, float *scale_out)
{
    float amax = 0.0f;
    for (int d = 0; d < D; d++) {
        float a = fabsf(x[d]);
        if (a > amax)
            amax = a;
    }
    float scale = amax / 127.0f;
    *scale_out = scale;
    for (int d = 0; d < D; d++) {
        if (scale == 0.0f) {
            codes[d] = 0;
            continue;
        }
        float r = nearbyintf(x[d] / scale); /* default rounding: half to even */
        if (r > 127.0f)
            r = 127.0f;
        if (r < -127.0f)
            r = -127.0f;
        codes[d] = (int8_t)r;
    }
}

/*
 * KV write ("PyTorch LLM Serving Engine", "Loading": K/V go to a physical cache
 * slot).  For token t with slot s = slot_mapping[t] >= 0, row (t, h) of k and v
 * goes to cache[s / S][h][s % S][:].  16-bit caches take the input bits as they
 * are (cache dtype must equal the input dtype); int8 caches take codes and the
 * row's scale.  Slots not named are left untouched.  Returns the number of
 * tokens whose slot was out of range (those are skipped).
 */
int pao_write_kv(int cache_dtype, int in_dtype, int num_blocks, int block_size,
                 int num_kv_heads, int head_dim, void *k_cache, void *v_cache,
                 float *k_scale, float *v_scale, const uint16_t *k,
                 const uint16_t *v, const int32_t *slot_mapping, int num_tokens)
{
    const int S = block_size, H = num_kv_heads, D = head_dim;
    int bad = 0;
    float *row = (float *)malloc(sizeof(float) * (size_t)D);
    for (int t = 0; t < num_tokens; t++) {
        int32_t s = slot_mapping[t];
        if (s < 0)
            continue;
        if ((int64_t)s >= (int64_t)num_blocks * S) {
            bad++;
            continue;
        }
        int blk = s / S, off = s % S;
        for (int h = 0; h < H; h++) {
            size_t src = ((size_t)t * H + h) * D;
            size_t dst_row = ((size_t)blk * H + h) * S + off;
            for (int which = 0; which < 2; which++) {
                const uint16_t *x = which ? v : k;
                void *cache = which ? v_cache : k_cache;
                if (cache_dtype == PAO_I8) {
                    for (int d = 0; d < D; d++)
                        row[d] = (float)elem16(in_dtype, x[src + d]);
                    float *sc = which ? v_scale : k_scale;
                    pao_quantize_row(row, D, (int8_t *)cache + dst_row * D,
                                     &sc[dst_row]);
                } else {
                    memcpy((uint16_t *)cache + dst_row * D, x + src,
                           sizeof(uint16_t) * (size_t)D);
                }
            }
        }
    }
    free(row);
    return bad;
}

/* The cache as the attention functions see it. */
typedef struct {
    int dtype, num_blocks, S, H, D;
    const void *k_cache, *v_cache;
    const float *k_scale, *v_scale;
} pao_cache;

/* Row number (in units of D elements) of logical position j, kv head kvh, read
 * through the sequence's block table: block table[j / S], offset j % S.  -1 when
 * the table entry is not a valid physical block. */
static long row_index(const pao_cache *c, const int32_t *table, int j, int kvh)
{
    int32_t phys = table[j / c->S];
    if (phys < 0 || phys >= c->num_blocks)
        return -1;
    return ((long)phys * c->H + kvh) * c->S + j % c->S;
}

static void load_row(const pao_cache *c, int which, long r, double *out)
{
    const void *base = which ? c->v_cache : c->k_cache;
    if (c->dtype == PAO_I8) {
        const int8_t *codes = (const int8_t *)base + (size_t)r * c->D;
        double scale = (double)(which ? c->v_scale : c->k_scale)[r];
        for (int d = 0; d < c->D; d++)
            out[d] = (double)codes[d] * scale;
    } else {
        const uint16_t *bits = (const uint16_t *)base + (size_t)r * c->D;
        for (int d = 0; d < c->D; d++)
            out[d] = elem16(c->dtype, bits[d]);
    }
}

/* The keys query position i of a sequence of (clamped) length L may see:
 * [*lo, *hi].  Empty when *hi < *lo. */
static void key_range(int i, int L, int window, int *lo, int *hi)
{
    *hi = i < L - 1 ? i : L - 1;
    *lo = (window > 0 && i - window + 1 > 0) ? i - window + 1 : 0;
}

static int clamp_len(int L, int max_blocks_per_seq, int S)
{
    long cap = (long)max_blocks_per_seq * S;
    if (L < 0)
        return 0;
    return L > cap ? (int)cap : L;
}

/*
 * Attention over the paged cache, by its definition, in fp64.
 *
 * Sequence n owns queries cu_q_lens[n] .. cu_q_lens[n+1]-1 (rows of q, layout
 * [num_q_tokens][num_q_heads][D]); query c of the C_n queries sits at position
 * L_n - C_n + c where L_n = context_lens[n].  Decode is C_n = 1.  For query
 * head h, kv head h / (Hq / Hkv) is read (repeat_kv).
 *
 *   s_j = sm_scale * sum_d q_d k_{j,d}
 *   m = max_j s_j;  e_j = exp(s_j - m);  out = sum_j (e_j / sum e) v_j
 *
 * out is [num_q_tokens][num_q_heads][D] fp64.
 */
int pao_attention(int cache_dtype, int num_blocks, int block_size, int num_kv_heads,
                  int head_dim, const void *k_cache, const void *v_cache,
                  const float *k_scale, const float *v_scale, int q_dtype,
                  const uint16_t *q, int num_seqs, int num_q_heads,
                  const int32_t *cu_q_lens, const int32_t *block_tables,
                  int max_blocks_per_seq, const int32_t *context_lens, double sm_scale,
                  int window, double *out)
{
    pao_cache c = {cache_dtype, num_blocks, block_size, num_kv_heads, head_dim,
                   k_cache, v_cache, k_scale, v_scale};
    const int D = head_dim, Hq = num_q_heads, G = num_q_heads / num_kv_heads;
    int max_keys = max_blocks_per_seq * block_size;
    double *s = (double *)malloc(sizeof(double) * (size_t)(max_keys > 0 ? max_keys : 1));
    int *valid = (int *)malloc(sizeof(int) * (size_t)(max_keys > 0 ? max_keys : 1));
    double *qd = (double *)malloc(sizeof(double) * (size_t)D);
    double *row = (double *)malloc(sizeof(double) * (size_t)D);

    for (int n = 0; n < num_seqs; n++) {
        const int32_t *table = block_tables + (size_t)n * max_blocks_per_seq;
        int L = clamp_len(context_lens[n], max_blocks_per_seq, block_size);
        int C = cu_q_lens[n + 1] - cu_q_lens[n];
        for (int ci = 0; ci < C; ci++) {
            int tok = cu_q_lens[n] + ci;
            int i = L - C + ci; /* position of this query */
            int lo, hi;
            key_range(i, L, window, &lo, &hi);
            for (int h = 0; h < Hq; h++) {
                int kvh = h / G;
                double *o = out + ((size_t)tok * Hq + h) * D;
                for (int d = 0; d < D; d++) {
                    o[d] = 0.0;
                    qd[d] = elem16(q_dtype, q[((size_t)tok * Hq + h) * D + d]);
                }
                /* pass 1: scores and their maximum */
                double m = -INFINITY;
                int any = 0;
                for (int j = lo; j <= hi; j++) {
                    long r = row_index(&c, table, j, kvh);
                    valid[j] = r >= 0;
                    if (!valid[j])
                        continue;
                    load_row(&c, 0, r, row);
                    double dot = 0.0;
                    for (int d = 0; d < D; d++)
                        dot += qd[d] * row[d];
                    s[j] = sm_scale * dot;
                    if (s[j] > m)
                        m = s[j];
                    any = 1;
                }
                if (!any)
                    continue; /* no visible key: zeros */
                /* pass 2: normaliser, then the probability-weighted V rows */
                double l = 0.0;
                for (int j = lo; j <= hi; j++)
                    if (valid[j])
                        l += exp(s[j] - m);
                for (int j = lo; j <= hi; j++) {
                    if (!valid[j])
                        continue;
                    double p = exp(s[j] - m) / l;
                    load_row(&c, 1, row_index(&c, table, j, kvh), row);
                    for (int d = 0; d < D; d++)
                        o[d] += p * row[d];
                }
            }
        }
    }
    free(s);
    free(valid);
    free(qd);
    free(row);
    return 0;
}

/*
 * The same attention reached the way the pages' engines reach it: the keys are
 * walked in segments with a running maximum, normaliser and accumulator (the
 * online softmax of "PyTorch LLM Serving Engine", "Loading"), and the key range
 * is cut into partitions of part_tokens keys whose partial states are merged at
 * the end (split-K).  Segment lengths cycle through seg_lens[0..num_seg-1].
 *
 * Per segment with scores s_j:  m' = max(m, max_j s_j),  c = exp(m - m'),
 *   l = l*c + sum_j exp(s_j - m'),  o = o*c + sum_j exp(s_j - m') v_j.
 * Merge of partitions p:  M = max_p m_p,
 *   out = sum_p exp(m_p - M) o_p / sum_p exp(m_p - M) l_p.
 */
int pao_attention_online(int cache_dtype, int num_blocks, int block_size,
                         int num_kv_heads, int head_dim, const void *k_cache,
                         const void *v_cache, const float *k_scale, const float *v_scale,
                         int q_dtype, const uint16_t *q, int num_seqs, int num_q_heads,
                         const int32_t *cu_q_lens, const int32_t *block_tables,
                         int max_blocks_per_seq, const int32_t *context_lens,
                         double sm_scale, int window, int part_tokens,
                         const int32_t *seg_lens, int num_seg, double *out)
{
    pao_cache c = {cache_dtype, num_blocks, block_size, num_kv_heads, head_dim,
                   k_cache, v_cache, k_scale, v_scale};
    const int D = head_dim, Hq = num_q_heads, G = num_q_heads / num_kv_heads;
    int max_keys = max_blocks_per_seq * block_size;
    int max_parts = max_keys / (part_tokens > 0 ? part_tokens : 1) + 2;
    double *qd = (double *)malloc(sizeof(double) * (size_t)D);
    double *row = (double *)malloc(sizeof(double) * (size_t)D);
    double *pm = (double *)malloc(sizeof(double) * (size_t)max_parts);
    double *pl = (double *)malloc(sizeof(double) * (size_t)max_parts);
    double *po = (double *)malloc(sizeof(double) * (size_t)max_parts * D);
    double *seg_s = (double *)malloc(sizeof(double) * (size_t)(max_keys > 0 ? max_keys : 1));

    for (int n = 0; n < num_seqs; n++) {
        const int32_t *table = block_tables + (size_t)n * max_blocks_per_seq;
        int L = clamp_len(context_lens[n], max_blocks_per_seq, block_size);
        int C = cu_q_lens[n + 1] - cu_q_lens[n];
        for (int ci = 0; ci < C; ci++) {
            int tok = cu_q_lens[n] + ci;
            int i = L - C + ci;
            int lo, hi;
            key_range(i, L, window, &lo, &hi);
            for (int h = 0; h < Hq; h++) {
                int kvh = h / G;
                double *o = out + ((size_t)tok * Hq + h) * D;
                for (int d = 0; d < D; d++)
                    qd[d] = elem16(q_dtype, q[((size_t)tok * Hq + h) * D + d]);
                int np = 0;
                for (int p0 = lo; p0 <= hi; p0 += part_tokens, np++) {
                    int p1 = p0 + part_tokens - 1 < hi ? p0 + part_tokens - 1 : hi;
                    double m = -INFINITY, l = 0.0;
                    double *op = po + (size_t)np * D;
                    for (int d = 0; d < D; d++)
                        op[d] = 0.0;
                    int k = 0;
                    for (int j0 = p0; j0 <= p1; k++) {
                        int len = seg_lens[k % num_seg];
                        int j1 = j0 + len - 1 < p1 ? j0 + len - 1 : p1;
                        double mseg = -INFINITY;
                        for (int j = j0; j <= j1; j++) {
                            long r = row_index(&c, table, j, kvh);
                            if (r < 0) {
                                seg_s[j - j0] = -INFINITY;
                                continue;
                            }
                            load_row(&c, 0, r, row);
                            double dot = 0.0;
                            for (int d = 0; d < D; d++)
                                dot += qd[d] * row[d];
                            seg_s[j - j0] = sm_scale * dot;
                            if (seg_s[j - j0] > mseg)
                                mseg = seg_s[j - j0];
                        }
                        if (mseg > -INFINITY) {
                            double mn = m > mseg ? m : mseg;
                            double corr = m == -INFINITY ? 0.0 : exp(m - mn);
                            l *= corr;
                            for (int d = 0; d < D; d++)
                                op[d] *= corr;
                            for (int j = j0; j <= j1; j++) {
                                if (seg_s[j - j0] == -INFINITY)
                                    continue;
                                double e = exp(seg_s[j - j0] - mn);
                                l += e;
                                load_row(&c, 1, row_index(&c, table, j, kvh), row);
                                for (int d = 0; d < D; d++)
                                    op[d] += e * row[d];
                            }
                            m = mn;
                        }
                        j0 = j1 + 1;
                    }
                    pm[np] = m;
                    pl[np] = l;
                }
                /* split-K merge */
                double M = -INFINITY;
                for (int p = 0; p < np; p++)
                    if (pm[p] > M)
                        M = pm[p];
                for (int d = 0; d < D; d++)
                    o[d] = 0.0;
                if (M == -INFINITY)
                    continue;
                double den = 0.0;
                for (int p = 0; p < np; p++) {
                    if (pm[p] == -INFINITY)
                        continue;
                    double w = exp(pm[p] - M);
                    den += w * pl[p];
                    for (int d = 0; d < D; d++)
                        o[d] += w * po[(size_t)p * D + d];
                }
                for (int d = 0; d < D; d++)
                    o[d] /= den;
            }
        }
    }
    free(qd);
    free(row);
    free(pm);
    free(pl);
    free(po);
    free(seg_s);
    return 0;
}

/*
 * Weight-only INT8 linear layer ("PyTorch LLM Serving Engine", What is
 * implemented: symmetric per-output-channel INT8 weights; "MicroGen", Key
 * Features: static per-channel INT8 weight quantization).
 *
 * pao_quantize_weights: row n of w [n][k] (16-bit bit patterns, converted to
 * fp32 exactly) is one output channel, quantised by pao_quantize_row (the rule
 * of the INT8 KV rows: scale = amax/127, codes rounded half to even).
 *
 * pao_linear_int8: y[m][n] = sum_k x[m][k] * (code[n][k] * scale[n]) + bias[n],
 * every term and the sum in fp64 (bias optional: has_bias = 0 leaves it out).
 */
void pao_quantize_weights(int w_dtype, const uint16_t *w, int n, int k, int8_t *codes,
                          float *scales)
{
    float *row = (float *)malloc(sizeof(float) * (size_t)k);
    if (!row)
        return;
    for (int i = 0; i < n; i++) {
        for (int j = 0; j < k; j++) {
            uint16_t b = w[(size_t)i * k + j];
            row[j] = (float)(w_dtype == PAO_BF16 ? pao_bf16_to_double(b) : pao_f16_to_double(b));
        }
        pao_quantize_row(row, k, codes + (size_t)i * k, scales + i);
    }
    free(row);
}

void pao_linear_int8(const int8_t *codes, const float *scales, int x_dtype, const uint16_t *x,
                     int has_bias, const uint16_t *bias, int m, int n, int k, double *y)
{
    for (int r = 0; r < m; r++) {
        for (int i = 0; i < n; i++) {
            double s = 0.0;
            for (int j = 0; j < k; j++) {
                uint16_t xb = x[(size_t)r * k + j];
                double xv = x_dtype == PAO_BF16 ? pao_bf16_to_double(xb) : pao_f16_to_double(xb);
                s += xv * ((double)codes[(size_t)i * k + j] * (double)scales[i]);
            }
            if (has_bias)
                s += x_dtype == PAO_BF16 ? pao_bf16_to_double(bias[i]) : pao_f16_to_double(bias[i]);
            y[(size_t)r * n + i] = s;
        }
    }
}
