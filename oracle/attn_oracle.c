/*
 * FP64 reference ("oracle") for the fused attention forward.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing on the product path may link, load or call
 * this file; only the tests, the smoke check and the CPU-baseline leg of the
 * benchmark do. It shares no code, header or constant with the CUDA library.
 *
 * What it computes is the plain definition of scaled dot-product attention,
 * written out with no blocking, fusion or reordering:
 *
 *   s_ij = scale * sum_d q[b,i,h,d] * k[b,j,g,d]  (+ mask[b,i,j] if additive)
 *   s_ij = -inf                                    if causal and j > i + (Sk - Sq)
 *   m_i  = max_j s_ij                              (pass 1)
 *   p_ij = exp(s_ij - m_i),  l_i = sum_j p_ij      (pass 2)
 *   o[b,i,h,:] = sum_j (p_ij / l_i) * v[b,j,g,:]
 *   lse[b,h,i] = m_i + ln(l_i)
 *   a row with no finite s_ij gives o = 0, lse = -inf
 *
 * with g = floor(h / (Hq / Hkv)) (query heads grouped onto shared K/V heads).
 *
 * Sources:
 *  - "ATB engineering guide" (hwcomputing.csdn.net/6a59a88310ee7a33f28e5ce9),
 *    §5.1: the eager formula matmul(Q, K^T) * scale -> softmax -> matmul(., V);
 *    §4.1 pattern 2 (attention fusion); §2.1 and §8.2 (MQA/GQA via kv_head_num,
 *    causal flag, optional mask input).
 *  - "CANN-ATB图优化-昇腾NPU怎么把PyTorch计算图改造成融合算子", Pattern 2:
 *    Q·K^T -> Scale -> Mask -> Softmax -> ·V.
 *  - "ops-transformer：Transformer算子融合与推理加速实战", §2.2 and §3.2
 *    (the blockwise/online softmax reaches this same normalised result),
 *    §2.4 (FP32 statistics on chip; this oracle uses FP64 throughout),
 *    §4.2 (scale defaults to 1/sqrt(D); Q/K/V in (B,S,H,D)).
 *
 * Readings where the pages are silent: causal alignment is bottom-right
 * (key j visible to query i iff j <= i + Sk - Sq); the additive mask is FP32
 * (B,Sq,Sk) broadcast over heads; a non-finite or non-positive scale means
 * 1/sqrt(D); a fully masked row gives o = 0 and lse = -inf.
 *
 * Inputs are the raw 16-bit patterns of bf16 (dtype 0) or IEEE fp16 (dtype 1)
 * values; each is widened to double exactly.
 *
 * Optional rotary position embedding (oracle_attn_fwd_rope), applied to q and
 * k before the scores ("ATB engineering guide" §4.1 pattern 5, RoPE fused with
 * attention; §8.4, interleaved pairs with rotary base 10000): the pair
 * (x[2i], x[2i+1]) of a head vector at position pos turns by the angle
 * pos * base^(-2i/D):
 *   (x[2i], x[2i+1]) -> (x[2i] cos - x[2i+1] sin, x[2i+1] cos + x[2i] sin).
 * Query row i sits at position q_pos0 + i, key j at k_pos0 + j. (The page's
 * listing doubles the exponent and spans the whole hidden size; the per-head
 * form above is the reading taken.) With rope_round set, each rotated element
 * is then rounded to the nearest value of the input's 16-bit type (ties to
 * even), as §8.4's reference rotation hands back its result in the input's
 * half-precision type; without it the rotated vectors stay exact.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { ORACLE_DTYPE_BF16 = 0, ORACLE_DTYPE_F16 = 1 };
enum { ORACLE_MASK_NONE = 0, ORACLE_MASK_CAUSAL = 1, ORACLE_MASK_ADDITIVE = 2,
       ORACLE_MASK_CAUSAL_ADDITIVE = 3 };

/* bf16 is the upper half of an IEEE binary32: shift it back into place. */
static double widen_bf16(uint16_t bits) {
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* IEEE binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
static double widen_f16(uint16_t bits) {
    int sign = (bits >> 15) & 1;
    int expo = (bits >> 10) & 0x1f;
    int frac = bits & 0x3ff;
    double mag;
    if (expo == 0)
        mag = ldexp((double)frac, -24);                 /* zero / subnormal */
    else if (expo == 31)
        mag = frac ? NAN : INFINITY;
    else
        mag = ldexp((double)(1024 + frac), expo - 25);  /* (1 + f/1024) 2^(e-15) */
    return sign ? -mag : mag;
}

static double widen(uint16_t bits, int dtype) {
    return dtype == ORACLE_DTYPE_F16 ? widen_f16(bits) : widen_bf16(bits);
}

/* Nearest value of the 16-bit type (ties to even), as a double: bf16 keeps 8
 * significant bits and the binary32 exponent range (smallest normal 2^-126),
 * fp16 keeps 11 (smallest normal 2^-14); both underflow gradually and go to
 * infinity past their largest finite value. */
static double narrow(double x, int dtype) {
    if (x == 0.0 || !isfinite(x)) return x;
    const int bits = dtype == ORACLE_DTYPE_F16 ? 11 : 8;
    const int emin = dtype == ORACLE_DTYPE_F16 ? -14 : -126;
    const double maxf = dtype == ORACLE_DTYPE_F16 ? 65504.0 : ldexp(255.0, 120);
    int e;
    frexp(x, &e);                          /* |x| in [2^(e-1), 2^e) */
    int lead = e - 1;
    if (lead < emin) lead = emin;
    const double ulp = ldexp(1.0, lead - (bits - 1));
    const double r = nearbyint(x / ulp) * ulp;     /* x / ulp is exact; default rounding is to even */
    return fabs(r) > maxf ? copysign(INFINITY, x) : r;
}

/* Rotary position embedding of one head vector, in place. */
static void rope_rotate(double *x, int D, long long pos, double base, int round_to, int dtype) {
    for (int i = 0; i < D / 2; ++i) {
        const double theta = (double)pos * pow(base, -2.0 * i / D);
        const double c = cos(theta), s = sin(theta);
        const double x0 = x[2 * i], x1 = x[2 * i + 1];
        x[2 * i] = x0 * c - x1 * s;
        x[2 * i + 1] = x1 * c + x0 * s;
        if (round_to) {
            x[2 * i] = narrow(x[2 * i], dtype);
            x[2 * i + 1] = narrow(x[2 * i + 1], dtype);
        }
    }
}

int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/*
 * Attention for a list of (b, h) slices and the query rows [row_begin, row_end).
 *
 *   q    : (B, Sq, Hq, D)   16-bit patterns, row-major
 *   k, v : (B, Sk, Hkv, D)  16-bit patterns, row-major
 *   mask : (B, Sq, Sk) FP32, read only when mask_kind is additive
 *   o    : (n_slices, row_end - row_begin, D)   output, FP64
 *   lse  : (n_slices, row_end - row_begin)      output, FP64 (natural log)
 *   psum : optional (may be NULL), (n_slices, rows): sum_j of the normalised
 *          probabilities p_ij / l_i (1 for a row with a visible key, 0 otherwise)
 *
 * Returns 0 on success, -1 on an invalid argument.
 */
/* As oracle_attn_fwd, with q and k rotated (rope_base > 0) or not (rope_base = 0). */
int oracle_attn_fwd_rope(const uint16_t *q, const uint16_t *k, const uint16_t *v, int dtype,
                         const float *mask, int mask_kind,
                         int B, int Hq, int Hkv, int Sq, int Sk, int D, double scale,
                         int n_slices, const int32_t *slice_b, const int32_t *slice_h,
                         int row_begin, int row_end,
                         double *o, double *lse, double *psum, int n_threads,
                         double rope_base, long long q_pos0, long long k_pos0, int rope_round) {
    if (rope_base < 0.0 || (rope_base > 0.0 && (D % 2 != 0))) return -1;
    const int rope = rope_base > 0.0;
    if (!q || !k || !v || !o || !lse || !slice_b || !slice_h) return -1;
    if (B < 0 || Hq <= 0 || Hkv <= 0 || Sq < 0 || Sk < 0 || D <= 0) return -1;
    if (Hq % Hkv != 0) return -1;
    if (mask_kind < ORACLE_MASK_NONE || mask_kind > ORACLE_MASK_CAUSAL_ADDITIVE) return -1;
    int causal = (mask_kind == ORACLE_MASK_CAUSAL || mask_kind == ORACLE_MASK_CAUSAL_ADDITIVE);
    int additive = (mask_kind == ORACLE_MASK_ADDITIVE || mask_kind == ORACLE_MASK_CAUSAL_ADDITIVE);
    if (additive && !mask) return -1;
    if (row_begin < 0 || row_end > Sq || row_begin > row_end) return -1;
    if (!(scale > 0.0) || !isfinite(scale)) scale = 1.0 / sqrt((double)D);

    const int group = Hq / Hkv;            /* query heads per K/V head */
    const int rows = row_end - row_begin;
    const long long causal_offset = (long long)Sk - (long long)Sq;

#ifdef _OPENMP
    if (n_threads > 0) omp_set_num_threads(n_threads);
#else
    (void)n_threads;
#endif

    for (int s = 0; s < n_slices; ++s) {
        const int b = slice_b[s], h = slice_h[s];
        if (b < 0 || b >= B || h < 0 || h >= Hq) return -1;
        const int g = h / group;

        /* Widen this slice's K and V once: (Sk, D) each. */
        double *kd = (double *)malloc(sizeof(double) * ((size_t)Sk * D + 1));
        double *vd = (double *)malloc(sizeof(double) * ((size_t)Sk * D + 1));
        if (!kd || !vd) { free(kd); free(vd); return -1; }
        for (long long j = 0; j < Sk; ++j)
            for (int d = 0; d < D; ++d) {
                size_t src = (((size_t)b * Sk + j) * Hkv + g) * D + d;
                kd[j * D + d] = widen(k[src], dtype);
                vd[j * D + d] = widen(v[src], dtype);
            }
        if (rope)
            for (long long j = 0; j < Sk; ++j) rope_rotate(kd + j * D, D, k_pos0 + j, rope_base, rope_round, dtype);

        int failed = 0;
#pragma omp parallel
        {
            double *srow = (double *)malloc(sizeof(double) * ((size_t)Sk + 1));
            double *qd = (double *)malloc(sizeof(double) * (size_t)D);
            if (!srow || !qd) {
#pragma omp atomic write
                failed = 1;
            } else {
#pragma omp for schedule(dynamic, 4)
                for (int r = 0; r < rows; ++r) {
                    const long long i = (long long)row_begin + r;
                    double *orow = o + ((size_t)s * rows + r) * D;
                    for (int d = 0; d < D; ++d)
                        qd[d] = widen(q[(((size_t)b * Sq + i) * Hq + h) * D + d], dtype);
                    if (rope) rope_rotate(qd, D, q_pos0 + i, rope_base, rope_round, dtype);

                    /* Scores, then pass 1: the row maximum. */
                    double m = -INFINITY;
                    for (long long j = 0; j < Sk; ++j) {
                        if (causal && j > i + causal_offset) { srow[j] = -INFINITY; continue; }
                        double dot = 0.0;
                        for (int d = 0; d < D; ++d) dot += qd[d] * kd[j * D + d];
                        double sij = scale * dot;
                        if (additive) sij += (double)mask[((size_t)b * Sq + i) * Sk + j];
                        srow[j] = sij;
                        if (sij > m) m = sij;
                    }

                    if (m == -INFINITY) {          /* no visible key */
                        for (int d = 0; d < D; ++d) orow[d] = 0.0;
                        lse[(size_t)s * rows + r] = -INFINITY;
                        if (psum) psum[(size_t)s * rows + r] = 0.0;
                        continue;
                    }

                    /* Pass 2: exponentials and their sum. */
                    double l = 0.0;
                    for (long long j = 0; j < Sk; ++j) {
                        srow[j] = exp(srow[j] - m);
                        l += srow[j];
                    }

                    /* Normalised probabilities times V. */
                    double ps = 0.0;
                    for (int d = 0; d < D; ++d) orow[d] = 0.0;
                    for (long long j = 0; j < Sk; ++j) {
                        double pij = srow[j] / l;
                        ps += pij;
                        for (int d = 0; d < D; ++d) orow[d] += pij * vd[j * D + d];
                    }
                    lse[(size_t)s * rows + r] = m + log(l);
                    if (psum) psum[(size_t)s * rows + r] = ps;
                }
            }
            free(srow);
            free(qd);
        }
        free(kd);
        free(vd);
        if (failed) return -1;
    }
    return 0;
}

/*
 * The rotation alone (for checking a rotation kernel): x is a (B, S, H, D)
 * tensor of 16-bit patterns, row s at position pos0 + s; y receives the
 * rotated (and, with rope_round, re-rounded) values in FP64, same layout.
 * Returns 0, or -1 on an invalid argument.
 */
int oracle_rope_rotate(const uint16_t *x, int dtype, int B, int S, int H, int D, double base,
                       long long pos0, int rope_round, double *y) {
    if (!x || !y || B < 0 || S < 0 || H < 0 || D <= 0 || D % 2 != 0 || !(base > 0.0)) return -1;
    for (long long b = 0; b < B; ++b)
        for (long long s = 0; s < S; ++s)
            for (long long h = 0; h < H; ++h) {
                const size_t off = (((size_t)b * S + s) * H + h) * D;
                for (int d = 0; d < D; ++d) y[off + d] = widen(x[off + d], dtype);
                rope_rotate(y + off, D, pos0 + s, base, rope_round, dtype);
            }
    return 0;
}

int oracle_attn_fwd(const uint16_t *q, const uint16_t *k, const uint16_t *v, int dtype,
                    const float *mask, int mask_kind,
                    int B, int Hq, int Hkv, int Sq, int Sk, int D, double scale,
                    int n_slices, const int32_t *slice_b, const int32_t *slice_h,
                    int row_begin, int row_end,
                    double *o, double *lse, double *psum, int n_threads) {
    return oracle_attn_fwd_rope(q, k, v, dtype, mask, mask_kind, B, Hq, Hkv, Sq, Sk, D, scale,
                                n_slices, slice_b, slice_h, row_begin, row_end, o, lse, psum, n_threads,
                                0.0, 0, 0, 0);
}
