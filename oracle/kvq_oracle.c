/*
 * kvq_oracle.c -- plain, slow CPU oracle for the streamed QKV projection with
 * rotated, group-scaled, packed low-bit K/V and the packed-K/V attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the library links, imports or calls
 * this file; only the test suite, the smoke check and the benchmark's CPU
 * baseline do.  It shares no source with the CUDA path.
 *
 * Sources (web pages, by title and section):
 *  [I]  "Feature Request: Streamed QKV Projection and Packed Low-Bit K/V
 *       Support for Extreme Long-Sequence Attention" (comfy-kitchen issue 119):
 *       sections "Proposed backend capability" (Q kept BF16, K/V rotated,
 *       quantised, packed to 4 bits; attention decodes K/V tile by tile),
 *       "Potential reduction" (byte arithmetic), "Quality-oriented low-bit
 *       format" (orthogonal/Hadamard rotation, per-group scaling) and
 *       "Mixed precision for conditioning" (INT8 K/V for chosen token ranges).
 *  [V]  vram_lab.py ("VRAM Lab", ComfyUI-MAINodes): `_hadamard` (Sylvester
 *       doubling, divided by sqrt(n)), `_online_combine` and the kvi8r store
 *       docstring (rotated-basis identities q.k = (qH).(kH), P.V = (P.(VH)).H^T),
 *       `_fq_int4` (scale = group absmax / 7, round half to even), `_Int8KV`
 *       (rotated INT8 rows, absmax / 127), `_phase1_kv` (fused qkv row split
 *       into [q | k | v], heads of 128 contiguous columns) and `_norm_rope`
 *       (per-head RMSNorm on Q and K before attention).
 *
 * Precision.  Everything that decides an integer (the rotation feeding the
 * quantiser, the scale, the division and the rounding) runs in IEEE fp32 in a
 * fixed order: exactly the arithmetic the format is defined by.  Dot products,
 * RMSNorm statistics and the softmax accumulate in fp64 and are rounded to
 * fp32 where the definition hands a value on (the projection accumulator, the
 * attention output).  Build with -ffp-contract=off and without fast-math.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define HD 128 /* head dimension: the rotation is 128-point */

/* ------------------------------------------------------------------ number formats */

/* bfloat16 bits -> fp32 (exact: bf16 is the top half of an fp32). */
float kvqo_bf16_to_f32(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

/* fp32 -> bfloat16, round to nearest, ties to even (NaN stays NaN). */
uint16_t kvqo_f32_to_bf16(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    if ((u & 0x7FFFFFFFu) > 0x7F800000u) return (uint16_t)((u >> 16) | 0x0040u);
    uint32_t r = u + 0x7FFFu + ((u >> 16) & 1u);
    return (uint16_t)(r >> 16);
}

/* IEEE binary16 bits -> fp32 (exact). */
float kvqo_f16_to_f32(uint16_t h) {
    uint32_t sign = (uint32_t)(h & 0x8000u) << 16;
    uint32_t e = (h >> 10) & 0x1Fu;
    uint32_t m = h & 0x3FFu;
    uint32_t u;
    if (e == 0) {
        if (m == 0) {
            u = sign;
        } else { /* subnormal: m * 2^-24, exact in fp32 */
            float f = (float)m * 5.9604644775390625e-08f;
            memcpy(&u, &f, 4);
            u |= sign;
        }
    } else if (e == 31) {
        u = sign | 0x7F800000u | (m << 13);
    } else {
        u = sign | ((e - 15 + 127) << 23) | (m << 13);
    }
    float f;
    memcpy(&f, &u, 4);
    return f;
}

/* fp32 -> IEEE binary16, round to nearest, ties to even; overflow -> inf. */
uint16_t kvqo_f32_to_f16(float f) {
    uint32_t x;
    memcpy(&x, &f, 4);
    uint16_t sign = (uint16_t)((x >> 16) & 0x8000u);
    uint32_t ax = x & 0x7FFFFFFFu;
    if (ax >= 0x7F800000u) /* inf or NaN */
        return (uint16_t)(sign | 0x7C00u | (ax > 0x7F800000u ? 0x0200u : 0u));
    if (ax >= 0x47800000u) return (uint16_t)(sign | 0x7C00u); /* >= 65536 */
    int e = (int)(ax >> 23) - 127;
    if (e < -25) return sign; /* below half the smallest subnormal */
    uint32_t mant = (ax & 0x7FFFFFu) | 0x800000u; /* 24 significant bits */
    uint32_t q, rem, half;
    int shift;
    if (e < -14) { /* binary16 subnormal: keep bits down to 2^-24 */
        shift = 13 + (-14 - e);
        q = mant >> shift;
        rem = mant & ((1u << shift) - 1u);
        half = 1u << (shift - 1);
    } else {
        q = ((uint32_t)(e + 15) << 10) | ((mant >> 13) & 0x3FFu);
        rem = mant & 0x1FFFu;
        half = 0x1000u;
    }
    if (rem > half || (rem == half && (q & 1u))) q++; /* a carry may reach inf: correct */
    return (uint16_t)(sign | q);
}

/* ------------------------------------------------------------------ rotation */

/* c = fp32(1/sqrt(128)): the normalisation of the Sylvester Hadamard matrix
 * ([V] `_hadamard`: h / n**0.5). */
float kvqo_rot_scale(void) { return (float)(1.0 / sqrt(128.0)); }

/* y = x . H for one 128-vector, H = Sylvester Hadamard-128 / sqrt(128)
 * (symmetric, so x.H = H.x and H^T = H).  Computed as the unnormalised fast
 * Walsh-Hadamard transform, butterfly strides 1, 2, 4, ..., 64, each butterfly
 * (a, b) -> (a + b, a - b) in fp32, followed by one fp32 multiply by c.  This
 * order is part of the format: quantisation codes are decided on its result. */
void kvqo_rotate128(const float *x, float *y) {
    float v[HD];
    for (int i = 0; i < HD; ++i) v[i] = x[i];
    for (int h = 1; h < HD; h <<= 1) {
        for (int i = 0; i < HD; ++i) {
            if (i & h) continue;
            float a = v[i], b = v[i + h];
            v[i] = a + b;
            v[i + h] = a - b;
        }
    }
    const float c = kvqo_rot_scale();
    for (int i = 0; i < HD; ++i) y[i] = v[i] * c;
}

/* Rotate `rows` consecutive 128-vectors. */
void kvqo_rotate(const float *x, int64_t rows, float *y) {
    for (int64_t r = 0; r < rows; ++r) kvqo_rotate128(x + r * HD, y + r * HD);
}

/* ------------------------------------------------------------------ quantiser */

/* Quantise one rotated head vector y[128] ([I] "Quality-oriented low-bit
 * format": per-group scaling; [V] `_fq_int4`: scale = absmax/7, round half to
 * even).  For each group of `group` elements:
 *   amax = max |y|            (fp32)
 *   s    = fp16_rn(amax / Q)  (Q = 7 for bits=4, 127 for bits=8; IEEE division)
 *   code = 0                                  if s == 0
 *        = clamp(rint(y / float(s)), -Q, Q)   otherwise (IEEE division, ties to even)
 * Packing: bits=4 puts element 2i in the low nibble and 2i+1 in the high
 * nibble of byte i, as 4-bit two's complement (64 bytes per head); bits=8
 * stores one int8 per element (128 bytes per head).  `scales` gets 128/group
 * fp16 bit patterns. */
void kvqo_quant_head(const float *y, int group, int bits, uint8_t *codes, uint16_t *scales) {
    const float qmax = (bits == 4) ? 7.0f : 127.0f;
    int8_t q[HD];
    for (int g0 = 0; g0 < HD; g0 += group) {
        float amax = 0.0f;
        for (int i = g0; i < g0 + group; ++i) {
            float a = fabsf(y[i]);
            if (a > amax) amax = a;
        }
        uint16_t s16 = kvqo_f32_to_f16(amax / qmax);
        float s = kvqo_f16_to_f32(s16);
        scales[g0 / group] = s16;
        for (int i = g0; i < g0 + group; ++i) {
            float r = (s == 0.0f) ? 0.0f : nearbyintf(y[i] / s);
            if (r > qmax) r = qmax;
            if (r < -qmax) r = -qmax;
            q[i] = (int8_t)r;
        }
    }
    if (bits == 4) {
        for (int i = 0; i < HD / 2; ++i)
            codes[i] = (uint8_t)(((uint8_t)q[2 * i] & 0x0Fu) | (((uint8_t)q[2 * i + 1] & 0x0Fu) << 4));
    } else {
        for (int i = 0; i < HD; ++i) codes[i] = (uint8_t)q[i];
    }
}

/* Integer code of element i of a packed head (sign-extended nibble or int8). */
static int code_at(const uint8_t *codes, int bits, int i) {
    if (bits == 8) return (int)(int8_t)codes[i];
    int nib = (i & 1) ? (codes[i >> 1] >> 4) : (codes[i >> 1] & 0x0F);
    return (nib & 0x8) ? nib - 16 : nib;
}

/* Dequantise one packed head to fp32 in the rotated basis: code * float(s)
 * (exact in fp32: |code| <= 127 and s has 11 significant bits). */
void kvqo_dequant_head(const uint8_t *codes, const uint16_t *scales, int group, int bits, float *y) {
    for (int i = 0; i < HD; ++i) y[i] = (float)code_at(codes, bits, i) * kvqo_f16_to_f32(scales[i / group]);
}

static int check_fmt(int hidden, int group, int bits) {
    if (hidden <= 0 || hidden % HD) return 1;
    if (group != 32 && group != 64 && group != 128) return 1;
    if (bits != 4 && bits != 8) return 1;
    return 0;
}

/* ------------------------------------------------------------------ a1: rotate + quantise + pack */

/* K/V rows -> packed store, for the token rows listed in `rows`.
 * kv: BF16 bits, row t at kv + t*ld; K is columns [0, hidden), V is columns
 * [hidden, 2*hidden); head h of each is the 128 columns starting at h*128
 * ([V] `_phase1_kv` split).  Outputs are compact and token-major:
 *   codes [n_rows][heads][128*bits/8], scales [n_rows][heads][128/group]. */
int kvqo_kv_rotate_quant_pack(const uint16_t *kv, int64_t ld, int hidden, const int64_t *rows, int64_t n_rows,
                              int group, int bits, uint8_t *k_codes, uint8_t *v_codes, uint16_t *k_scales,
                              uint16_t *v_scales) {
    if (check_fmt(hidden, group, bits)) return 1;
    const int heads = hidden / HD, cb = HD * bits / 8, sg = HD / group;
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < n_rows; ++r) {
        const uint16_t *row = kv + rows[r] * ld;
        float x[HD], y[HD];
        for (int kvi = 0; kvi < 2; ++kvi) {
            uint8_t *cd = kvi ? v_codes : k_codes;
            uint16_t *sc = kvi ? v_scales : k_scales;
            for (int h = 0; h < heads; ++h) {
                for (int i = 0; i < HD; ++i) x[i] = kvqo_bf16_to_f32(row[kvi * hidden + h * HD + i]);
                kvqo_rotate128(x, y);
                kvqo_quant_head(y, group, bits, cd + (r * heads + h) * cb, sc + (r * heads + h) * sg);
            }
        }
    }
    return 0;
}

/* a1b: compact packed rows (layout of kvqo_kv_rotate_quant_pack) -> BF16 K/V
 * rows [n_rows][2*hidden]: dequantise, rotate back (H^T = H), round to BF16. */
int kvqo_kv_unpack(const uint8_t *k_codes, const uint8_t *v_codes, const uint16_t *k_scales, const uint16_t *v_scales,
                   int64_t n_rows, int hidden, int group, int bits, uint16_t *kv_out) {
    if (check_fmt(hidden, group, bits)) return 1;
    const int heads = hidden / HD, cb = HD * bits / 8, sg = HD / group;
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < n_rows; ++r) {
        float x[HD], y[HD];
        for (int kvi = 0; kvi < 2; ++kvi) {
            const uint8_t *cd = kvi ? v_codes : k_codes;
            const uint16_t *sc = kvi ? v_scales : k_scales;
            for (int h = 0; h < heads; ++h) {
                kvqo_dequant_head(cd + (r * heads + h) * cb, sc + (r * heads + h) * sg, group, bits, x);
                kvqo_rotate128(x, y);
                for (int i = 0; i < HD; ++i)
                    kv_out[r * 2 * hidden + kvi * hidden + h * HD + i] = kvqo_f32_to_bf16(y[i]);
            }
        }
    }
    return 0;
}

/* ------------------------------------------------------------------ a2: QKV projection + epilogue */

/* Per-head RMSNorm of one 128-vector in place: v * (1/sqrt(mean(v^2) + eps)) * w
 * ([V] `_norm_rope`: q_norm / k_norm applied per head before attention). */
static void rmsnorm128(float *v, const float *w, float eps) {
    double ss = 0.0;
    for (int i = 0; i < HD; ++i) ss += (double)v[i] * (double)v[i];
    double r = 1.0 / sqrt(ss / HD + (double)eps);
    for (int i = 0; i < HD; ++i) v[i] = (float)((double)v[i] * r * (double)w[i]);
}

/* Split-half rotary position embedding of one head vector, in place
 * ([V] `_norm_rope`: "fused RMSNorm + split-half RoPE", rot_dim = twice the
 * table's frequency count; the table itself is the caller's).  With h =
 * rot_dim/2 and (c_i, s_i) = cs[2i], cs[2i+1] for i < h:
 *   y_i     = x_i c_i - x_{i+h} s_i
 *   y_{i+h} = x_{i+h} c_i + x_i s_i
 * dims >= rot_dim unchanged; fp64 products and sum, rounded to fp32. */
static void rope_split_half(float *v, const float *cs, int rot_dim) {
    const int h = rot_dim / 2;
    for (int i = 0; i < h; ++i) {
        const double c = cs[2 * i], sn = cs[2 * i + 1], a = v[i], b = v[i + h];
        v[i] = (float)(a * c - b * sn);
        v[i + h] = (float)(b * c + a * sn);
    }
}

/* For each listed token row t: acc = x[t] . W^T ([I] "Proposed backend
 * capability": the fused QKV GEMM), accumulated in fp64 and rounded to fp32.
 * Columns [0,C) are Q, [C,2C) K, [2C,3C) V, head h = 128 columns from h*128.
 * Q: optional RMSNorm (q_norm_w[128], may be NULL) -> optional split-half
 * RoPE (rope_cs: rot_dim floats per token row, (cos, sin) pairs, row t at
 * rope_cs + t*rot_dim; NULL = none) -> rotate -> q_f32 and its BF16 rounding
 * q_bf16.  K: optional RMSNorm (k_norm_w) -> optional RoPE -> rotate -> quantise.
 * V: rotate -> quantise.  The rotation and quantiser take the fp32
 * accumulator, with no BF16 rounding in between.  Outputs compact token-major
 * as in kvqo_kv_rotate_quant_pack; q_f32 / q_bf16 are [n_rows][C].  k_rot and
 * v_rot (optional, [n_rows][C] fp32) receive the rotated K and V vectors that
 * the quantiser is given, so a caller can see how close each code and scale
 * sits to a rounding boundary. */
int kvqo_qkv_proj(const uint16_t *x, const uint16_t *w, int hidden, const int64_t *rows, int64_t n_rows, int group,
                  int bits, const float *q_norm_w, const float *k_norm_w, float eps, const float *rope_cs, int rot_dim,
                  float *q_f32, uint16_t *q_bf16, uint8_t *k_codes, uint8_t *v_codes, uint16_t *k_scales,
                  uint16_t *v_scales, float *k_rot, float *v_rot) {
    if (check_fmt(hidden, group, bits)) return 1;
    if (rope_cs && (rot_dim < 2 || rot_dim > HD || rot_dim % 2)) return 1;
    const int C = hidden, heads = C / HD, cb = HD * bits / 8, sg = HD / group;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t r = 0; r < n_rows; ++r) {
        const uint16_t *xr = x + rows[r] * (int64_t)C;
        float *xf = (float *)malloc(sizeof(float) * (size_t)C);
        float *acc = (float *)malloc(sizeof(float) * (size_t)3 * C);
        for (int k = 0; k < C; ++k) xf[k] = kvqo_bf16_to_f32(xr[k]);
        for (int o = 0; o < 3 * C; ++o) {
            const uint16_t *wr = w + (int64_t)o * C;
            double s = 0.0;
            for (int k = 0; k < C; ++k) s += (double)xf[k] * (double)kvqo_bf16_to_f32(wr[k]);
            acc[o] = (float)s;
        }
        float y[HD];
        for (int h = 0; h < heads; ++h) {
            float *q = acc + h * HD, *kk = acc + C + h * HD, *vv = acc + 2 * C + h * HD;
            if (q_norm_w) rmsnorm128(q, q_norm_w, eps);
            if (rope_cs) rope_split_half(q, rope_cs + rows[r] * rot_dim, rot_dim);
            kvqo_rotate128(q, y);
            for (int i = 0; i < HD; ++i) {
                if (q_f32) q_f32[r * C + h * HD + i] = y[i];
                if (q_bf16) q_bf16[r * C + h * HD + i] = kvqo_f32_to_bf16(y[i]);
            }
            if (k_norm_w) rmsnorm128(kk, k_norm_w, eps);
            if (rope_cs) rope_split_half(kk, rope_cs + rows[r] * rot_dim, rot_dim);
            kvqo_rotate128(kk, y);
            if (k_rot) memcpy(k_rot + r * C + h * HD, y, sizeof(y));
            kvqo_quant_head(y, group, bits, k_codes + (r * heads + h) * cb, k_scales + (r * heads + h) * sg);
            kvqo_rotate128(vv, y);
            if (v_rot) memcpy(v_rot + r * C + h * HD, y, sizeof(y));
            kvqo_quant_head(y, group, bits, v_codes + (r * heads + h) * cb, v_scales + (r * heads + h) * sg);
        }
        free(xf);
        free(acc);
    }
    return 0;
}

/* ------------------------------------------------------------------ a4: packed-K/V attention */

/* Attention of the listed query rows against a packed K/V store
 * ([I] "Proposed backend capability": attention consumes Q BF16 and packed
 * K/V; [V] kvi8r docstring: in the rotated basis q.k = (qH).(kH) and
 * P.V = (P.(VH)).H^T, so rotated Q against rotated K/V, then one un-rotation).
 *
 * q: BF16 bits, rotated basis, row i at q + i*ldq, head h at columns h*128.
 * Store (the library's layout): head-major, codes [heads][n_pad][128*bits/8],
 * scales [heads][n_pad][128/group]; keys 0..n_kv-1 are used.
 * For each listed row i and head h:
 *   s_j = (q . k^_j) * sm_scale,  k^_j = code * float(scale)  (dequantised, exact)
 *   p_j = exp(s_j - max_j s_j),   o = sum_j p_j v^_j / sum_j p_j
 *   out[r] = o . H                (un-rotation: the fp32 rotation above)
 * Plain two-pass softmax over all keys; dot products and sums in fp64, o
 * rounded to fp32 before the un-rotation.  out: fp32 [n_rows][heads*128]. */
static void attend_head(const float *qf, const float *Kd, const float *Vd, int64_t n_kv, float sm_scale, float *o_out,
                        double *p) {
    double m = -HUGE_VAL;
    for (int64_t j = 0; j < n_kv; ++j) {
        const float *k = Kd + j * HD;
        double s = 0.0;
        for (int d = 0; d < HD; ++d) s += (double)qf[d] * (double)k[d];
        s *= (double)sm_scale;
        p[j] = s;
        if (s > m) m = s;
    }
    double l = 0.0;
    for (int64_t j = 0; j < n_kv; ++j) {
        p[j] = exp(p[j] - m);
        l += p[j];
    }
    double o[HD];
    for (int d = 0; d < HD; ++d) o[d] = 0.0;
    for (int64_t j = 0; j < n_kv; ++j) {
        const float *v = Vd + j * HD;
        for (int d = 0; d < HD; ++d) o[d] += p[j] * (double)v[d];
    }
    float of[HD];
    for (int d = 0; d < HD; ++d) of[d] = (float)(o[d] / l);
    kvqo_rotate128(of, o_out);
}

int kvqo_attention(const uint16_t *q, int64_t ldq, int heads, const uint8_t *k_codes, const uint8_t *v_codes,
                   const uint16_t *k_scales, const uint16_t *v_scales, int64_t n_kv, int64_t n_pad, int group,
                   int bits, float sm_scale, const int64_t *rows, int64_t n_rows, float *out) {
    if (check_fmt(heads * HD, group, bits) || n_kv < 1 || n_pad < n_kv) return 1;
    const int cb = HD * bits / 8, sg = HD / group, C = heads * HD;
    float *Kd = (float *)malloc(sizeof(float) * (size_t)n_kv * HD);
    float *Vd = (float *)malloc(sizeof(float) * (size_t)n_kv * HD);
    if (!Kd || !Vd) {
        free(Kd);
        free(Vd);
        return 2;
    }
    for (int h = 0; h < heads; ++h) {
#pragma omp parallel for schedule(static)
        for (int64_t j = 0; j < n_kv; ++j) {
            int64_t t = (int64_t)h * n_pad + j;
            kvqo_dequant_head(k_codes + t * cb, k_scales + t * sg, group, bits, Kd + j * HD);
            kvqo_dequant_head(v_codes + t * cb, v_scales + t * sg, group, bits, Vd + j * HD);
        }
#pragma omp parallel
        {
            double *p = (double *)malloc(sizeof(double) * (size_t)n_kv);
#pragma omp for schedule(dynamic, 1)
            for (int64_t r = 0; r < n_rows; ++r) {
                float qf[HD];
                for (int d = 0; d < HD; ++d) qf[d] = kvqo_bf16_to_f32(q[rows[r] * ldq + h * HD + d]);
                attend_head(qf, Kd, Vd, n_kv, sm_scale, out + r * C + h * HD, p);
            }
            free(p);
        }
    }
    free(Kd);
    free(Vd);
    return 0;
}

/* Causal attention over the same store (a reading: the pages only name a
 * general packed-K/V attention primitive, [I] "Proposed backend capability";
 * the causal form is the standard prefix mask).  Listed row i sits at key
 * position q_pos0 + i and attends keys j <= q_pos0 + i, j < n_kv, which is
 * the attention above over the prefix of min(n_kv, q_pos0 + i + 1) keys.
 * q_pos0 >= 0, so every row sees key 0. */
int kvqo_attention_causal(const uint16_t *q, int64_t ldq, int heads, const uint8_t *k_codes, const uint8_t *v_codes,
                          const uint16_t *k_scales, const uint16_t *v_scales, int64_t n_kv, int64_t n_pad, int group,
                          int bits, float sm_scale, int64_t q_pos0, const int64_t *rows, int64_t n_rows, float *out) {
    if (check_fmt(heads * HD, group, bits) || n_kv < 1 || n_pad < n_kv || q_pos0 < 0) return 1;
    const int cb = HD * bits / 8, sg = HD / group, C = heads * HD;
    float *Kd = (float *)malloc(sizeof(float) * (size_t)n_kv * HD);
    float *Vd = (float *)malloc(sizeof(float) * (size_t)n_kv * HD);
    if (!Kd || !Vd) {
        free(Kd);
        free(Vd);
        return 2;
    }
    for (int h = 0; h < heads; ++h) {
#pragma omp parallel for schedule(static)
        for (int64_t j = 0; j < n_kv; ++j) {
            int64_t t = (int64_t)h * n_pad + j;
            kvqo_dequant_head(k_codes + t * cb, k_scales + t * sg, group, bits, Kd + j * HD);
            kvqo_dequant_head(v_codes + t * cb, v_scales + t * sg, group, bits, Vd + j * HD);
        }
#pragma omp parallel
        {
            double *p = (double *)malloc(sizeof(double) * (size_t)n_kv);
#pragma omp for schedule(dynamic, 1)
            for (int64_t r = 0; r < n_rows; ++r) {
                float qf[HD];
                for (int d = 0; d < HD; ++d) qf[d] = kvqo_bf16_to_f32(q[rows[r] * ldq + h * HD + d]);
                const int64_t vis = q_pos0 + rows[r] + 1;
                attend_head(qf, Kd, Vd, vis < n_kv ? vis : n_kv, sm_scale, out + r * C + h * HD, p);
            }
            free(p);
        }
    }
    free(Kd);
    free(Vd);
    return 0;
}

/* Mixed-precision store ([I] "Mixed precision for conditioning": chosen
 * token ranges at INT8, the rest at rotated INT4).  Each of the n_ranges
 * ranges [start, start+len) has its own head-major store of `bits` (4 or 8)
 * with row capacity cap (codes [heads][cap][128*bits/8], scales
 * [heads][cap][128/group]); key j of the sequence is row j - start of the
 * range holding it.  Both precisions are in the same rotated basis, so the
 * attention is the one above over the concatenated, dequantised keys. */
int kvqo_attention_mixed(const uint16_t *q, int64_t ldq, int heads, int n_ranges, const int64_t *starts,
                         const int64_t *lens, const int *bitss, const int64_t *caps, const uint8_t *const *k_codes,
                         const uint8_t *const *v_codes, const uint16_t *const *k_scales,
                         const uint16_t *const *v_scales, int group, float sm_scale, const int64_t *rows,
                         int64_t n_rows, float *out) {
    int64_t n_kv = 0;
    for (int g = 0; g < n_ranges; ++g) {
        if (check_fmt(heads * HD, group, bitss[g]) || lens[g] < 1 || caps[g] < lens[g] || starts[g] != n_kv) return 1;
        n_kv += lens[g];
    }
    const int sg = HD / group, C = heads * HD;
    float *Kd = (float *)malloc(sizeof(float) * (size_t)n_kv * HD);
    float *Vd = (float *)malloc(sizeof(float) * (size_t)n_kv * HD);
    if (!Kd || !Vd) {
        free(Kd);
        free(Vd);
        return 2;
    }
    for (int h = 0; h < heads; ++h) {
        for (int g = 0; g < n_ranges; ++g) {
            const int cb = HD * bitss[g] / 8;
#pragma omp parallel for schedule(static)
            for (int64_t j = 0; j < lens[g]; ++j) {
                int64_t t = (int64_t)h * caps[g] + j;
                kvqo_dequant_head(k_codes[g] + t * cb, k_scales[g] + t * sg, group, bitss[g], Kd + (starts[g] + j) * HD);
                kvqo_dequant_head(v_codes[g] + t * cb, v_scales[g] + t * sg, group, bitss[g], Vd + (starts[g] + j) * HD);
            }
        }
#pragma omp parallel
        {
            double *p = (double *)malloc(sizeof(double) * (size_t)n_kv);
#pragma omp for schedule(dynamic, 1)
            for (int64_t r = 0; r < n_rows; ++r) {
                float qf[HD];
                for (int d = 0; d < HD; ++d) qf[d] = kvqo_bf16_to_f32(q[rows[r] * ldq + h * HD + d]);
                attend_head(qf, Kd, Vd, n_kv, sm_scale, out + r * C + h * HD, p);
            }
            free(p);
        }
    }
    free(Kd);
    free(Vd);
    return 0;
}

/* ------------------------------------------------------------------ next row f3: attention over key chunks */

/* One query row and head against one chunk of keys ([V] `_blockwise_attention`
 * and `_blockwise_attention_q`: each K/V block gives a partial result and its
 * log-sum-exp, later merged by `_online_combine`).  In the rotated basis, with
 * s_j = (q . k^_j) * sm_scale over the chunk's keys:
 *   o   = sum_j exp(s_j - m) v^_j / sum_j exp(s_j - m),   m = max_j s_j
 *   lse = m + log(sum_j exp(s_j - m))      (= log sum_j exp(s_j))
 * o is NOT un-rotated (the merge works in the rotated basis, and the single
 * un-rotation comes at the end).  fp64 throughout. */
static void partial_head(const float *qf, const float *Kd, const float *Vd, int64_t n_kv, float sm_scale, double *o,
                         double *lse, double *p) {
    double m = -HUGE_VAL;
    for (int64_t j = 0; j < n_kv; ++j) {
        const float *k = Kd + j * HD;
        double s = 0.0;
        for (int d = 0; d < HD; ++d) s += (double)qf[d] * (double)k[d];
        s *= (double)sm_scale;
        p[j] = s;
        if (s > m) m = s;
    }
    double l = 0.0;
    for (int64_t j = 0; j < n_kv; ++j) {
        p[j] = exp(p[j] - m);
        l += p[j];
    }
    for (int d = 0; d < HD; ++d) o[d] = 0.0;
    for (int64_t j = 0; j < n_kv; ++j) {
        const float *v = Vd + j * HD;
        for (int d = 0; d < HD; ++d) o[d] += p[j] * (double)v[d];
    }
    for (int d = 0; d < HD; ++d) o[d] /= l;
    *lse = m + log(l);
}

/* Partial attention of the listed query rows against one key chunk given as a
 * range table (layout and arguments as kvqo_attention_mixed).  Outputs, fp64:
 *   o_out   [n_rows][heads][128]  normalised output in the rotated basis
 *   lse_out [n_rows][heads]       natural log of sum_j exp(s_j) over the chunk */
int kvqo_attention_partial(const uint16_t *q, int64_t ldq, int heads, int n_ranges, const int64_t *starts,
                           const int64_t *lens, const int *bitss, const int64_t *caps, const uint8_t *const *k_codes,
                           const uint8_t *const *v_codes, const uint16_t *const *k_scales,
                           const uint16_t *const *v_scales, int group, float sm_scale, const int64_t *rows,
                           int64_t n_rows, double *o_out, double *lse_out) {
    int64_t n_kv = 0;
    for (int g = 0; g < n_ranges; ++g) {
        if (check_fmt(heads * HD, group, bitss[g]) || lens[g] < 1 || caps[g] < lens[g] || starts[g] != n_kv) return 1;
        n_kv += lens[g];
    }
    if (n_kv < 1) return 1;
    const int sg = HD / group;
    float *Kd = (float *)malloc(sizeof(float) * (size_t)n_kv * HD);
    float *Vd = (float *)malloc(sizeof(float) * (size_t)n_kv * HD);
    if (!Kd || !Vd) {
        free(Kd);
        free(Vd);
        return 2;
    }
    for (int h = 0; h < heads; ++h) {
        for (int g = 0; g < n_ranges; ++g) {
            const int cb = HD * bitss[g] / 8;
#pragma omp parallel for schedule(static)
            for (int64_t j = 0; j < lens[g]; ++j) {
                int64_t t = (int64_t)h * caps[g] + j;
                kvqo_dequant_head(k_codes[g] + t * cb, k_scales[g] + t * sg, group, bitss[g], Kd + (starts[g] + j) * HD);
                kvqo_dequant_head(v_codes[g] + t * cb, v_scales[g] + t * sg, group, bitss[g], Vd + (starts[g] + j) * HD);
            }
        }
#pragma omp parallel
        {
            double *p = (double *)malloc(sizeof(double) * (size_t)n_kv);
#pragma omp for schedule(dynamic, 1)
            for (int64_t r = 0; r < n_rows; ++r) {
                float qf[HD];
                for (int d = 0; d < HD; ++d) qf[d] = kvqo_bf16_to_f32(q[rows[r] * ldq + h * HD + d]);
                partial_head(qf, Kd, Vd, n_kv, sm_scale, o_out + (r * heads + h) * HD, lse_out + r * heads + h, p);
            }
            free(p);
        }
    }
    free(Kd);
    free(Vd);
    return 0;
}

/* log(exp(a) + exp(b)), computed from the larger argument. */
static double log_add_exp(double a, double b) {
    const double hi = a > b ? a : b, lo = a > b ? b : a;
    return hi + log1p(exp(lo - hi));
}

/* Merge of two partial results over disjoint key sets ([V] `_online_combine`):
 *   new = log(exp(lse_a) + exp(lse_b))
 *   o   = o_a * exp(lse_a - new) + o_b * exp(lse_b - new)
 * written into (o_a, lse_a).  n_vec vectors of 128, one lse each; fp64. */
void kvqo_lse_merge(double *o_a, double *lse_a, const double *o_b, const double *lse_b, int64_t n_vec) {
    for (int64_t i = 0; i < n_vec; ++i) {
        const double nw = log_add_exp(lse_a[i], lse_b[i]);
        const double wa = exp(lse_a[i] - nw), wb = exp(lse_b[i] - nw);
        for (int d = 0; d < HD; ++d) o_a[i * HD + d] = o_a[i * HD + d] * wa + o_b[i * HD + d] * wb;
        lse_a[i] = nw;
    }
}

/* The end of the chunked attention: each merged vector rounded to fp32 and
 * un-rotated once (the rotation of the format; H^T = H). */
void kvqo_partial_finish(const double *o, int64_t n_vec, float *out) {
    for (int64_t i = 0; i < n_vec; ++i) {
        float of[HD];
        for (int d = 0; d < HD; ++d) of[d] = (float)o[i * HD + d];
        kvqo_rotate128(of, out + i * HD);
    }
}

/* Number of OpenMP threads the oracle runs with (1 without OpenMP). */
#ifdef _OPENMP
#include <omp.h>
int kvqo_threads(void) { return omp_get_max_threads(); }
/* Sets the OpenMP threads of later calls (n >= 1). */
void kvqo_set_threads(int n) {
    if (n >= 1) omp_set_num_threads(n);
}
#else
int kvqo_threads(void) { return 1; }
void kvqo_set_threads(int n) { (void)n; }
#endif
