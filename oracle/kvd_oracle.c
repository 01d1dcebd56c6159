/*
 * kvd_oracle.c — plain, slow, fp64 CPU oracle for paged GQA decode attention.
 *
 * TEST INFRASTRUCTURE.  Only the test suite, the smoke check and the CPU
 * baseline leg of the benchmark may load this library.  It shares no code,
 * header, table or constant with the CUDA library and is written straight
 * from the definitions on the pages:
 *
 *  - FP8 E4M3 storage (1 sign, 4 exponent, 3 mantissa bits, max 448; store
 *    x / scale, multiply the scale back on read) and E5M2 (1·5·2 bits, max
 *    57,344): page "LLM에서 KV 캐시는 얼마나 생길까"
 *    (froggydisk.github.io/kv-cache-per-request), section "KV 캐시를 줄이는
 *    기법", FP8 format table and the paragraph after it.
 *  - Mixed-precision pages, one precision per block with the retention mask
 *    beside it: page "The KV Cache Is the New Memory Wall", §5.5.
 *  - Low-bit KV (INT4 / 2-bit codes with per-group scale and zero point): same
 *    page, §3.2 (2-bit storage raises decode intensity to 64 FLOP/B), §4.2,
 *    §4.6 and Tab. 7 (KIVI 2-bit, KVQuant INT4); the group layout is this
 *    oracle's reading (the pages give none).
 *  - Angle-domain keys (a radius and a code of the direction; the logit is
 *    ||q||·r̃·cos of the two codes): page "기술 요약: Spherical KV"
 *    (gist.science/ko/paper/2605.18856), §2.1; the direction code and the
 *    cosine's form are this oracle's reading (the page defines neither).
 *  - Paged cache: fixed 16-token blocks and a per-request block table that
 *    maps the request's j-th block to a physical block; the kernel walks the
 *    table in order, so scattered blocks give the same result: same page and
 *    section, PagedAttention paragraphs and the block-table example.
 *  - Decode attention per query head: softmax(q·Kᵀ/√d_h)·V, with groups of
 *    query heads sharing one KV head (GQA): same page, section "KV 캐시란".
 *  - Cumulative importance score
 *      s_i(t) = s_i(t-1) + (1/|L|) Σ_ℓ (1/H) Σ_h α_{ℓ,h}(t)[i]:
 *    page "기술 요약: 모든 사고가 HBM 을 필요로 하는 것은 아님"
 *    (gist.science/ko/paper/2605.09490), section "2. 중요도 점수화".
 *
 * Everything is fp64 except the FP8 quantise step, whose scale and x/scale
 * division are single-precision IEEE operations (the scale is an fp32 value
 * per (token, KV head)); the code choice is decided in that precision.
 *
 * Layout of the oracle's own pool (unrelated to the CUDA library's layout):
 * values  [num_blocks][n_kv][block_size][d_h]   (fp64, or e4m3 codes)
 * scales  [num_blocks][n_kv][block_size]        (fp32, FP8 mode only)
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define KVDO_OK 0
#define KVDO_ERR_INDEX 1   /* a block id or slot outside the pool */
#define KVDO_ERR_EMPTY 2   /* a head attends to no valid position */

/* ------------------------------------------------------------------ e4m3 */

/* Value of an E4M3 code: sign, 4-bit exponent with bias 7, 3-bit mantissa.
 * Exponent field 0 holds subnormals m·2^-9; S.1111.111 is NaN and there is
 * no infinity, so the largest finite magnitude is 1.75·2^8 = 448. */
double kvdo_e4m3_decode(uint8_t code) {
    int sign = code >> 7;
    int e = (code >> 3) & 0xF;
    int m = code & 0x7;
    double v;
    if (e == 0xF && m == 0x7) return NAN;
    if (e == 0)
        v = ldexp((double)m, -9);
    else
        v = ldexp(1.0 + m / 8.0, e - 7);
    return sign ? -v : v;
}

/* Nearest E4M3 code to y: the enumeration of all 127 non-negative finite
 * codes picks the closest value, a tie goes to the code with an even
 * mantissa, and magnitudes beyond 448 saturate to 448. */
uint8_t kvdo_e4m3_encode(float y) {
    if (isnan(y)) return 0x7F;
    int neg = signbit(y) ? 1 : 0;
    double a = fabs((double)y);
    int best = 0;
    double best_d = INFINITY;
    for (int c = 0; c <= 0x7E; ++c) {
        double d = fabs(a - kvdo_e4m3_decode((uint8_t)c));
        if (d < best_d || (d == best_d && (c & 1) == 0)) {
            best = c;
            best_d = d;
        }
    }
    if (a > 448.0) best = 0x7E;
    return (uint8_t)((neg << 7) | best);
}

void kvdo_e4m3_decode_array(const uint8_t* codes, int64_t n, double* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = kvdo_e4m3_decode(codes[i]);
}

void kvdo_e4m3_encode_array(const float* y, int64_t n, uint8_t* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = kvdo_e4m3_encode(y[i]);
}

/* One (token, KV head) row of d values: scale = absmax/448 in fp32 (1 when
 * the row is all zero), code_i = e4m3(x_i / scale) with an fp32 division. */
void kvdo_quantize_row(const float* x, int d, uint8_t* codes, float* scale_out) {
    float amax = 0.0f;
    for (int i = 0; i < d; ++i) {
        float a = fabsf(x[i]);
        if (a > amax) amax = a;
    }
    float scale = (amax == 0.0f) ? 1.0f : amax / 448.0f;
    for (int i = 0; i < d; ++i) {
        float y = x[i] / scale;
        codes[i] = kvdo_e4m3_encode(y);
    }
    *scale_out = scale;
}

void kvdo_quantize_rows(const float* x, int64_t rows, int d, uint8_t* codes, float* scales) {
    for (int64_t r = 0; r < rows; ++r) kvdo_quantize_row(x + r * d, d, codes + r * d, scales + r);
}

/* ------------------------------------------------------------------ e5m2 */

/* Value of an E5M2 code: sign, 5-bit exponent with bias 15, 2-bit mantissa.
 * Exponent field 0 holds subnormals m·2^-16; field 31 holds infinity (mantissa
 * 0) and NaN, so the largest finite magnitude is 1.75·2^15 = 57,344 (the
 * page's format table: 1·5·2 bits, 57,344). */
double kvdo_e5m2_decode(uint8_t code) {
    int sign = code >> 7;
    int e = (code >> 2) & 0x1F;
    int m = code & 0x3;
    double v;
    if (e == 0x1F) v = (m == 0) ? INFINITY : NAN;
    else if (e == 0) v = ldexp((double)m, -16);
    else v = ldexp(1.0 + m / 4.0, e - 15);
    return sign ? -v : v;
}

/* Nearest finite E5M2 code to y: enumeration of the 124 non-negative finite
 * codes, a tie goes to the even mantissa, magnitudes beyond 57,344 saturate. */
uint8_t kvdo_e5m2_encode(float y) {
    if (isnan(y)) return 0x7F;
    int neg = signbit(y) ? 1 : 0;
    double a = fabs((double)y);
    int best = 0;
    double best_d = INFINITY;
    for (int c = 0; c <= 0x7B; ++c) {
        double d = fabs(a - kvdo_e5m2_decode((uint8_t)c));
        if (d < best_d || (d == best_d && (c & 1) == 0)) {
            best = c;
            best_d = d;
        }
    }
    if (a > 57344.0) best = 0x7B;
    return (uint8_t)((neg << 7) | best);
}

void kvdo_e5m2_decode_array(const uint8_t* codes, int64_t n, double* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = kvdo_e5m2_decode(codes[i]);
}

void kvdo_e5m2_encode_array(const float* y, int64_t n, uint8_t* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = kvdo_e5m2_encode(y[i]);
}

/* Block precision codes of a mixed pool: 0 = BF16 values, 1 = E4M3 codes,
 * 2 = E5M2 codes, each 8-bit format with a per-(token, head) fp32 scale. */
#define KVDO_FMT_BF16 0
#define KVDO_FMT_E4M3 1
#define KVDO_FMT_E5M2 2

static double fmt_decode(int fmt, uint8_t code) {
    return fmt == KVDO_FMT_E5M2 ? kvdo_e5m2_decode(code) : kvdo_e4m3_decode(code);
}

/* A row in an 8-bit format: scale = absmax / (the format's largest value) in
 * fp32 (1 for an all-zero row), code_i = nearest code of the fp32 x_i/scale. */
void kvdo_quantize_row_fmt(const float* x, int d, int fmt, uint8_t* codes, float* scale_out) {
    const float top = fmt == KVDO_FMT_E5M2 ? 57344.0f : 448.0f;
    float amax = 0.0f;
    for (int i = 0; i < d; ++i) {
        float a = fabsf(x[i]);
        if (a > amax) amax = a;
    }
    float scale = (amax == 0.0f) ? 1.0f : amax / top;
    for (int i = 0; i < d; ++i) {
        float y = x[i] / scale;
        codes[i] = fmt == KVDO_FMT_E5M2 ? kvdo_e5m2_encode(y) : kvdo_e4m3_encode(y);
    }
    *scale_out = scale;
}

void kvdo_quantize_rows_fmt(const float* x, int64_t rows, int d, int fmt, uint8_t* codes, float* scales) {
    for (int64_t r = 0; r < rows; ++r) kvdo_quantize_row_fmt(x + r * d, d, fmt, codes + r * d, scales + r);
}

/* ----------------------------------------------------------- paged cache */

/* Write N new tokens into the pool.  Token n goes to slot slot_mapping[n] =
 * physical_block·block_size + offset (negative: skipped).  k_new, v_new are
 * [N][n_kv][d_h].  BF16 mode (fp8 == 0) stores the values; FP8 mode stores
 * per-(token, head) codes and scales for K and V separately. */
int kvdo_append(int n_kv, int d_h, int block_size, int64_t num_blocks, int fp8,
                const float* k_new, const float* v_new, const int64_t* slot_mapping, int64_t N,
                double* k_pool, double* v_pool,
                uint8_t* k_codes, uint8_t* v_codes, float* k_scales, float* v_scales) {
    for (int64_t n = 0; n < N; ++n) {
        int64_t slot = slot_mapping[n];
        if (slot < 0) continue;
        int64_t blk = slot / block_size;
        int64_t off = slot % block_size;
        if (blk >= num_blocks) return KVDO_ERR_INDEX;
        for (int h = 0; h < n_kv; ++h) {
            const float* ks = k_new + (n * n_kv + h) * d_h;
            const float* vs = v_new + (n * n_kv + h) * d_h;
            int64_t row = (blk * n_kv + h) * block_size + off;
            if (!fp8) {
                for (int i = 0; i < d_h; ++i) {
                    k_pool[row * d_h + i] = ks[i];
                    v_pool[row * d_h + i] = vs[i];
                }
            } else {
                kvdo_quantize_row(ks, d_h, k_codes + row * d_h, k_scales + row);
                kvdo_quantize_row(vs, d_h, v_codes + row * d_h, v_scales + row);
            }
        }
    }
    return KVDO_OK;
}

/* Append into a mixed-precision pool: block p holds its tokens in format
 * block_fmt[p] (BF16 values, or E4M3 / E5M2 codes with a row scale).  k_val,
 * v_val receive what attention reads (the value, or code value × scale), and
 * for 8-bit blocks the codes and scales are kept too.  Layout as kvdo_append. */
int kvdo_append_mixed(int n_kv, int d_h, int block_size, int64_t num_blocks, const uint8_t* block_fmt,
                      const float* k_new, const float* v_new, const int64_t* slot_mapping, int64_t N,
                      double* k_val, double* v_val, uint8_t* k_codes, uint8_t* v_codes, float* k_scales,
                      float* v_scales) {
    for (int64_t n = 0; n < N; ++n) {
        int64_t slot = slot_mapping[n];
        if (slot < 0) continue;
        int64_t blk = slot / block_size;
        int64_t off = slot % block_size;
        if (blk >= num_blocks) return KVDO_ERR_INDEX;
        int fmt = block_fmt[blk];
        for (int h = 0; h < n_kv; ++h) {
            const float* ks = k_new + (n * n_kv + h) * d_h;
            const float* vs = v_new + (n * n_kv + h) * d_h;
            int64_t row = (blk * n_kv + h) * block_size + off;
            if (fmt == KVDO_FMT_BF16) {
                for (int i = 0; i < d_h; ++i) {
                    k_val[row * d_h + i] = ks[i];
                    v_val[row * d_h + i] = vs[i];
                }
                continue;
            }
            kvdo_quantize_row_fmt(ks, d_h, fmt, k_codes + row * d_h, k_scales + row);
            kvdo_quantize_row_fmt(vs, d_h, fmt, v_codes + row * d_h, v_scales + row);
            for (int i = 0; i < d_h; ++i) {
                k_val[row * d_h + i] = fmt_decode(fmt, k_codes[row * d_h + i]) * (double)k_scales[row];
                v_val[row * d_h + i] = fmt_decode(fmt, v_codes[row * d_h + i]) * (double)v_scales[row];
            }
        }
    }
    return KVDO_OK;
}

/* ------------------------------------------------------------ low-bit KV */

/* Nearest IEEE half-precision value to x, ties to the even significand, with
 * magnitudes beyond the largest finite half (65,504) saturated to it: 10
 * fraction bits, exponent bias 15, subnormal spacing 2^-24.  Written from the
 * format definition (the result is returned as a double holding that value). */
double kvdo_round_half_sat(double x) {
    if (x == 0.0 || isnan(x)) return x;
    double a = fabs(x);
    int e = ilogb(a);               /* 2^e <= a < 2^(e+1) */
    if (e < -14) e = -14;           /* below the normal range: fixed spacing 2^-24 */
    double ulp = ldexp(1.0, e - 10);
    double r = rint(a / ulp) * ulp; /* a / ulp is exact: ulp is a power of two */
    if (r > 65504.0) r = 65504.0;
    return x < 0 ? -r : r;
}

void kvdo_round_half_sat_array(const double* x, int64_t n, double* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = kvdo_round_half_sat(x[i]);
}

/* Low-bit row quantisation with per-group scale and zero point (the group
 * layout is not on the pages; page "The KV Cache Is the New Memory Wall",
 * §4.2, §4.6, Tab. 7, names INT4 / 2-bit KV with group scales).  For each group
 * of `group` consecutive values of a (token, KV head) row, in single precision:
 *   mn, mx   = min and max of the group,
 *   scale    = half(fp32((mx - mn) / (2^bits - 1))), 1 if that rounds to 0,
 *   zero     = half(mn),
 *   code_i   = clamp(rint(fp32(fp32(x_i - zero) / scale)), 0, 2^bits - 1),
 * half() = the nearest half-precision value, saturating; rint ties to even.
 * The value read back is code·scale + zero.  codes [d], scales and zeros
 * [d / group] (values that are exact half-precision numbers). */
void kvdo_quantize_row_lowbit(const float* x, int d, int bits, int group, uint8_t* codes, float* scales,
                              float* zeros) {
    const int top = (1 << bits) - 1;
    for (int g0 = 0, gi = 0; g0 < d; g0 += group, ++gi) {
        float mn = x[g0], mx = x[g0];
        for (int i = g0 + 1; i < g0 + group; ++i) {
            if (x[i] < mn) mn = x[i];
            if (x[i] > mx) mx = x[i];
        }
        float span = mx - mn;
        float s = (float)kvdo_round_half_sat((double)(span / (float)top));
        if (s == 0.0f) s = 1.0f;
        float z = (float)kvdo_round_half_sat((double)mn);
        for (int i = g0; i < g0 + group; ++i) {
            float diff = x[i] - z;
            float y = diff / s;
            double r = rint((double)y);
            if (r < 0.0) r = 0.0;
            if (r > (double)top) r = (double)top;
            codes[i] = (uint8_t)r;
        }
        scales[gi] = s;
        zeros[gi] = z;
    }
}

void kvdo_quantize_rows_lowbit(const float* x, int64_t rows, int d, int bits, int group, uint8_t* codes,
                               float* scales, float* zeros) {
    const int ng = d / group;
    for (int64_t r = 0; r < rows; ++r)
        kvdo_quantize_row_lowbit(x + r * d, d, bits, group, codes + r * d, scales + r * ng, zeros + r * ng);
}

/* Append into a low-bit pool: every (token, KV head) row of K and of V is
 * quantised as above.  k_val, v_val [num_blocks][n_kv][block_size][d_h] receive
 * the values attention reads (code·scale + zero, fp64); codes likewise, and
 * scales / zeros [num_blocks][n_kv][block_size][d_h / group]. */
int kvdo_append_lowbit(int n_kv, int d_h, int block_size, int64_t num_blocks, int bits, int group,
                       const float* k_new, const float* v_new, const int64_t* slot_mapping, int64_t N,
                       double* k_val, double* v_val, uint8_t* k_codes, uint8_t* v_codes, float* k_scales,
                       float* k_zeros, float* v_scales, float* v_zeros) {
    const int ng = d_h / group;
    for (int64_t n = 0; n < N; ++n) {
        int64_t slot = slot_mapping[n];
        if (slot < 0) continue;
        int64_t blk = slot / block_size;
        int64_t off = slot % block_size;
        if (blk >= num_blocks) return KVDO_ERR_INDEX;
        for (int h = 0; h < n_kv; ++h) {
            int64_t row = (blk * n_kv + h) * block_size + off;
            kvdo_quantize_row_lowbit(k_new + (n * n_kv + h) * d_h, d_h, bits, group, k_codes + row * d_h,
                                     k_scales + row * ng, k_zeros + row * ng);
            kvdo_quantize_row_lowbit(v_new + (n * n_kv + h) * d_h, d_h, bits, group, v_codes + row * d_h,
                                     v_scales + row * ng, v_zeros + row * ng);
            for (int i = 0; i < d_h; ++i) {
                k_val[row * d_h + i] = k_codes[row * d_h + i] * (double)k_scales[row * ng + i / group] +
                                       (double)k_zeros[row * ng + i / group];
                v_val[row * d_h + i] = v_codes[row * d_h + i] * (double)v_scales[row * ng + i / group] +
                                       (double)v_zeros[row * ng + i / group];
            }
        }
    }
    return KVDO_OK;
}

/* ------------------------------------------------------- angle-domain keys */

/* One key row in the angle domain (page "기술 요약: Spherical KV", §2.1, Angle-Domain
 * Attention): the key k splits into a radius r = ||k|| and a direction; the cache keeps a
 * quantised radius r̃ and a code of the direction, and a logit is ||q||·r̃·f_b(c_q, c_k), f_b
 * the cosine of two direction codes.  The page defines neither the code nor f_b; this oracle
 * reads them as:
 *   c = the E4M3 codes of the row at its absmax scale (kvdo_quantize_row: they depend on the
 *       direction only, not on ||k||), d = their values (kvdo_e4m3_decode);
 *   r̃ = the nearest half-precision value of ||k|| (saturating);
 *   f_b(c_q, c_k) = <d_q, d_k> / (||d_q||·||d_k||).
 * So the key attention sees is w·d with w = fp32(r̃ / ||d||), computed in fp64 (w = 0 for a
 * zero row); codes [d], *w_out, *r_out (r̃). */
void kvdo_angle_key_row(const float* x, int d, uint8_t* codes, float* w_out, float* r_out) {
    float scale;
    kvdo_quantize_row(x, d, codes, &scale);
    double r2 = 0.0, d2 = 0.0;
    for (int i = 0; i < d; ++i) {
        double c = kvdo_e4m3_decode(codes[i]);
        r2 += (double)x[i] * (double)x[i];
        d2 += c * c;
    }
    double rh = kvdo_round_half_sat(sqrt(r2));
    *r_out = (float)rh;
    *w_out = d2 > 0.0 ? (float)(rh / sqrt(d2)) : 0.0f;
}

void kvdo_angle_key_rows(const float* x, int64_t rows, int d, uint8_t* codes, float* w, float* r) {
    for (int64_t i = 0; i < rows; ++i) kvdo_angle_key_row(x + i * d, d, codes + i * d, w + i, r + i);
}

/* The query side of the same cosine: each row q becomes (||q|| / ||d_q||)·d_q, d_q the values of
 * its E4M3 codes at its absmax scale (0 for a zero row), so that <q', w·d_k> = ||q||·r̃·f_b. */
void kvdo_angle_query(const float* q, int64_t rows, int d, double* out) {
    uint8_t* codes = (uint8_t*)malloc((size_t)d);
    for (int64_t i = 0; i < rows; ++i) {
        float scale;
        const float* x = q + i * d;
        kvdo_quantize_row(x, d, codes, &scale);
        double q2 = 0.0, d2 = 0.0;
        for (int j = 0; j < d; ++j) {
            double c = kvdo_e4m3_decode(codes[j]);
            q2 += (double)x[j] * (double)x[j];
            d2 += c * c;
        }
        double f = d2 > 0.0 ? sqrt(q2) / sqrt(d2) : 0.0;
        for (int j = 0; j < d; ++j) out[i * d + j] = f * kvdo_e4m3_decode(codes[j]);
    }
    free(codes);
}

/* Append into an angle-domain pool: K rows as kvdo_angle_key_row (codes and the factor w in
 * k_scales), V rows FP8 as kvdo_quantize_row (codes and scale).  Layout as kvdo_append. */
int kvdo_append_angle(int n_kv, int d_h, int block_size, int64_t num_blocks, const float* k_new,
                      const float* v_new, const int64_t* slot_mapping, int64_t N, uint8_t* k_codes,
                      uint8_t* v_codes, float* k_scales, float* v_scales, float* k_radius) {
    for (int64_t n = 0; n < N; ++n) {
        int64_t slot = slot_mapping[n];
        if (slot < 0) continue;
        int64_t blk = slot / block_size;
        int64_t off = slot % block_size;
        if (blk >= num_blocks) return KVDO_ERR_INDEX;
        for (int h = 0; h < n_kv; ++h) {
            int64_t row = (blk * n_kv + h) * block_size + off;
            kvdo_angle_key_row(k_new + (n * n_kv + h) * d_h, d_h, k_codes + row * d_h, k_scales + row,
                               k_radius + row);
            kvdo_quantize_row(v_new + (n * n_kv + h) * d_h, d_h, v_codes + row * d_h, v_scales + row);
        }
    }
    return KVDO_OK;
}

/* Read back an FP8 pool as values: code value times its row's scale. */
void kvdo_dequant_pool(const uint8_t* codes, const float* scales, int64_t rows, int d_h, double* out) {
    for (int64_t r = 0; r < rows; ++r)
        for (int i = 0; i < d_h; ++i)
            out[r * d_h + i] = kvdo_e4m3_decode(codes[r * d_h + i]) * (double)scales[r];
}

/* ------------------------------------------------------ decode attention */

/* One decode step of GQA attention for B requests over the paged pool.
 *
 * q          [B][n_q][d_h]
 * k_pool, v_pool  [num_blocks][n_kv][block_size][d_h] values
 * block_table [B][max_blocks]: logical block j of request b -> physical block
 * seq_lens   [B]: attended positions 0 .. seq_lens[b]-1
 * retain     [num_blocks] or NULL: bit o of retain[p] clear = slot o of block
 *            p is evicted and takes no part (its logit is -inf)
 * Query head h reads KV head h / (n_q / n_kv) (consecutive groups).
 *
 * Outputs: out [B][n_q][d_h] = Σ_t α_t V_t; lse [B][n_q] = log Σ_t exp(l_t);
 * alpha (optional) [B][n_q][alpha_stride] = softmax weights per position;
 * logits (optional) [B][n_q][alpha_stride] = l_t (-inf where evicted).
 */
int kvdo_decode(int n_q, int n_kv, int d_h, int block_size, int64_t num_blocks,
                const double* q, const double* k_pool, const double* v_pool,
                const int32_t* block_table, int max_blocks, const int32_t* seq_lens, int B,
                const uint16_t* retain, double softmax_scale,
                double* out, double* lse, double* alpha, double* logits, int64_t alpha_stride) {
    int g = n_q / n_kv;
    int status = KVDO_OK;
    for (int b = 0; b < B; ++b) {
        int ctx = seq_lens[b];
        if (ctx < 0 || ctx > max_blocks * block_size) return KVDO_ERR_INDEX;
        double* l = (double*)malloc(sizeof(double) * (size_t)(ctx > 0 ? ctx : 1));
        for (int h = 0; h < n_q; ++h) {
            int kvh = h / g;
            const double* qh = q + ((int64_t)b * n_q + h) * d_h;
            double m = -INFINITY;
            /* logits through the block table */
            for (int t = 0; t < ctx; ++t) {
                int32_t p = block_table[(int64_t)b * max_blocks + t / block_size];
                int o = t % block_size;
                if (p < 0 || p >= num_blocks) { free(l); return KVDO_ERR_INDEX; }
                if (retain && !((retain[p] >> o) & 1u)) { l[t] = -INFINITY; continue; }
                const double* kt = k_pool + (((int64_t)p * n_kv + kvh) * block_size + o) * d_h;
                double dot = 0.0;
                for (int i = 0; i < d_h; ++i) dot += qh[i] * kt[i];
                l[t] = softmax_scale * dot;
                if (l[t] > m) m = l[t];
            }
            double* oh = out + ((int64_t)b * n_q + h) * d_h;
            for (int i = 0; i < d_h; ++i) oh[i] = 0.0;
            if (logits)
                for (int t = 0; t < ctx; ++t) logits[((int64_t)b * n_q + h) * alpha_stride + t] = l[t];
            if (m == -INFINITY) {      /* nothing to attend to */
                lse[(int64_t)b * n_q + h] = -INFINITY;
                if (alpha)
                    for (int t = 0; t < ctx; ++t) alpha[((int64_t)b * n_q + h) * alpha_stride + t] = 0.0;
                status = KVDO_ERR_EMPTY;
                continue;
            }
            /* softmax */
            double sum = 0.0;
            for (int t = 0; t < ctx; ++t) sum += exp(l[t] - m);
            lse[(int64_t)b * n_q + h] = m + log(sum);
            for (int t = 0; t < ctx; ++t) {
                double a = exp(l[t] - m) / sum;
                if (alpha) alpha[((int64_t)b * n_q + h) * alpha_stride + t] = a;
                if (a == 0.0) continue;
                int32_t p = block_table[(int64_t)b * max_blocks + t / block_size];
                int o = t % block_size;
                const double* vt = v_pool + (((int64_t)p * n_kv + kvh) * block_size + o) * d_h;
                for (int i = 0; i < d_h; ++i) oh[i] += a * vt[i];
            }
        }
        free(l);
    }
    return status;
}

/* ------------------------------------------------------- importance score */

/* One decode step's update of the cumulative importance score:
 * s[b][i] += (1/L) Σ_ℓ (1/H) Σ_h alpha[ℓ][b][h][i] for i < seq_lens[b],
 * with alpha [L][B][H][stride] and s [B][stride]. */
void kvdo_score_update(const double* alpha, int L, int B, int H, const int32_t* seq_lens,
                       int64_t stride, double* s) {
    for (int b = 0; b < B; ++b) {
        for (int i = 0; i < seq_lens[b]; ++i) {
            double over_layers = 0.0;
            for (int ly = 0; ly < L; ++ly) {
                double over_heads = 0.0;
                for (int h = 0; h < H; ++h)
                    over_heads += alpha[(((int64_t)ly * B + b) * H + h) * stride + i];
                over_layers += over_heads / H;
            }
            s[(int64_t)b * stride + i] += over_layers / L;
        }
    }
}

/* ------------------------------------------------------------- tier plan */

/* Tier assignment every Δ steps: page "기술 요약: 모든 사고가 HBM 을 필요로 하는 것은
 * 아님", section "1. 4 단계 분류" (protected tokens — prompt, sinks, recent window — stay
 * in HBM; mid-importance tokens go to host memory, T1) and section "4. 시스템 구현"
 * (reassignment every Δ = 64 steps), at the granularity of a 16-token block.
 *
 * For request b of length len, block j covers positions [bs·j, min(bs·j+bs, len)).
 *   importance[b][j] = the fp32 sum of scores[b][pos] over those positions, added in
 *     position order (positions at or past `stride` count 0);
 *   block j is protected when one of its positions is < protect_prompt or
 *     ≥ len − protect_recent;
 *   the unprotected blocks, sorted by (importance, j) ascending, give their first t1
 *     entries tier 1 and the rest tier 0; protected blocks get 0; j ≥ ⌈len/bs⌉ gets −1.
 * A length outside [1, max_blocks·bs] counts as 0 blocks.  The sum is single precision
 * because the tier is an integer decided by comparing sums: both sides of a parity test
 * take that decision in the same precision. */
typedef struct {
    float imp;
    int j;
} kvdo_block_key;

static int kvdo_block_key_cmp(const void* a, const void* b) {
    const kvdo_block_key* x = (const kvdo_block_key*)a;
    const kvdo_block_key* y = (const kvdo_block_key*)b;
    if (x->imp < y->imp) return -1;
    if (x->imp > y->imp) return 1;
    return (x->j > y->j) - (x->j < y->j);
}

void kvdo_tier_plan(const float* scores, int64_t stride, const int32_t* seq_lens, int B, int max_blocks,
                    int block_size, int protect_prompt, int protect_recent, int t1, float* importance,
                    int8_t* tier) {
    kvdo_block_key* keys = (kvdo_block_key*)malloc(sizeof(kvdo_block_key) * (size_t)(max_blocks > 0 ? max_blocks : 1));
    for (int b = 0; b < B; ++b) {
        const int64_t len = seq_lens[b];
        int64_t nb = (len + block_size - 1) / block_size;
        if (len < 1 || nb > max_blocks) nb = 0;
        float* imp = importance + (int64_t)b * max_blocks;
        int8_t* tr = tier + (int64_t)b * max_blocks;
        int n_free = 0;
        for (int j = 0; j < max_blocks; ++j) {
            imp[j] = 0.0f;
            tr[j] = -1;
            if (j >= nb) continue;
            int prot = 0;
            for (int64_t pos = (int64_t)j * block_size; pos < (int64_t)(j + 1) * block_size && pos < len; ++pos) {
                if (pos < stride) imp[j] += scores[(int64_t)b * stride + pos];
                if (pos < protect_prompt || pos >= len - protect_recent) prot = 1;
            }
            tr[j] = 0;
            if (!prot) {
                keys[n_free].imp = imp[j];
                keys[n_free].j = j;
                ++n_free;
            }
        }
        qsort(keys, (size_t)n_free, sizeof(kvdo_block_key), kvdo_block_key_cmp);
        for (int r = 0; r < n_free && r < t1; ++r) tr[keys[r].j] = 1;
    }
    free(keys);
}
