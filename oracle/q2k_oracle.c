/*
 * CPU oracle for the Q2_K decode projections.  TEST INFRASTRUCTURE ONLY: the
 * tests, the smoke check and the bench's CPU-baseline leg call it; the CUDA
 * library never does, and the two share no code.
 *
 * Plain, slow, obviously correct C.  Floating point is fp64 unless the
 * method fixes a precision (the q8_1 encoding decides integers in fp32, and
 * the dequantised rows are bf16 by definition).
 *
 * Sources (the metrale docs pages):
 *  - engram_v41.rs, `ENGRAM_ROW_BYTES` and the `wkv_q2k` field doc: one Q2_K
 *    super-block is 84 bytes and holds 256 weights; a weight matrix is
 *    `[out, in/256]` blocks, row-major, as GGUF ships it; `y = x W^T`.
 *  - engram_v41.rs, `rows_from_q2k`: rows are dequantised to bf16, one block
 *    per 256-wide row, in `[token][col]` order.
 *  - attn_v41/decode.rs, `q_kv_projections`: one q8_1 quantisation feeds
 *    both the `wq_a` and `wkv` projections (m <= 8).
 *  - moe_v41/init.rs, `MoeV41::new`: gate and up run as one expert batch,
 *    SwiGLU is fused with the q8_1 requantisation of `h`, and the expert
 *    outputs are accumulated with the route weights.
 *
 * Readings taken where the pages are silent (each listed in the design
 * notes):
 *  - Q2_K byte order: scales[16] | qs[64] | d (fp16 LE) | dmin (fp16 LE).
 *    Weight p in [0,256) lies in sub-block j = p/16; scales[j] low nibble is
 *    the scale, high nibble the min; its 2-bit code is bits
 *    2*((p%128)/32) .. +1 of qs[32*(p/128) + p%32];
 *    w_p = d*(scales[j]&15)*q_p - dmin*(scales[j]>>4).
 *  - q8_1 block (36 bytes, 32 values): fp16 d, fp16 s, int8 q[32];
 *    d32 = amax/127 (fp32 divide), q = round-half-away(x/d32) (fp32 divide,
 *    0 when amax == 0), d = fp16_rn(d32), s = fp16_rn(f32(d) * sum(q)).
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <string.h>

#define Q2K_BYTES 84
#define Q2K_WEIGHTS 256
#define Q8_1_BYTES 36
#define Q8_1_VALUES 32

/* ---- scalar formats ------------------------------------------------------ */

/* IEEE binary16 bits -> exact double. */
double oracle_fp16_to_double(uint16_t h)
{
    int sign = h >> 15;
    int e = (h >> 10) & 31;
    int f = h & 1023;
    double v;
    if (e == 0)
        v = ldexp((double)f, -24);
    else if (e == 31)
        v = f ? NAN : INFINITY;
    else
        v = ldexp((double)(f + 1024), e - 25);
    return sign ? -v : v;
}

/* bf16 bits -> exact double. */
double oracle_bf16_to_double(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return (double)f;
}

/* Finite float -> binary16 bits, round to nearest, ties to even. */
uint16_t oracle_f32_to_fp16(float x)
{
    uint16_t sign = signbit(x) ? 0x8000 : 0;
    double a = fabs((double)x);
    if (isnan(x))
        return 0x7E00;
    if (a >= 65520.0) /* halfway between 65504 and 2^16 rounds to even -> inf */
        return sign | 0x7C00;
    if (a < ldexp(1.0, -14)) {
        /* subnormal range: quantum 2^-24; n == 1024 is the smallest normal */
        double n = nearbyint(a * ldexp(1.0, 24));
        return sign | (uint16_t)n;
    }
    int ex;
    frexp(a, &ex); /* a = fr * 2^ex, fr in [0.5, 1) */
    int e = ex - 1; /* a in [2^e, 2^(e+1)) */
    double n = nearbyint(ldexp(a, 10 - e)); /* 11-bit significand */
    if (n == 2048.0) {
        n = 1024.0;
        e += 1;
    }
    if (e + 15 >= 31)
        return sign | 0x7C00;
    return sign | (uint16_t)(((e + 15) << 10) | ((int)n - 1024));
}

/* Finite float -> bf16 bits, round to nearest, ties to even. */
uint16_t oracle_f32_to_bf16(float x)
{
    uint32_t u;
    memcpy(&u, &x, 4);
    if (isnan(x))
        return (uint16_t)((u >> 16) | 0x40);
    uint16_t sign = (uint16_t)((u >> 16) & 0x8000);
    double a = fabs((double)x);
    if (a == 0.0)
        return sign;
    int ex;
    frexp(a, &ex);
    int e = ex - 1;
    if (e < -126)
        e = -126; /* bf16 subnormals share fp32's exponent floor */
    double q = ldexp(1.0, e - 7); /* 8-bit significand quantum */
    double n = nearbyint(a / q);
    double r = n * q;
    if (r >= ldexp(1.0, 128))
        return sign | 0x7F80;
    float rf = (float)r; /* exact: r is a bf16 value */
    uint32_t ru;
    memcpy(&ru, &rf, 4);
    return sign | (uint16_t)(ru >> 16);
}

/* Round hi+lo (an exact value split as a double-double, |lo| <= ulp(hi)/2)
 * to the nearest float, ties to even, without double rounding. */
static float round_dd_to_f32(double hi, double lo)
{
    float f = (float)hi;
    double back = (double)f;
    if (back == hi || lo == 0.0)
        return f;
    /* The only double-rounding hazard: hi sits exactly half-way between two
     * floats; then the sign of lo decides. */
    float up = nextafterf(f, INFINITY), dn = nextafterf(f, -INFINITY);
    double mid_up = ((double)f + (double)up) * 0.5;
    double mid_dn = ((double)f + (double)dn) * 0.5;
    if (hi == mid_up && lo < 0)
        return f;
    if (hi == mid_up && lo > 0)
        return up;
    if (hi == mid_dn && lo > 0)
        return f;
    if (hi == mid_dn && lo < 0)
        return dn;
    return f;
}

/* ---- Q2_K ----------------------------------------------------------------- */

static uint16_t rd16(const uint8_t* p) { return (uint16_t)(p[0] | (p[1] << 8)); }

/* 2-bit code of weight p in a block. */
static int q2k_code(const uint8_t* blk, int p)
{
    const uint8_t* qs = blk + 16;
    int byte = qs[32 * (p / 128) + (p % 32)];
    int shift = 2 * ((p % 128) / 32);
    return (byte >> shift) & 3;
}

/* Exact decoded weights of one 84-byte block (fp64; exact for every fp16
 * d/dmin whose products span at most 53 bits, which holds for any block
 * whose d and dmin lie within 2^33 of each other). */
void oracle_q2k_decode_block(const uint8_t* blk, double* w)
{
    double d = oracle_fp16_to_double(rd16(blk + 80));
    double dmin = oracle_fp16_to_double(rd16(blk + 82));
    for (int p = 0; p < Q2K_WEIGHTS; ++p) {
        int sc = blk[p / 16];
        w[p] = d * (double)(sc & 15) * (double)q2k_code(blk, p) - dmin * (double)(sc >> 4);
    }
}

/* bf16 bits of every weight of one block: the exact value rounded once to
 * fp32 and then to bf16. */
void oracle_q2k_decode_block_bf16(const uint8_t* blk, uint16_t* out)
{
    double d = oracle_fp16_to_double(rd16(blk + 80));
    double dmin = oracle_fp16_to_double(rd16(blk + 82));
    for (int p = 0; p < Q2K_WEIGHTS; ++p) {
        int sc = blk[p / 16];
        double a = d * (double)(sc & 15) * (double)q2k_code(blk, p); /* exact */
        double b = dmin * (double)(sc >> 4);                          /* exact */
        double s = a - b;
        double bb = s - a; /* TwoSum of a and -b */
        double err = (a - (s - bb)) + (-b - bb);
        out[p] = oracle_f32_to_bf16(round_dd_to_f32(s, err));
    }
}

/* Gather + dequantise: out[r, :] = bf16(decode(table row ids[r])), each row
 * K/256 blocks.  ids == NULL means rows 0..n_rows-1.  An id outside
 * [0, n_table_rows) yields a zero row; returns how many ids were bad. */
int64_t oracle_q2k_dequant_rows(const uint8_t* table, int64_t n_table_rows, int64_t K,
                                const int32_t* ids, int64_t n_rows, uint16_t* out)
{
    int64_t nb = K / Q2K_WEIGHTS, bad = 0;
    for (int64_t r = 0; r < n_rows; ++r) {
        int64_t src = ids ? (int64_t)ids[r] : r;
        uint16_t* o = out + r * K;
        if (src < 0 || src >= n_table_rows) {
            memset(o, 0, (size_t)K * 2);
            ++bad;
            continue;
        }
        for (int64_t b = 0; b < nb; ++b)
            oracle_q2k_decode_block_bf16(table + (src * nb + b) * Q2K_BYTES, o + b * Q2K_WEIGHTS);
    }
    return bad;
}

/* Exact decoded matrix [N, K] (fp64). */
void oracle_q2k_decode_matrix(const uint8_t* W, int64_t N, int64_t K, double* out)
{
    int64_t nb = K / Q2K_WEIGHTS;
    for (int64_t n = 0; n < N; ++n)
        for (int64_t b = 0; b < nb; ++b)
            oracle_q2k_decode_block(W + (n * nb + b) * Q2K_BYTES, out + n * K + b * Q2K_WEIGHTS);
}

/* y[t, n] = sum_k w[n, k] * x[t, k]; W Q2_K [N, K], x fp64 [m, K],
 * y fp64 [m, N].  Naive, fp64 accumulation in k order. */
void oracle_q2k_matvec(const uint8_t* W, int64_t N, int64_t K, const double* x, int64_t m,
                       double* y)
{
    int64_t nb = K / Q2K_WEIGHTS;
    double w[Q2K_WEIGHTS];
    for (int64_t t = 0; t < m; ++t)
        for (int64_t n = 0; n < N; ++n)
            y[t * N + n] = 0.0;
    for (int64_t n = 0; n < N; ++n) {
        for (int64_t b = 0; b < nb; ++b) {
            oracle_q2k_decode_block(W + (n * nb + b) * Q2K_BYTES, w);
            for (int64_t t = 0; t < m; ++t) {
                double acc = 0.0;
                const double* xr = x + t * K + b * Q2K_WEIGHTS;
                for (int p = 0; p < Q2K_WEIGHTS; ++p)
                    acc += w[p] * xr[p];
                y[t * N + n] += acc;
            }
        }
    }
}

/* ---- Q3_K ------------------------------------------------------------------ */
/* moe_v41/init.rs, `MoeV41::new`, names Q3_K twins of the single-matrix and
 * experts MMVQ kernels; the pages give no Q3_K layout.  Reading: GGUF's
 * Q3_K, 110 bytes per 256 weights:
 *   hmask[32] | qs[64] | scales[12] | d (fp16 LE).
 * Weight p lies in sub-block j = p/16 with a signed 6-bit scale (stored + 32):
 * low nibble in scales[j] (j < 8) or the high nibble of scales[j-8]
 * (j >= 8); the top two bits at bit 2*(j/4) of scales[8 + j%4].  Its code is
 * the 2-bit field laid out as in Q2_K (at byte 32 of the block) minus 4,
 * unless bit p/32 of hmask[p%32] is set.  w_p = d * scale_j * code_p. */
#define Q3K_BYTES 110

static int q3k_scale(const uint8_t* sc, int j)
{
    int low = j < 8 ? (sc[j] & 15) : (sc[j - 8] >> 4);
    int high = (sc[8 + j % 4] >> (2 * (j / 4))) & 3;
    return (low | (high << 4)) - 32;
}

static int q3k_code(const uint8_t* blk, int p)
{
    const uint8_t* hmask = blk;
    const uint8_t* qs = blk + 32;
    int lo = (qs[32 * (p / 128) + (p % 32)] >> (2 * ((p % 128) / 32))) & 3;
    int hi = (hmask[p % 32] >> (p / 32)) & 1;
    return hi ? lo : lo - 4;
}

/* Exact decoded weights of one 110-byte block (d * integer in [-128, 128]). */
void oracle_q3k_decode_block(const uint8_t* blk, double* w)
{
    double d = oracle_fp16_to_double(rd16(blk + 108));
    for (int p = 0; p < Q2K_WEIGHTS; ++p)
        w[p] = d * (double)q3k_scale(blk + 96, p / 16) * (double)q3k_code(blk, p);
}

/* Exact decoded matrix [N, K] (fp64). */
void oracle_q3k_decode_matrix(const uint8_t* W, int64_t N, int64_t K, double* out)
{
    int64_t nb = K / Q2K_WEIGHTS;
    for (int64_t n = 0; n < N; ++n)
        for (int64_t b = 0; b < nb; ++b)
            oracle_q3k_decode_block(W + (n * nb + b) * Q3K_BYTES, out + n * K + b * Q2K_WEIGHTS);
}

/* y[t, n] = sum_k w[n, k] * x[t, k] for a Q3_K W [N, K]; fp64, k order. */
void oracle_q3k_matvec(const uint8_t* W, int64_t N, int64_t K, const double* x, int64_t m,
                       double* y)
{
    int64_t nb = K / Q2K_WEIGHTS;
    double w[Q2K_WEIGHTS];
    for (int64_t t = 0; t < m; ++t)
        for (int64_t n = 0; n < N; ++n)
            y[t * N + n] = 0.0;
    for (int64_t n = 0; n < N; ++n) {
        for (int64_t b = 0; b < nb; ++b) {
            oracle_q3k_decode_block(W + (n * nb + b) * Q3K_BYTES, w);
            for (int64_t t = 0; t < m; ++t) {
                double acc = 0.0;
                const double* xr = x + t * K + b * Q2K_WEIGHTS;
                for (int p = 0; p < Q2K_WEIGHTS; ++p)
                    acc += w[p] * xr[p];
                y[t * N + n] += acc;
            }
        }
    }
}

/* ---- q8_1 ----------------------------------------------------------------- */

/* bf16 x [m, K] with row stride ldx (elements) -> q8_1 rows, K/32 blocks of
 * 36 bytes per row, rows contiguous. */
void oracle_q8_1_quantize_rows(const uint16_t* x, int64_t m, int64_t K, int64_t ldx, uint8_t* out)
{
    int64_t nblk = K / Q8_1_VALUES;
    for (int64_t t = 0; t < m; ++t) {
        for (int64_t b = 0; b < nblk; ++b) {
            float v[Q8_1_VALUES];
            float amax = 0.0f;
            for (int i = 0; i < Q8_1_VALUES; ++i) {
                v[i] = (float)oracle_bf16_to_double(x[t * ldx + b * Q8_1_VALUES + i]);
                float a = fabsf(v[i]);
                if (a > amax)
                    amax = a;
            }
            volatile float d32 = amax / 127.0f; /* IEEE fp32 divide */
            int8_t q[Q8_1_VALUES];
            int sumq = 0;
            for (int i = 0; i < Q8_1_VALUES; ++i) {
                int qi = 0;
                if (amax != 0.0f) {
                    volatile float r = v[i] / d32; /* IEEE fp32 divide */
                    qi = (int)roundf(r);           /* half away from zero */
                }
                q[i] = (int8_t)qi;
                sumq += qi;
            }
            uint16_t dh = oracle_f32_to_fp16(d32);
            float df = (float)oracle_fp16_to_double(dh);
            volatile float sf = df * (float)sumq; /* fp32 multiply */
            uint16_t sh = oracle_f32_to_fp16(sf);
            uint8_t* o = out + (t * nblk + b) * Q8_1_BYTES;
            o[0] = (uint8_t)(dh & 0xFF);
            o[1] = (uint8_t)(dh >> 8);
            o[2] = (uint8_t)(sh & 0xFF);
            o[3] = (uint8_t)(sh >> 8);
            memcpy(o + 4, q, Q8_1_VALUES);
        }
    }
}

/* q8_1 rows -> the values they stand for, f32(d) * q, exact in fp64. */
void oracle_q8_1_dequant_rows(const uint8_t* xq, int64_t m, int64_t K, double* x)
{
    int64_t nblk = K / Q8_1_VALUES;
    for (int64_t t = 0; t < m; ++t)
        for (int64_t b = 0; b < nblk; ++b) {
            const uint8_t* blk = xq + (t * nblk + b) * Q8_1_BYTES;
            double d = oracle_fp16_to_double(rd16(blk));
            for (int i = 0; i < Q8_1_VALUES; ++i)
                x[t * K + b * Q8_1_VALUES + i] = d * (double)(int8_t)blk[4 + i];
        }
}

/* ---- dense and elementwise ------------------------------------------------ */

/* y[t, n] = sum_k x[t, k] * W[n, k], bf16 inputs, fp64 accumulation. */
void oracle_dense_gemm_bf16(const uint16_t* x, int64_t m, int64_t K, int64_t ldx,
                            const uint16_t* W, int64_t N, double* y)
{
    for (int64_t t = 0; t < m; ++t)
        for (int64_t n = 0; n < N; ++n) {
            double acc = 0.0;
            for (int64_t k = 0; k < K; ++k)
                acc += oracle_bf16_to_double(x[t * ldx + k]) * oracle_bf16_to_double(W[n * K + k]);
            y[t * N + n] = acc;
        }
}

/* silu(z) = z / (1 + e^-z), fp64. */
double oracle_silu(double z) { return z / (1.0 + exp(-z)); }

/* h[i] = silu(g[i]) * u[i] over n values, fp64. */
void oracle_swiglu(const double* g, const double* u, int64_t n, double* h)
{
    for (int64_t i = 0; i < n; ++i)
        h[i] = oracle_silu(g[i]) * u[i];
}

/* y[n] = sum_e w[e] * v[e, n] over E rows of length N, in e order, fp64. */
void oracle_weighted_sum(const double* v, const float* w, int64_t E, int64_t N, double* y)
{
    for (int64_t n = 0; n < N; ++n) {
        double acc = 0.0;
        for (int64_t e = 0; e < E; ++e)
            acc += (double)w[e] * v[e * N + n];
        y[n] = acc;
    }
}

/* fp64 values -> bf16 bits (fp64 -> fp32 -> bf16, each round to nearest). */
void oracle_round_bf16(const double* v, int64_t n, uint16_t* out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = oracle_f32_to_bf16((float)v[i]);
}

/* ---- engram n-gram hash ------------------------------------------------
 * engram_v41.rs, `EngramHasher::hash`: the input tokens are first mapped
 * through token_map into the sequence cache at start_pos..; then for every
 * position, the current token and the max_ngram-1 before it (a token before
 * the sequence start, or any token at or past an unmapped one (-1), reads as
 * pad_id) are combined per layer by wrapping i64 products and xor, and each
 * n-gram length i = 1..max_ngram-1 gives n_heads row ids:
 *   rolling_i = (t_0*mult_0) ^ ... ^ (t_i*mult_i)
 *   out[s][layer][(i-1)*n_heads + h] = rem_euclid(rolling_i, prime[layer][i-1][h])
 *                                       + offset[layer][(i-1)*n_heads + h]
 * Returns 0, -1 for a token id outside token_map (the cache entries before
 * it are written, as on the page), -2 when the positions pass max_seq. */
static int64_t wrapping_mul_i64(int64_t a, int64_t b) { return (int64_t)((uint64_t)a * (uint64_t)b); }

static int64_t rem_euclid_i64(int64_t a, int64_t p)
{
    int64_t r = a % p;
    return r < 0 ? r + p : r;
}

int oracle_engram_hash(const int64_t* token_map, int64_t vocab, int64_t* cache, int64_t max_seq,
                       const uint32_t* input_ids, int64_t seqlen, int64_t start_pos, int max_ngram,
                       int n_layers, int n_heads, const int64_t* multipliers, const int64_t* primes,
                       const int64_t* offsets, int64_t pad_id, int64_t* out)
{
    if (start_pos + seqlen > max_seq)
        return -2;
    for (int64_t s = 0; s < seqlen; ++s) {
        if ((int64_t)input_ids[s] >= vocab)
            return -1;
        cache[start_pos + s] = token_map[input_ids[s]];
    }
    const int cols = (max_ngram - 1) * n_heads;
    int64_t tokens[64];
    if (max_ngram > 64)
        return -2;
    for (int64_t s = 0; s < seqlen; ++s) {
        const int64_t pos = start_pos + s;
        int blocked = 0;
        for (int shift = 0; shift < max_ngram; ++shift) {
            const int64_t src = cache[pos >= shift ? pos - shift : 0];
            blocked = blocked || pos < shift || src == -1;
            tokens[shift] = blocked ? pad_id : src;
        }
        for (int li = 0; li < n_layers; ++li) {
            const int64_t* mults = multipliers + (int64_t)li * max_ngram;
            int64_t rolling = wrapping_mul_i64(tokens[0], mults[0]);
            for (int i = 1; i < max_ngram; ++i) {
                rolling ^= wrapping_mul_i64(tokens[i], mults[i]);
                for (int h = 0; h < n_heads; ++h) {
                    const int col = (i - 1) * n_heads + h;
                    const int64_t prime = primes[((int64_t)li * (max_ngram - 1) + (i - 1)) * n_heads + h];
                    out[(s * n_layers + li) * cols + col] =
                        rem_euclid_i64(rolling, prime) + offsets[(int64_t)li * cols + col];
                }
            }
        }
    }
    return 0;
}

/* ---- engram gate ---------------------------------------------------------
 * engram_v41.rs, module doc, step 4, and engram_v41/apply.rs, `apply` (the
 * `gate_k` launch over [tokens, hc] with streams, kv, qk, dim, hc, eps): a
 * normalised dot of each stream against its key, a signed-sqrt sigmoid, and
 * h += gate * value, in place on the fp32 streams [T, hc, dim].
 * Readings (the pages give the words above and the arguments only):
 *  - kv row t is [key_0 | ... | key_{hc-1} | value], dim values each: one key
 *    per stream plus one shared value (engram_v41.rs module doc, "one key per
 *    hyper-connection stream plus one shared value"), keys first;
 *  - kv is the projection's output held as bf16 (the page's `kv` buffer is
 *    bf16): every kv value is rounded to bf16 (fp32 RN, then bf16 RN) first;
 *  - "normalised dot": the stream and the key are RMS-normalised with eps,
 *    rms(z) = sqrt(mean(z^2) + eps), weighted by q_weight and k_weight (only
 *    their product qk = q_weight * k_weight enters), and the dot is scaled by
 *    1/sqrt(dim): s = sum_i qk_i h_i k_i / (rms(h) rms(k) sqrt(dim));
 *  - "signed-sqrt sigmoid": g = 1 / (1 + exp(-sign(s) sqrt(|s|)));
 *  - h_i += g * v_i for every i.
 * fp64 throughout (the inputs are fp32 values). */
void oracle_engram_gate(const float* streams, const float* kv, int64_t ld_kv, const float* qk, int64_t tokens,
                        int64_t hc, int64_t dim, float eps, double* out, double* gates)
{
    for (int64_t t = 0; t < tokens; ++t) {
        const float* v32 = kv + t * ld_kv + hc * dim;
        for (int64_t c = 0; c < hc; ++c) {
            const float* h = streams + (t * hc + c) * dim;
            const float* k32 = kv + t * ld_kv + c * dim;
            const float* q = qk + c * dim;
            double shh = 0.0, skk = 0.0, shk = 0.0;
            for (int64_t i = 0; i < dim; ++i) {
                const double hv = h[i];
                const double kk = oracle_bf16_to_double(oracle_f32_to_bf16(k32[i]));
                shh += hv * hv;
                skk += kk * kk;
                shk += (double)q[i] * hv * kk;
            }
            const double rh = sqrt(shh / (double)dim + (double)eps);
            const double rk = sqrt(skk / (double)dim + (double)eps);
            const double s = shk / (rh * rk * sqrt((double)dim));
            const double ss = s < 0.0 ? -sqrt(-s) : sqrt(s);
            const double g = 1.0 / (1.0 + exp(-ss));
            if (gates)
                gates[t * hc + c] = g;
            double* o = out + (t * hc + c) * dim;
            for (int64_t i = 0; i < dim; ++i)
                o[i] = (double)h[i] + g * oracle_bf16_to_double(oracle_f32_to_bf16(v32[i]));
        }
    }
}

int oracle_block_bytes(void) { return Q2K_BYTES; }
int oracle_q3k_block_bytes(void) { return Q3K_BYTES; }
int oracle_q8_1_block_bytes(void) { return Q8_1_BYTES; }
