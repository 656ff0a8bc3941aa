/*
 * mq_oracle.c -- plain, slow CPU oracle for the q4_K x q8_0 decode matvec.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg may load this library.  It shares no code,
 * header, table or constant with the CUDA library; the two meet only on the
 * byte images produced by the seeded input generator.
 *
 * What it follows:
 *   - "07 . R3 -- Small-model per-token overhead", section 1: decode uses an
 *     MMVQ kernel, a dp4a integer dot product of q4_K weights with
 *     q8_0-quantized activations.  The byte formats are not printed on the
 *     pages; this file uses the GGUF-compatible reading stated next to each
 *     function (144-byte q4_K super-block: f16 d, f16 dmin, twelve bytes of
 *     6-bit scale/min pairs, 128 bytes of 4-bit quants; 34-byte q8_0 block:
 *     f16 scale and 32 int8).
 *   - "04 . 8o -- Killing the CPU stall at decode start", sections 1 and 3.1:
 *     the FFN multiplies by a row-concatenated gate/up weight ffn_gu (gate rows
 *     first, then up rows), then SwiGLU (SiLU(gate) * up), then down.
 *   - "Part 4 . Lecture 08 -- Graph-Resident Decode", section 8: the
 *     quantizer's scan is a max over magnitudes, so it is exactly
 *     order-independent.
 *
 * Precision: every matvec and SiLU value is accumulated in binary64.  The one
 * place fp32 is part of the definition is the q8_0 quantizer (fp32 amax,
 * fp32 IEEE division d = amax/127 and x/d, round half away from zero), built
 * with -ffp-contract=off and without fast-math so those steps are exact IEEE.
 *
 * Parity pins live in tests/test_oracle_*.py; every function below has at
 * least one pin that does not re-type its own formula.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define MQO_QK_K 256
#define MQO_Q4K_BYTES 144
#define MQO_QK8 32
#define MQO_Q8_BYTES 34

/* ---------------------------------------------------------------------------
 * IEEE 754 binary16 <-> binary32, from the format's definition
 * (1 sign bit, 5 exponent bits with bias 15, 10 fraction bits).
 * ------------------------------------------------------------------------- */
float mqo_f16_to_f32(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 31;
    int f = h & 1023;
    double v;
    if (e == 0) {
        v = ldexp((double)f, -24);                 /* zero or subnormal: f * 2^-24 */
    } else if (e == 31) {
        v = (f == 0) ? INFINITY : NAN;
    } else {
        v = ldexp((double)(1024 + f), e - 25);     /* (1 + f/1024) * 2^(e-15) */
    }
    return (float)(sign ? -v : v);
}

/* round a non-negative double to an integer, ties to even */
static double mqo_round_half_even(double y)
{
    double fl = floor(y);
    double diff = y - fl;
    if (diff > 0.5) return fl + 1.0;
    if (diff < 0.5) return fl;
    return (fmod(fl, 2.0) == 0.0) ? fl : fl + 1.0;
}

/* binary64 -> binary16, round to nearest, ties to even */
uint16_t mqo_f64_to_f16(double x)
{
    uint16_t sign = signbit(x) ? 0x8000u : 0u;
    double a = fabs(x);
    if (isnan(x)) return (uint16_t)(sign | 0x7E00u);
    /* 65520 is the midpoint between 65504 (largest finite, odd mantissa) and
     * 2^16; ties go to the even neighbour, which overflows to infinity. */
    if (a >= 65520.0) return (uint16_t)(sign | 0x7C00u);
    if (a < ldexp(1.0, -14)) {
        /* subnormal range: quantum 2^-24; n == 1024 rolls into the smallest normal */
        double n = mqo_round_half_even(ldexp(a, 24));
        return (uint16_t)(sign | (uint16_t)n);
    }
    int E;
    (void)frexp(a, &E);             /* a = m * 2^E, m in [0.5, 1) */
    int e = E - 1;                  /* a in [2^e, 2^(e+1)) */
    double n = mqo_round_half_even(ldexp(a, 10 - e));   /* in [1024, 2048] */
    uint32_t bits = ((uint32_t)(e + 15) << 10) + (uint32_t)(n - 1024.0);
    return (uint16_t)(sign | bits);  /* a carry to 2048 moves into the exponent */
}

/* binary32 -> binary16: every binary32 value is exact in binary64, so the
 * same single rounding applies */
uint16_t mqo_f32_to_f16(float x) { return mqo_f64_to_f16((double)x); }

void mqo_f64_to_f16_array(const double* x, int64_t n, uint16_t* out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = mqo_f64_to_f16(x[i]);
}

static uint16_t mqo_le16(const uint8_t* p) { return (uint16_t)(p[0] | (p[1] << 8)); }

/* ---------------------------------------------------------------------------
 * q8_0 quantization of one column of K floats (K a multiple of 32).
 * Per 32-value block: amax = max |x_i| (fp32); d = amax / 127 (fp32 IEEE);
 * q_i = round_half_away(x_i / d) clamped to [-127, 127], all zero if d == 0;
 * stored: binary16(d) little-endian, then the 32 int8 values.
 * ------------------------------------------------------------------------- */
void mqo_quantize_q8_0(const float* x, int64_t K, uint8_t* out)
{
    for (int64_t b = 0; b < K / MQO_QK8; ++b) {
        const float* xb = x + b * MQO_QK8;
        uint8_t* ob = out + b * MQO_Q8_BYTES;
        float amax = 0.0f;
        for (int i = 0; i < MQO_QK8; ++i) {
            float a = fabsf(xb[i]);
            if (a > amax) amax = a;
        }
        float d = amax / 127.0f;
        uint16_t dh = mqo_f32_to_f16(d);
        ob[0] = (uint8_t)(dh & 0xFF);
        ob[1] = (uint8_t)(dh >> 8);
        for (int i = 0; i < MQO_QK8; ++i) {
            int q = 0;
            if (d != 0.0f) {
                float r = roundf(xb[i] / d);
                if (r > 127.0f) r = 127.0f;
                if (r < -127.0f) r = -127.0f;
                q = (int)r;
            }
            ob[2 + i] = (uint8_t)(int8_t)q;
        }
    }
}

/* one q8_0 block -> (f32 scale, 32 ints) */
static void mqo_unpack_q8_0(const uint8_t* blk, double* dq, int q[32])
{
    *dq = (double)mqo_f16_to_f32(mqo_le16(blk));
    for (int i = 0; i < MQO_QK8; ++i) q[i] = (int)(int8_t)blk[2 + i];
}

/* ---------------------------------------------------------------------------
 * q4_K super-block unpack (GGUF-compatible reading).
 *   bytes 0-1  d     (binary16, little-endian)
 *   bytes 2-3  dmin  (binary16)
 *   bytes 4-15 s[12]: for j < 4: sc_j = s[j] & 63, m_j = s[j+4] & 63;
 *                     for j >= 4: sc_j = (s[j+4] & 15) | ((s[j-4] >> 6) << 4),
 *                                 m_j  = (s[j+4] >> 4) | ((s[j]   >> 6) << 4).
 *   bytes 16-143 qs[128], four 32-byte chunks; in chunk c, byte i holds
 *              element i of sub-block 2c in its low nibble and element i of
 *              sub-block 2c+1 in its high nibble.
 * Weight of element 32j+i: w = d * sc_j * q - dmin * m_j.
 * ------------------------------------------------------------------------- */
void mqo_unpack_q4K(const uint8_t* blk, double* d, double* dmin, int sc[8], int m[8], int q[256])
{
    const uint8_t* s = blk + 4;
    const uint8_t* qs = blk + 16;
    *d = (double)mqo_f16_to_f32(mqo_le16(blk));
    *dmin = (double)mqo_f16_to_f32(mqo_le16(blk + 2));
    for (int j = 0; j < 8; ++j) {
        if (j < 4) {
            sc[j] = s[j] & 63;
            m[j] = s[j + 4] & 63;
        } else {
            sc[j] = (s[j + 4] & 15) | ((s[j - 4] >> 6) << 4);
            m[j] = (s[j + 4] >> 4) | ((s[j] >> 6) << 4);
        }
    }
    for (int c = 0; c < 4; ++c) {
        for (int i = 0; i < 32; ++i) {
            uint8_t byte = qs[32 * c + i];
            q[32 * (2 * c) + i] = byte & 15;
            q[32 * (2 * c + 1) + i] = byte >> 4;
        }
    }
}

/* dequantize one q4_K row of K weights to binary64 (the plain definition) */
void mqo_dequant_q4K_row(const uint8_t* row, int64_t K, double* w)
{
    double d, dmin;
    int sc[8], m[8], q[256];
    for (int64_t b = 0; b < K / MQO_QK_K; ++b) {
        mqo_unpack_q4K(row + b * MQO_Q4K_BYTES, &d, &dmin, sc, m, q);
        for (int j = 0; j < 8; ++j)
            for (int i = 0; i < 32; ++i)
                w[b * MQO_QK_K + 32 * j + i] = d * sc[j] * q[32 * j + i] - dmin * m[j];
    }
}

/* dequantize one q8_0 column of K values to binary64 */
void mqo_dequant_q8_0(const uint8_t* xq, int64_t K, double* x)
{
    double dq;
    int q[32];
    for (int64_t b = 0; b < K / MQO_QK8; ++b) {
        mqo_unpack_q8_0(xq + b * MQO_Q8_BYTES, &dq, q);
        for (int i = 0; i < 32; ++i) x[b * MQO_QK8 + i] = dq * q[i];
    }
}

/* ---------------------------------------------------------------------------
 * Per-32-block integer sums of one column:
 *   sumi[r][J] = sum_i q4(r, 32J+i) * q8(32J+i)   (int32)
 *   sumq[J]    = sum_i q8(32J+i)                  (int32)
 * ------------------------------------------------------------------------- */
void mqo_block_sums(const uint8_t* W, const uint8_t* xq, int64_t rows, int64_t K,
                    int32_t* sumi, int32_t* sumq)
{
    const int64_t nb = K / MQO_QK_K, nq = K / MQO_QK8;
    double d, dmin, dq;
    int sc[8], m[8], q[256], q8[32];
    for (int64_t J = 0; J < nq; ++J) {
        mqo_unpack_q8_0(xq + J * MQO_Q8_BYTES, &dq, q8);
        int32_t s = 0;
        for (int i = 0; i < 32; ++i) s += q8[i];
        sumq[J] = s;
    }
    for (int64_t r = 0; r < rows; ++r) {
        const uint8_t* row = W + r * nb * MQO_Q4K_BYTES;
        for (int64_t b = 0; b < nb; ++b) {
            mqo_unpack_q4K(row + b * MQO_Q4K_BYTES, &d, &dmin, sc, m, q);
            for (int j = 0; j < 8; ++j) {
                int64_t J = b * 8 + j;
                mqo_unpack_q8_0(xq + J * MQO_Q8_BYTES, &dq, q8);
                int32_t s = 0;
                for (int i = 0; i < 32; ++i) s += q[32 * j + i] * q8[i];
                sumi[r * nq + J] = s;
            }
        }
    }
}

/* ---------------------------------------------------------------------------
 * Other weight types of the pages' models (GGUF-compatible readings), for the
 * same MMVQ dot product against q8_0 activations:
 *   q4_0, 32 weights in 18 bytes: [0:2] f16 d, [2:18] sixteen bytes; byte i
 *         holds weight i in its low nibble and weight i+16 in its high
 *         nibble; w = d * (q - 8) with q in 0..15.
 *   q8_0, 32 weights in 34 bytes, the activation's own block format:
 *         w = d * q with q an int8.
 * The type is named by its block size in bytes (18 or 34).
 * ------------------------------------------------------------------------- */
#define MQO_Q4_0_BYTES 18

/* one weight block -> (f64 scale, 32 signed integer weights w/d) */
static void mqo_unpack_wblock(int block_bytes, const uint8_t* blk, double* d, int q[32])
{
    *d = (double)mqo_f16_to_f32(mqo_le16(blk));
    if (block_bytes == MQO_Q4_0_BYTES) {
        for (int i = 0; i < 16; ++i) {
            q[i] = (blk[2 + i] & 15) - 8;
            q[i + 16] = (blk[2 + i] >> 4) - 8;
        }
    } else {
        for (int i = 0; i < MQO_QK8; ++i) q[i] = (int)(int8_t)blk[2 + i];
    }
}

/* dequantize one row of K weights of a 32-weight block type to binary64 */
void mqo_dequant_w_row(int block_bytes, const uint8_t* row, int64_t K, double* w)
{
    double d;
    int q[32];
    for (int64_t b = 0; b < K / MQO_QK8; ++b) {
        mqo_unpack_wblock(block_bytes, row + b * block_bytes, &d, q);
        for (int i = 0; i < MQO_QK8; ++i) w[b * MQO_QK8 + i] = d * q[i];
    }
}

/* y = sum_b dq8_b * (d_b * sumi_b) with sumi_b = sum_i q_bi * q8_bi (int), and
 * T = sum_b |that product|, for one row of a 32-weight block type */
static void mqo_row_dot_w(int block_bytes, const uint8_t* row, const uint8_t* xq, int64_t K, double* y, double* T)
{
    double acc = 0.0, tsum = 0.0, d, dq;
    int q[32], q8[32];
    for (int64_t b = 0; b < K / MQO_QK8; ++b) {
        mqo_unpack_wblock(block_bytes, row + b * block_bytes, &d, q);
        mqo_unpack_q8_0(xq + b * MQO_Q8_BYTES, &dq, q8);
        int64_t sumi = 0;
        for (int i = 0; i < MQO_QK8; ++i) sumi += (int64_t)q[i] * q8[i];
        const double t = dq * (d * (double)sumi);
        acc += t;
        tsum += fabs(t);
    }
    *y = acc;
    if (T) *T = tsum;
}

/* y[c][t], T[c][t] for the listed rows (all rows when row_ids is NULL) */
void mqo_matvec_w(int block_bytes, const uint8_t* W, const uint8_t* xq, int64_t rows, int64_t K, int64_t ncols,
                  const int64_t* row_ids, int64_t n_ids, double* y, double* T)
{
    const int64_t rb = K / MQO_QK8 * block_bytes, cb = K / MQO_QK8 * MQO_Q8_BYTES;
    const int64_t n = row_ids ? n_ids : rows;
    for (int64_t c = 0; c < ncols; ++c)
        for (int64_t t = 0; t < n; ++t) {
            const int64_t r = row_ids ? row_ids[t] : t;
            mqo_row_dot_w(block_bytes, W + r * rb, xq + c * cb, K, &y[c * n + t], T ? &T[c * n + t] : 0);
        }
}

/* ---------------------------------------------------------------------------
 * One output row of the matvec, via the per-block integer sums:
 *   y = sum_b sum_j dq8_J * (d_b * sc_bj * sumi_J - dmin_b * m_bj * sumq_J)
 * plus T = sum of |each of the two products| (the tolerance scale).
 * This equals the dot product of the dequantized row with the dequantized
 * activation, regrouped per 32-block (a pin checks that).
 * ------------------------------------------------------------------------- */
static void mqo_row_dot(const uint8_t* row, const uint8_t* xq, int64_t K, double* y, double* T)
{
    double acc = 0.0, tsum = 0.0;
    double d, dmin, dq;
    int sc[8], m[8], q[256], q8[32];
    for (int64_t b = 0; b < K / MQO_QK_K; ++b) {
        mqo_unpack_q4K(row + b * MQO_Q4K_BYTES, &d, &dmin, sc, m, q);
        for (int j = 0; j < 8; ++j) {
            mqo_unpack_q8_0(xq + (b * 8 + j) * MQO_Q8_BYTES, &dq, q8);
            int64_t sumi = 0, sumq = 0;
            for (int i = 0; i < 32; ++i) {
                sumi += (int64_t)q[32 * j + i] * q8[i];
                sumq += q8[i];
            }
            double t1 = dq * (d * sc[j] * (double)sumi);
            double t2 = dq * (dmin * m[j] * (double)sumq);
            acc += t1 - t2;
            tsum += fabs(t1) + fabs(t2);
        }
    }
    *y = acc;
    if (T) *T = tsum;
}

/* y[c][r], T[c][r] for all rows and ncols columns; xq is [ncols][K/32] blocks */
void mqo_matvec(const uint8_t* W, const uint8_t* xq, int64_t rows, int64_t K, int64_t ncols,
                double* y, double* T)
{
    const int64_t rb = K / MQO_QK_K * MQO_Q4K_BYTES, cb = K / MQO_QK8 * MQO_Q8_BYTES;
    for (int64_t c = 0; c < ncols; ++c)
        for (int64_t r = 0; r < rows; ++r)
            mqo_row_dot(W + r * rb, xq + c * cb, K, &y[c * rows + r], T ? &T[c * rows + r] : 0);
}

/* the same for a list of row indices: y[c][t] is row row_ids[t] */
void mqo_matvec_rows(const uint8_t* W, const uint8_t* xq, int64_t K, int64_t ncols,
                     const int64_t* row_ids, int64_t n_ids, double* y, double* T)
{
    const int64_t rb = K / MQO_QK_K * MQO_Q4K_BYTES, cb = K / MQO_QK8 * MQO_Q8_BYTES;
    for (int64_t c = 0; c < ncols; ++c)
        for (int64_t t = 0; t < n_ids; ++t)
            mqo_row_dot(W + row_ids[t] * rb, xq + c * cb, K, &y[c * n_ids + t], T ? &T[c * n_ids + t] : 0);
}

/* ---------------------------------------------------------------------------
 * SwiGLU gate: h = SiLU(g) * u = g / (1 + exp(-g)) * u, binary64.
 * ------------------------------------------------------------------------- */
double mqo_silu(double g) { return g / (1.0 + exp(-g)); }

void mqo_silu_mul(const double* g, const double* u, int64_t n, double* h)
{
    for (int64_t i = 0; i < n; ++i) h[i] = mqo_silu(g[i]) * u[i];
}

/* ---------------------------------------------------------------------------
 * The whole FFN for ncols columns, as a plain chain of the steps above:
 *   xq = q8_0(x); [g; u] = W_gu . xq (gate rows 0..I-1, up rows I..2I-1);
 *   h = SiLU(g) * u; hq = q8_0(fp32(h)); y = W_down . hq.
 * The quantizer's input is fp32 by definition, so h is rounded once to fp32
 * before it is re-quantized.  Scratch: gu [2I] doubles, h [I] doubles,
 * hf [I] floats, xq_scratch [H/32*34] bytes.  Outputs y [ncols][H] and
 * hq_out [ncols][I/32*34] (the re-quantized h of every column).
 * ------------------------------------------------------------------------- */
void mqo_ffn(const uint8_t* W_gu, const uint8_t* W_down, const float* x, int64_t H, int64_t I,
             int64_t ncols, uint8_t* xq_scratch, double* gu, double* h, float* hf,
             uint8_t* hq_out, double* y)
{
    const int64_t hqb = I / MQO_QK8 * MQO_Q8_BYTES;
    for (int64_t c = 0; c < ncols; ++c) {
        mqo_quantize_q8_0(x + c * H, H, xq_scratch);
        mqo_matvec(W_gu, xq_scratch, 2 * I, H, 1, gu, 0);
        mqo_silu_mul(gu, gu + I, I, h);
        for (int64_t i = 0; i < I; ++i) hf[i] = (float)h[i];
        uint8_t* hq = hq_out + c * hqb;
        mqo_quantize_q8_0(hf, I, hq);
        mqo_matvec(W_down, hq, H, I, 1, y + c * H, 0);
    }
}

/* ---------------------------------------------------------------------------
 * Prefill ("07 . R3 -- Small-model per-token overhead", section 1: the 7B
 * prefill GEMM runs in half precision over a resident f16 copy of the
 * weights, dequantized once).
 * ------------------------------------------------------------------------- */

/* the f16 copy of one q4_K row: each weight d*sc*q - dmin*m in binary64
 * (the plain definition above), rounded once to binary16; scratch holds K doubles */
void mqo_dequant_q4K_f16_row(const uint8_t* row, int64_t K, double* scratch, uint16_t* out)
{
    mqo_dequant_q4K_row(row, K, scratch);
    for (int64_t k = 0; k < K; ++k) out[k] = mqo_f64_to_f16(scratch[k]);
}

/* y[i][j] = sum over k of W16[rows[j]][k] * X16[toks[i]][k], the binary16
 * values taken exactly and the products summed in binary64; T[i][j] = the sum
 * of the products' magnitudes (the scale of the float tolerance) */
void mqo_gemm_f16(const uint16_t* W16, const uint16_t* X16, int64_t K, const int64_t* rows, int64_t nr,
                  const int64_t* toks, int64_t nt, double* y, double* T)
{
    for (int64_t i = 0; i < nt; ++i) {
        const uint16_t* x = X16 + toks[i] * K;
        for (int64_t j = 0; j < nr; ++j) {
            const uint16_t* w = W16 + rows[j] * K;
            double sum = 0.0, mag = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                double prod = (double)mqo_f16_to_f32(w[k]) * (double)mqo_f16_to_f32(x[k]);
                sum += prod;
                mag += fabs(prod);
            }
            y[i * nr + j] = sum;
            T[i * nr + j] = mag;
        }
    }
}
