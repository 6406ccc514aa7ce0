/*
 * CPU oracle for GGUF block-quantized GEMV / GEMM / routed-expert FFN.
 *
 * TEST INFRASTRUCTURE ONLY. Only the test suite, the package smoke check and
 * the benchmark's CPU-baseline leg may load this library. It shares no code
 * with the CUDA library: its own IEEE binary16 conversion, its own block
 * decoding, its own arithmetic. Plain single-threaded C, no SIMD intrinsics.
 * Build with -ffp-contract=off so that every float expression below rounds
 * exactly where it is written (no fused multiply-add is introduced).
 *
 * Sources (web pages; "Quantization" etc. are section names on them):
 *  - cera README, "Quantization": weights in Q4_0/Q4_1/Q8_0/Q4_K, activations
 *    quantized dynamically to Q8_0 for an integer GEMV.
 *  - alice-llm docs, "Quantization Block Specs" table: Q4_K = d(f16) + dmin(f16)
 *    + scales[12] + qs[128] per 256 elements; Q8_0 = d(f16) + qs[32]; Q5_K =
 *    d(f16) + dmin(f16) + scales[12] + qh[32] + qs[128] (176 bytes); Q6_K =
 *    ql[128] + qh[64] + scales[16] + d(f16) per 256 elements (210 bytes).
 *  - alice-llm docs, "aarch64 NEON Quantized Matvec Bench", design notes: the
 *    Q6_K six-bit quants are assembled from ql and qh, qh's bit pairs feeding
 *    the four quadrants; "Computation Path (Q4_K)" item 2: Q6_K x Q8_K is an
 *    integer dot, multiplied out only at the scales.
 *  - alice-llm docs, "Computation Path (Q4_K)": quantize the input to Q8_K
 *    (256 elements, f32 scale, i8 values, i16 block sums); 8 sub-blocks x 32
 *    integer accumulation with 6-bit packed scales and mins; result
 *    d * d_q8 * sum(scale*q4*q8) - dmin * d_q8 * sum(min*bsum).
 *  - alice-llm docs, "Phase 4 - i8 Dynamic Quantization + SDOT": per-chunk
 *    amax, scale 127/amax, round to int8.
 *  - cera README, "Supported models" (lfm2moe): each token picks 4 of 32
 *    experts; the routed FFN output is the router-weighted sum of the experts'
 *    outputs. alice-llm "WGSL Shader Architecture": SwiGLU = silu(gate) * up.
 *
 * Readings where the pages are silent (the plainest ones):
 *  - Q4_0/Q4_1/Q8_1 layouts and the Q4_K 6-bit scale packing are the standard
 *    GGUF ones; activation scale d = amax/127 in fp32, q = round-half-away of
 *    x * (1/d) clamped to [-127, 127], d stored as fp16 (round to nearest
 *    even) for Q8_0/Q8_1 and as fp32 for Q8_K; Q8_1 also stores
 *    s = fp16(d * sum(q)) and the Q4_1 x Q8_1 dot uses s for its offset term.
 *  - Q5_K: Q4_K's nibbles, scales and mins, with a fifth bit for element i
 *    in qh[i % 32], bit i / 32 (the sub-block); value = d * sc * q5 - dmin * m.
 *  - Q6_K element order: the standard GGUF one. Half h = i / 128 of the
 *    superblock, quadrant q = (i % 128) / 32, l = i % 32: low four bits from
 *    ql[64h + l + 32(q & 1)] (low nibble for q < 2, high for q >= 2), high
 *    two bits from qh[32h + l] bits 2q, 2q+1; value = d * scales[i / 16] *
 *    (q6 - 32) with int8 scales.
 *  - Quantization decisions are taken in fp32, the precision the pages'
 *    quantizer works in. Everything after the integer block dots is fp64.
 *
 * Parity pins for every function live in the CPU test suite (closed forms,
 * brute-force dequantize-and-dot in exact rationals, invariants, a literal
 * hand-written block fixture).
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

enum { ORC_Q4_0 = 2, ORC_Q4_1 = 3, ORC_Q8_0 = 8, ORC_Q8_1 = 9, ORC_Q4_K = 12, ORC_Q5_K = 13, ORC_Q6_K = 14,
       ORC_Q8_K = 15 };
enum { ORC_OK = 0, ORC_BAD = -1 };

/* ------------------------------------------------------------------ binary16 */

/* Exact value of an IEEE 754 binary16 bit pattern. */
double oracle_half_to_double(uint16_t h)
{
    int sign = h >> 15;
    int e = (h >> 10) & 31;
    int f = h & 1023;
    double v;
    if (e == 0)
        v = ldexp((double)f, -24);               /* subnormal: f * 2^-24 */
    else if (e == 31)
        v = f ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + f), e - 25);   /* (1 + f/1024) * 2^(e-15) */
    return sign ? -v : v;
}

/* Round a float to binary16, nearest-even, keeping subnormals. */
uint16_t oracle_float_to_half(float xf)
{
    double x = (double)xf;                       /* exact */
    uint16_t sign = signbit(x) ? 0x8000 : 0;
    double a = fabs(x);
    if (isnan(x)) return 0x7e00;
    if (a >= 65520.0) return sign | 0x7c00;      /* at or past the halfway point above 65504 */
    if (a < ldexp(1.0, -14)) {                   /* subnormal range: multiples of 2^-24 */
        double q = nearbyint(a * ldexp(1.0, 24)); /* default rounding mode: nearest-even */
        return sign | (uint16_t)q;               /* q == 1024 encodes the smallest normal */
    }
    int ex;
    frexp(a, &ex);                               /* a in [2^(ex-1), 2^ex) */
    int E = ex - 1;
    double s = nearbyint(ldexp(a, 10 - E));      /* significand in [1024, 2048] */
    if (s == 2048.0) { s = 1024.0; E += 1; }
    if (E + 15 >= 31) return sign | 0x7c00;
    return sign | (uint16_t)(((E + 15) << 10) | ((int)s - 1024));
}

static uint16_t rd_u16(const uint8_t* p) { return (uint16_t)(p[0] | (p[1] << 8)); }
static void wr_u16(uint8_t* p, uint16_t v) { p[0] = (uint8_t)v; p[1] = (uint8_t)(v >> 8); }
static double rd_h(const uint8_t* p) { return oracle_half_to_double(rd_u16(p)); }
static float rd_f32(const uint8_t* p) { float f; memcpy(&f, p, 4); return f; }
static void wr_f32(uint8_t* p, float f) { memcpy(p, &f, 4); }

/* ------------------------------------------------------ activation quantizers */

/* One block of n floats -> scale d (fp32) and int8 quants, as the pages' Phase-4
 * quantizer does it: amax, d = amax/127, q = round(x / d) via x * (1/d). */
static float quantize_block(const float* x, int n, int8_t* q)
{
    float amax = 0.0f;
    for (int i = 0; i < n; i++) {
        float a = fabsf(x[i]);
        if (a > amax) amax = a;
    }
    float d = amax / 127.0f;
    float id = (d != 0.0f) ? 1.0f / d : 0.0f;
    for (int i = 0; i < n; i++) {
        float v = roundf(x[i] * id);             /* half away from zero */
        if (v > 127.0f) v = 127.0f;
        if (v < -127.0f) v = -127.0f;
        q[i] = (int8_t)v;
    }
    return d;
}

/* Q8_0: per 32 elements, fp16 d then 32 int8 (34 bytes). */
void oracle_quantize_q8_0(int64_t M, int64_t K, const float* x, uint8_t* out)
{
    int64_t nb = K / 32;
    for (int64_t m = 0; m < M; m++)
        for (int64_t b = 0; b < nb; b++) {
            int8_t q[32];
            float d = quantize_block(x + m * K + 32 * b, 32, q);
            uint8_t* blk = out + (m * nb + b) * 34;
            wr_u16(blk, oracle_float_to_half(d));
            memcpy(blk + 2, q, 32);
        }
}

/* Q8_1: as Q8_0 plus s = fp16(d * sum q) (36 bytes: d, s, qs[32]). */
void oracle_quantize_q8_1(int64_t M, int64_t K, const float* x, uint8_t* out)
{
    int64_t nb = K / 32;
    for (int64_t m = 0; m < M; m++)
        for (int64_t b = 0; b < nb; b++) {
            int8_t q[32];
            float d = quantize_block(x + m * K + 32 * b, 32, q);
            int sum = 0;
            for (int i = 0; i < 32; i++) sum += q[i];
            float s = d * (float)sum;
            uint8_t* blk = out + (m * nb + b) * 36;
            wr_u16(blk, oracle_float_to_half(d));
            wr_u16(blk + 2, oracle_float_to_half(s));
            memcpy(blk + 4, q, 32);
        }
}

/* Q8_K: per 256 elements, fp32 d, 256 int8, 16 int16 sums of 16 quants (292 bytes). */
void oracle_quantize_q8_k(int64_t M, int64_t K, const float* x, uint8_t* out)
{
    int64_t ns = K / 256;
    for (int64_t m = 0; m < M; m++)
        for (int64_t s = 0; s < ns; s++) {
            int8_t q[256];
            float d = quantize_block(x + m * K + 256 * s, 256, q);
            uint8_t* blk = out + (m * ns + s) * 292;
            wr_f32(blk, d);
            memcpy(blk + 4, q, 256);
            for (int i = 0; i < 16; i++) {
                int sum = 0;
                for (int j = 0; j < 16; j++) sum += q[16 * i + j];
                wr_u16(blk + 260 + 2 * i, (uint16_t)(int16_t)sum);
            }
        }
}

/* ---------------------------------------------------------------- decoding */

/* Quant (nibble) of element i of a 16-byte Q4_0/Q4_1 nibble array. */
static int nib32(const uint8_t* qs, int i) { return i < 16 ? (qs[i] & 15) : (qs[i - 16] >> 4); }

/* Six-bit scale and min of sub-block j from the twelve Q4_K scale bytes. */
void oracle_q4k_scale_min(const uint8_t* S, int j, int* sc, int* mn)
{
    if (j < 4) {
        *sc = S[j] & 63;
        *mn = S[j + 4] & 63;
    } else {
        *sc = (S[j + 4] & 15) | ((S[j - 4] >> 6) << 4);
        *mn = (S[j + 4] >> 4) | ((S[j] >> 6) << 4);
    }
}

/* Quant of element i (0..255) of a Q4_K superblock's qs[128]. */
static int nib256(const uint8_t* qs, int i)
{
    int g = i / 64, r = i % 64;
    return r < 32 ? (qs[32 * g + r] & 15) : (qs[32 * g + r - 32] >> 4);
}

/* Five-bit quant (0..31) of element i (0..255) of a Q5_K superblock. */
static int q5k_quant(const uint8_t* blk, int i)
{
    return nib256(blk + 48, i) | (((blk[16 + i % 32] >> (i / 32)) & 1) << 4);
}

/* Six-bit quant (0..63) of element i (0..255) of a Q6_K superblock. */
static int q6k_quant(const uint8_t* blk, int i)
{
    int h = i / 128, q = (i % 128) / 32, l = i % 32;
    int b = blk[64 * h + l + 32 * (q & 1)];
    int lo = q < 2 ? (b & 15) : (b >> 4);
    int hi = (blk[128 + 32 * h + l] >> (2 * q)) & 3;
    return lo | (hi << 4);
}

/* Dequantized value of element k of a weight row, in fp64 (exact). */
double oracle_weight_value(int fmt, const uint8_t* row, int64_t k)
{
    switch (fmt) {
    case ORC_Q4_0: { const uint8_t* b = row + (k / 32) * 18; return rd_h(b) * (nib32(b + 2, (int)(k % 32)) - 8); }
    case ORC_Q4_1: { const uint8_t* b = row + (k / 32) * 20; return rd_h(b) * nib32(b + 4, (int)(k % 32)) + rd_h(b + 2); }
    case ORC_Q8_0: { const uint8_t* b = row + (k / 32) * 34; return rd_h(b) * (int8_t)b[2 + k % 32]; }
    case ORC_Q4_K: {
        const uint8_t* b = row + (k / 256) * 144;
        int i = (int)(k % 256), sc, mn;
        oracle_q4k_scale_min(b + 4, i / 32, &sc, &mn);
        return rd_h(b) * sc * nib256(b + 16, i) - rd_h(b + 2) * mn;
    }
    case ORC_Q5_K: {
        const uint8_t* b = row + (k / 256) * 176;
        int i = (int)(k % 256), sc, mn;
        oracle_q4k_scale_min(b + 4, i / 32, &sc, &mn);
        return rd_h(b) * sc * q5k_quant(b, i) - rd_h(b + 2) * mn;
    }
    case ORC_Q6_K: {
        const uint8_t* b = row + (k / 256) * 210;
        int i = (int)(k % 256);
        return rd_h(b + 208) * (int8_t)b[192 + i / 16] * (q6k_quant(b, i) - 32);
    }
    }
    return NAN;
}

/* Dequantized value of element k of a quantized activation row (fp64, exact). */
double oracle_act_value(int fmt, const uint8_t* row, int64_t k)
{
    switch (fmt) {
    case ORC_Q8_0: { const uint8_t* b = row + (k / 32) * 34; return rd_h(b) * (int8_t)b[2 + k % 32]; }
    case ORC_Q8_1: { const uint8_t* b = row + (k / 32) * 36; return rd_h(b) * (int8_t)b[4 + k % 32]; }
    case ORC_Q8_K: { const uint8_t* b = row + (k / 256) * 292; return (double)rd_f32(b) * (int8_t)b[4 + k % 256]; }
    }
    return NAN;
}

/* ------------------------------------------------------------ block dots */

/* y = W_row . x_row, from per-block exact integer dots and fp64 scale terms.
 * *absterms receives the sum of |term| over the terms the sum is made of
 * (the scale for the rounding-error bound of any fp32 evaluation). */
static double row_dot(int wfmt, const uint8_t* w, const uint8_t* x, int64_t K, double* absterms)
{
    double y = 0.0, at = 0.0;
    if (wfmt == ORC_Q4_0 || wfmt == ORC_Q8_0) {
        int wb = wfmt == ORC_Q4_0 ? 18 : 34;
        for (int64_t b = 0; b < K / 32; b++) {
            const uint8_t* wbk = w + b * wb;
            const uint8_t* xbk = x + b * 34;
            int64_t isum = 0;
            for (int i = 0; i < 32; i++) {
                int qw = wfmt == ORC_Q4_0 ? nib32(wbk + 2, i) - 8 : (int8_t)wbk[2 + i];
                isum += (int64_t)qw * (int8_t)xbk[2 + i];
            }
            double t = rd_h(wbk) * rd_h(xbk) * (double)isum;   /* exact in fp64 */
            y += t;
            at += fabs(t);
        }
    } else if (wfmt == ORC_Q4_1) {
        for (int64_t b = 0; b < K / 32; b++) {
            const uint8_t* wbk = w + b * 20;
            const uint8_t* xbk = x + b * 36;
            int64_t isum = 0;
            for (int i = 0; i < 32; i++) isum += (int64_t)nib32(wbk + 4, i) * (int8_t)xbk[4 + i];
            double t1 = rd_h(wbk) * rd_h(xbk) * (double)isum;  /* d_w d_x sum(q q_x) */
            double t2 = rd_h(wbk + 2) * rd_h(xbk + 2);          /* m_w s_x */
            y += t1 + t2;
            at += fabs(t1) + fabs(t2);
        }
    } else if (wfmt == ORC_Q4_K || wfmt == ORC_Q5_K) {
        int sb = wfmt == ORC_Q4_K ? 144 : 176;
        for (int64_t s = 0; s < K / 256; s++) {
            const uint8_t* wbk = w + s * sb;
            const uint8_t* xbk = x + s * 292;
            double dx = (double)rd_f32(xbk);
            int64_t isum_sc = 0, isum_m = 0;
            for (int j = 0; j < 8; j++) {
                int sc, mn;
                oracle_q4k_scale_min(wbk + 4, j, &sc, &mn);
                int64_t sj = 0, xs = 0;
                for (int i = 32 * j; i < 32 * j + 32; i++) {
                    int qx = (int8_t)xbk[4 + i];
                    int qw = wfmt == ORC_Q4_K ? nib256(wbk + 16, i) : q5k_quant(wbk, i);
                    sj += (int64_t)qw * qx;
                    xs += qx;
                }
                isum_sc += sc * sj;
                isum_m += mn * xs;
            }
            double t1 = dx * rd_h(wbk) * (double)isum_sc;
            double t2 = dx * rd_h(wbk + 2) * (double)isum_m;
            y += t1 - t2;
            at += fabs(t1) + fabs(t2);
        }
    } else if (wfmt == ORC_Q6_K) {
        /* per superblock: isum = sum_j sc_j * sum_{i in sub-block j} (q6_i - 32) * qx_i */
        for (int64_t s = 0; s < K / 256; s++) {
            const uint8_t* wbk = w + s * 210;
            const uint8_t* xbk = x + s * 292;
            int64_t isum = 0;
            for (int j = 0; j < 16; j++) {
                int64_t sj = 0;
                for (int i = 16 * j; i < 16 * j + 16; i++)
                    sj += (int64_t)(q6k_quant(wbk, i) - 32) * (int8_t)xbk[4 + i];
                isum += (int64_t)(int8_t)wbk[192 + j] * sj;
            }
            double t = (double)rd_f32(xbk) * rd_h(wbk + 208) * (double)isum;
            y += t;
            at += fabs(t);
        }
    }
    *absterms = at;
    return y;
}

static int64_t wrow_bytes(int fmt, int64_t K)
{
    switch (fmt) {
    case ORC_Q4_0: return K / 32 * 18;
    case ORC_Q4_1: return K / 32 * 20;
    case ORC_Q8_0: return K / 32 * 34;
    case ORC_Q4_K: return K / 256 * 144;
    case ORC_Q5_K: return K / 256 * 176;
    case ORC_Q6_K: return K / 256 * 210;
    }
    return -1;
}

static int act_fmt_for(int wfmt)
{
    switch (wfmt) {
    case ORC_Q4_0: case ORC_Q8_0: return ORC_Q8_0;
    case ORC_Q4_1: return ORC_Q8_1;
    case ORC_Q4_K: case ORC_Q5_K: case ORC_Q6_K: return ORC_Q8_K;
    }
    return -1;
}

static int64_t xrow_bytes(int afmt, int64_t K)
{
    switch (afmt) {
    case ORC_Q8_0: return K / 32 * 34;
    case ORC_Q8_1: return K / 32 * 36;
    case ORC_Q8_K: return K / 256 * 292;
    }
    return -1;
}

/* y[m][n] = sum_k W[n][k] * X[m][k] for weight rows n in [n0, n1) (all M tokens).
 * W: N rows of wfmt blocks; X: M rows of the paired activation format.
 * y and absterms are [M][N] (full N stride); only columns n0..n1-1 are written. */
int oracle_matmul_rows(int wfmt, int64_t M, int64_t N, int64_t K, const uint8_t* W,
                       const uint8_t* X, int64_t n0, int64_t n1, double* y, double* absterms)
{
    int afmt = act_fmt_for(wfmt);
    if (afmt < 0 || K % 256 != 0 || n0 < 0 || n1 > N) return ORC_BAD;
    int64_t wr = wrow_bytes(wfmt, K), xr = xrow_bytes(afmt, K);
    for (int64_t m = 0; m < M; m++)
        for (int64_t n = n0; n < n1; n++) {
            double at;
            y[m * N + n] = row_dot(wfmt, W + n * wr, X + m * xr, K, &at);
            if (absterms) absterms[m * N + n] = at;
        }
    return ORC_OK;
}

int oracle_matmul(int wfmt, int64_t M, int64_t N, int64_t K, const uint8_t* W,
                  const uint8_t* X, double* y, double* absterms)
{
    return oracle_matmul_rows(wfmt, M, N, K, W, X, 0, N, y, absterms);
}

/* ------------------------------------------------------ dense SwiGLU gate / up */

/* The gate and up projections of a dense SwiGLU FFN and their combination
 * (alice-llm docs "WGSL Shader Architecture": swiglu_fused_q4k computes
 * silu(gate) * up; "The GPU Optimization Journey" phase 4):
 *   g = W_gate[f] . X[m],  u = W_up[f] . X[m]    (the block formula, fp64)
 *   h[m][f] = silu(g) * u = g / (1 + exp(-g)) * u (fp64)
 * gu_aux [M][F][4] = (g, u, absterms(g), absterms(u)); may be NULL. */
int oracle_swiglu(int wfmt, int64_t M, int64_t F, int64_t K, const uint8_t* Wg, const uint8_t* Wu,
                  const uint8_t* X, double* h, double* gu_aux)
{
    int afmt = act_fmt_for(wfmt);
    if (afmt < 0 || K % 256 != 0 || M < 0 || F < 0) return ORC_BAD;
    int64_t wr = wrow_bytes(wfmt, K), xr = xrow_bytes(afmt, K);
    for (int64_t m = 0; m < M; m++)
        for (int64_t f = 0; f < F; f++) {
            double ag, au;
            double g = row_dot(wfmt, Wg + f * wr, X + m * xr, K, &ag);
            double u = row_dot(wfmt, Wu + f * wr, X + m * xr, K, &au);
            h[m * F + f] = g / (1.0 + exp(-g)) * u;
            if (gu_aux) {
                double* a = gu_aux + (m * F + f) * 4;
                a[0] = g; a[1] = u; a[2] = ag; a[3] = au;
            }
        }
    return ORC_OK;
}

/* --------------------------------------------------------- routed expert FFN */

/* One (token, slot) pair's down projection, added into the token's output:
 *   o = W_down[e] . hq   (K values, fp64; W_down[e] rows of F elements)
 *   y[k] += w * o[k],  y_abs[k] += |w| * absterms(o[k])  (y_abs may be NULL) */
static void moe_down_pair(int64_t K, int64_t F, const uint8_t* Wd_e, double w, const uint8_t* hq,
                          double* y, double* y_abs)
{
    for (int64_t k = 0; k < K; k++) {
        double ao;
        double o = row_dot(ORC_Q4_0, Wd_e + k * (F / 32 * 18), hq, F, &ao);
        y[k] += w * o;
        if (y_abs) y_abs[k] += fabs(w) * ao;
    }
}

/* For each token t and slot s (expert e = ids[t][s], router weight w = rw[t][s]):
 *   g = W_gate[e] . xq[t],  u = W_up[e] . xq[t]          (F values, fp64)
 *   h = silu(g) * u = g / (1 + exp(-g)) * u               (fp64)
 *   hq = Q8_0(h rounded to fp32)                          (decisions in fp32)
 *   o = W_down[e] . hq                                    (K values, fp64)
 *   y[t] = sum_s w * o                                    (fp64)
 * Outputs (each may be NULL): y [T][K], y_abs [T][K] = sum_s |w| * absterms(o),
 * h [T][topk][F], hq [T][topk] rows of Q8_0 over F, gu_aux [T][topk][F][4] =
 * (g, u, absterms(g), absterms(u)). Returns ORC_BAD for shapes it cannot take or
 * an expert id outside [0, E) or repeated within a token. */
int oracle_moe(int64_t T, int64_t K, int64_t F, int64_t E, int64_t topk,
               const uint8_t* Wg, const uint8_t* Wu, const uint8_t* Wd,
               const int32_t* ids, const float* rw, const uint8_t* xq,
               double* y, double* y_abs, double* h_out, uint8_t* hq_out, double* gu_aux,
               double* scratch /* at least 2*F doubles */)
{
    if (K % 256 || F % 256) return ORC_BAD;
    int64_t wgr = F * (K / 32 * 18);           /* bytes of one expert's gate (or up) matrix */
    int64_t wdr = K * (F / 32 * 18);           /* bytes of one expert's down matrix */
    int64_t xr = K / 32 * 34, hr = F / 32 * 34;
    double* h = scratch;                       /* F doubles */
    float* hf = (float*)(scratch + F);         /* F floats */
    uint8_t hq_local[65536];
    if (hr > (int64_t)sizeof hq_local) return ORC_BAD;
    for (int64_t t = 0; t < T; t++) {
        for (int64_t s = 0; s < topk; s++) {
            int e = ids[t * topk + s];
            if (e < 0 || e >= E) return ORC_BAD;
            for (int64_t s2 = 0; s2 < s; s2++) if (ids[t * topk + s2] == e) return ORC_BAD;
        }
        for (int64_t k = 0; k < K; k++) { y[t * K + k] = 0.0; if (y_abs) y_abs[t * K + k] = 0.0; }
        for (int64_t s = 0; s < topk; s++) {
            int e = ids[t * topk + s];
            double w = (double)rw[t * topk + s];
            const uint8_t* xt = xq + t * xr;
            for (int64_t f = 0; f < F; f++) {
                double ag, au;
                double g = row_dot(ORC_Q4_0, Wg + e * wgr + f * (K / 32 * 18), xt, K, &ag);
                double u = row_dot(ORC_Q4_0, Wu + e * wgr + f * (K / 32 * 18), xt, K, &au);
                h[f] = g / (1.0 + exp(-g)) * u;
                hf[f] = (float)h[f];
                if (h_out) h_out[(t * topk + s) * F + f] = h[f];
                if (gu_aux) {
                    double* a = gu_aux + ((t * topk + s) * F + f) * 4;
                    a[0] = g; a[1] = u; a[2] = ag; a[3] = au;
                }
            }
            oracle_quantize_q8_0(1, F, hf, hq_local);
            if (hq_out) memcpy(hq_out + (t * topk + s) * hr, hq_local, (size_t)hr);
            moe_down_pair(K, F, Wd + e * wdr, w, hq_local, y + t * K, y_abs ? y_abs + t * K : 0);
        }
    }
    return ORC_OK;
}

/* The routed FFN's second half from given hidden quantisations (the same
 * definition as oracle_moe from hq on): for token t and slot s with
 * valid[t][s] != 0 (valid may be NULL: every pair), expert e = ids[t][s],
 *   o = W_down[e] . hq[t][s],  y[t] = sum_s rw[t][s] * o   (fp64)
 * and y_abs [T][K] = sum_s |rw| * absterms(o) (may be NULL). hq: [T][topk]
 * rows of Q8_0 over F. ORC_BAD for shapes it cannot take or a valid pair's
 * expert id outside [0, E). */
int oracle_moe_down(int64_t T, int64_t K, int64_t F, int64_t E, int64_t topk, const uint8_t* Wd,
                    const int32_t* ids, const float* rw, const int32_t* valid, const uint8_t* hq,
                    double* y, double* y_abs)
{
    if (K % 256 || F % 256) return ORC_BAD;
    int64_t wdr = K * (F / 32 * 18), hr = F / 32 * 34;
    for (int64_t t = 0; t < T; t++) {
        for (int64_t k = 0; k < K; k++) { y[t * K + k] = 0.0; if (y_abs) y_abs[t * K + k] = 0.0; }
        for (int64_t s = 0; s < topk; s++) {
            int64_t i = t * topk + s;
            if (valid && !valid[i]) continue;
            int e = ids[i];
            if (e < 0 || e >= E) return ORC_BAD;
            moe_down_pair(K, F, Wd + e * wdr, (double)rw[i], hq + i * hr, y + t * K, y_abs ? y_abs + t * K : 0);
        }
    }
    return ORC_OK;
}

/* ---------------------------------------------------------- offline weight repack */

/* The packed weight layout of cq_repack, written out byte by byte from its
 * definition (the library's own layout, specified in include/cq.h). The pages
 * repack weights at load for their NPU and CPU kernels -- cera README,
 * "Qualcomm Hexagon" -> "Accelerated Kernels" (Q4_0 / Q8_0 weights repacked
 * into tiles); alice-llm docs, "Phase 6 -> Block-Packed Weight Layout" (rows
 * interleaved so that one load serves several rows) -- but print no layout for
 * a GPU, so the layout itself is a reading: rows in groups of 16, K in
 * segments of 4 blocks; the unit (group G, segment s) of 64 * BB bytes sits at
 * byte (s * ceil(N / 16) + G) * 64 * BB and holds
 *   - per row r of the group: the scale fields of blocks 0..3 of the segment
 *     (Q4_1: d, m = block bytes 0..3; Q4_0 / Q8_0: d = block bytes 0..1), rows
 *     16 (Q4_1) or 8 bytes apart;
 *   - then, per half h (Q8_0: h = 0, 1; Q4_0 / Q4_1: h = 0), per row r, per
 *     lane t = 0..3, per block j = 0..3: quant bytes 16h + 4t .. 16h + 4t + 3 of
 *     block j (offsets within the block's quant array).
 * Rows at or past N are zero. Returns the packed size in bytes, or -1. */
int64_t oracle_repack_size(int fmt, int64_t N, int64_t K)
{
    int64_t bb = fmt == ORC_Q4_0 ? 18 : fmt == ORC_Q4_1 ? 20 : fmt == ORC_Q8_0 ? 34 : 0;
    if (bb == 0 || N < 0 || K <= 0 || K % 256 != 0) return -1;
    return (N + 15) / 16 * (K / 128) * 64 * bb;
}

int oracle_repack(int fmt, int64_t N, int64_t K, const uint8_t* W, uint8_t* out)
{
    int64_t size = oracle_repack_size(fmt, N, K);
    if (size < 0) return ORC_BAD;
    int64_t bb = fmt == ORC_Q4_0 ? 18 : fmt == ORC_Q4_1 ? 20 : 34;
    int64_t ng = (N + 15) / 16, ns = K / 128, unit = 64 * bb, wrow = K / 32 * bb;
    int scale_bytes = fmt == ORC_Q4_1 ? 4 : 2;       /* per block */
    int quant_off = fmt == ORC_Q4_1 ? 4 : 2;         /* quants' offset in the block */
    int halves = fmt == ORC_Q8_0 ? 2 : 1;
    int64_t scale_region = 16 * 4 * scale_bytes;
    memset(out, 0, (size_t)size);
    for (int64_t s = 0; s < ns; s++)
        for (int64_t G = 0; G < ng; G++) {
            uint8_t* u = out + (s * ng + G) * unit;
            for (int r = 0; r < 16; r++) {
                int64_t row = 16 * G + r;
                if (row >= N) continue;
                for (int j = 0; j < 4; j++) {
                    const uint8_t* blk = W + row * wrow + (4 * s + j) * bb;
                    for (int i = 0; i < scale_bytes; i++)
                        u[r * 4 * scale_bytes + j * scale_bytes + i] = blk[i];
                    for (int h = 0; h < halves; h++)
                        for (int t = 0; t < 4; t++)
                            for (int i = 0; i < 4; i++)
                                u[scale_region + h * 1024 + ((r * 4 + t) * 4 + j) * 4 + i] =
                                    blk[quant_off + 16 * h + 4 * t + i];
                }
            }
        }
    return ORC_OK;
}
