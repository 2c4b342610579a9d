/*
 * NVFP4 oracle: a plain, slow, CPU-only statement of what the NVFP4 W4A4
 * linear / MLP hot path computes.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file.  Only the test suite, the smoke check and the CPU-baseline
 * leg of the benchmark use it.  It shares no code, header, table or constant
 * generator with the CUDA library.
 *
 * Build: gcc -O2 -std=c11 -ffp-contract=off -fno-fast-math -fopenmp -shared -fPIC
 * (-ffp-contract=off: every fp32 step below is one IEEE-754 binary32 operation
 * rounded to nearest-even; no fused multiply-adds).
 *
 * Sources (cited by page title and section):
 *  [P0]  "PERFORMANCE -- verified hot-path audit and prioritized fixes"
 *        (nvfp4-megamoe-kernel PERFORMANCE_AUDIT.md), section P0: the
 *        activation global scale is amax clamped to >= 1e-8, divided by
 *        6.0 * 448.0, and is kept on the device as a (1,) tensor.
 *  [P8]  same page, section P8 items 1-2: RMSNorm fused with the next
 *        linear's input quantization; FP4 quantization fused into the
 *        producer's epilogue.
 *  [GLU] "CUDA: NVFP4 prefill on Blackwell leaves ~1.45x performance on the
 *        table" (llama.cpp discussion 28514), list "What the patch does",
 *        item 2: GLU output quantized directly into the next GEMM's
 *        activation format, gate and up sharing one quantized input,
 *        batched-row rms_norm; item 3: FP4 MMA accumulated in place.
 *  [FMT] the NVFP4 number format: E2M1 element codes with the magnitude set
 *        {0, 0.5, 1, 1.5, 2, 3, 4, 6}, one E4M3 scale (max 448) per 16
 *        consecutive elements along K, one FP32 per-tensor global scale,
 *        round-to-nearest-even (OCP Microscaling Formats v1.0 for the E2M1
 *        and E4M3 encodings).
 *  [SFL] the 128-row x 4-column scale-factor tile layout that the Blackwell
 *        block-scaled MMA reads (public PTX ISA / cuBLAS "block scaling
 *        factors layout").
 *  [ROPE] "PERFORMANCE -- verified hot-path audit and prioritized fixes",
 *        section P5 (RoPE on the last rope_dim columns of each head, as
 *        (even, odd) pairs, in float32 from bf16 and back) and the list of
 *        structural targets, item 3 (RoPE fused into the Q/KV GEMM epilogue).
 *
 * Readings taken where the sources are silent are stated at each function.
 */
#include <stdint.h>
#include <stddef.h>
#include <math.h>
#include <string.h>
#include <stdlib.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------ */
/* bf16 <-> binary64                                                   */
/* ------------------------------------------------------------------ */

double oracle_bf16_value(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return (double)f;
}

/* Round a binary64 value to the nearest bf16 (8 significant bits, binary32
 * exponent range), ties to even, in ONE rounding step.  Finite inputs only. */
uint16_t oracle_bf16_from_double(double d)
{
    if (d == 0.0) return signbit(d) ? 0x8000 : 0x0000;
    int e;
    frexp(d, &e);                 /* |d| = m * 2^e, m in [0.5, 1) */
    int exp_unbiased = e - 1;     /* |d| in [2^x, 2^(x+1)) */
    if (exp_unbiased < -126) exp_unbiased = -126;   /* bf16 subnormal quantum */
    double quantum = ldexp(1.0, exp_unbiased - 7);
    double r = nearbyint(d / quantum) * quantum;    /* default mode: nearest-even */
    float f = (float)r;           /* exact: r has <= 8 significant bits */
    uint32_t u;
    memcpy(&u, &f, 4);
    return (uint16_t)(u >> 16);
}

/* ------------------------------------------------------------------ */
/* E2M1 (element codes)                                                */
/* ------------------------------------------------------------------ */

/* The eight magnitudes of [FMT], indexed by the low three bits of a code;
 * bit 3 is the sign (OCP E2M1: 1 sign, 2 exponent, 1 mantissa bit). */
static const double E2M1_MAGNITUDE[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};

double oracle_e2m1_value(int code)
{
    double m = E2M1_MAGNITUDE[code & 7];
    return (code & 8) ? -m : m;
}

/* Encode a binary32 value as E2M1 by round-to-nearest-even over the finite
 * value set [FMT]: the representable magnitude nearest |q| wins; on an exact
 * tie the code with an even mantissa bit (code bit 0 == 0) wins.  Values
 * beyond 6 take 6 (saturation: E2M1 has no Inf/NaN).
 * Reading: the sign bit is kept even when the magnitude rounds to zero
 * (-0.1 -> 0x8), as an IEEE round-to-nearest of a negative value gives -0. */
int oracle_e2m1_encode(float q)
{
    double a = fabs((double)q);
    if (a > 6.0) a = 6.0;   /* saturate first: far beyond 6 every distance rounds alike */
    int best = 0;
    double best_err = fabs(a - E2M1_MAGNITUDE[0]);
    for (int c = 1; c < 8; c++) {
        double err = fabs(a - E2M1_MAGNITUDE[c]);
        if (err < best_err || (err == best_err && (c & 1) == 0 && (best & 1) == 1)) {
            best = c;
            best_err = err;
        }
    }
    return signbit(q) ? (best | 8) : best;
}

/* ------------------------------------------------------------------ */
/* E4M3 (block scales), the "fn" variant: bias 7, no Inf, 0x7F = NaN     */
/* ------------------------------------------------------------------ */

double oracle_e4m3_value(int byte)
{
    int s = (byte >> 7) & 1, e = (byte >> 3) & 15, m = byte & 7;
    double v;
    if (e == 15 && m == 7) return NAN;
    if (e == 0) v = ldexp((double)m, -9);                 /* subnormal: m/8 * 2^-6 */
    else v = ldexp(1.0 + m / 8.0, e - 7);
    return s ? -v : v;
}

/* Encode a non-negative binary32 scale as an unsigned E4M3 byte: nearest
 * finite value among 0x00..0x7E, ties to the even mantissa (byte bit 0 == 0),
 * saturating at 448 (0x7E) [FMT].  Reading: scales are unsigned, so the sign
 * bit is always 0; subnormal E4M3 values are used. */
static double E4M3_VALUE[128];

__attribute__((constructor)) static void init_e4m3_table(void)
{
    for (int c = 0; c < 128; c++) E4M3_VALUE[c] = oracle_e4m3_value(c);
}

int oracle_e4m3_encode(float s)
{
    double a = (double)s;
    if (a > 448.0) a = 448.0;   /* saturate first (satfinite) */
    int best = 0;
    double best_err = fabs(a - E4M3_VALUE[0]);
    for (int c = 1; c <= 0x7E; c++) {
        double err = fabs(a - E4M3_VALUE[c]);
        if (err < best_err || (err == best_err && (c & 1) == 0 && (best & 1) == 1)) {
            best = c;
            best_err = err;
        }
    }
    return best;
}

/* ------------------------------------------------------------------ */
/* Per-tensor global scale [P0]                                        */
/* ------------------------------------------------------------------ */

/* amax over |x| of a row-pitched bf16 matrix (the bf16 -> fp32 widening is
 * exact, so the max is exact). */
float oracle_amax_bf16(const uint16_t* x, int64_t rows, int64_t cols, int64_t ld)
{
    double amax = 0.0;
    for (int64_t r = 0; r < rows; r++)
        for (int64_t c = 0; c < cols; c++) {
            double v = fabs(oracle_bf16_value(x[r * ld + c]));
            if (v > amax) amax = v;
        }
    return (float)amax;
}

/* [P0]: amax clamped below at 1e-8 (a binary32 clamp, as the page clamps a
 * float32 tensor), divided by 6.0 * 448.0 = 2688 in binary64 (a Python
 * float), and stored as a binary32 device value.  For binary32 operands the
 * binary64 quotient rounded to binary32 equals the correctly rounded
 * binary32 quotient. */
float oracle_global_scale_from_amax(float amax)
{
    float clamp = (float)1e-8;
    double a = (double)(amax > clamp ? amax : clamp);
    return (float)(a / (6.0 * 448.0));
}

float oracle_global_scale(const uint16_t* x, int64_t rows, int64_t cols, int64_t ld)
{
    return oracle_global_scale_from_amax(oracle_amax_bf16(x, rows, cols, ld));
}

/* ------------------------------------------------------------------ */
/* Block quantization [FMT]                                            */
/* ------------------------------------------------------------------ */

/* Quantize one 16-element block given the global scale g.
 * Reading (the sources fix the formats, not the arithmetic order), in
 * binary32, one rounding per operation:
 *    d     = 6 * g
 *    s_raw = amax16 / d                  -> scale byte sc = E4M3(s_raw)
 *    den   = value(sc) * g
 *    q_i   = x_i / den                   -> code_i = E2M1(q_i)
 * so that x_i ~= E2M1(code_i) * E4M3(sc) * g.  A block whose scale rounds
 * to zero stores +0 codes. */
static void quantize_block16(const float* x, float g, uint8_t* sc_out, uint8_t* nib_out)
{
    float amax = 0.0f;
    for (int i = 0; i < 16; i++) {
        float a = fabsf(x[i]);
        if (a > amax) amax = a;
    }
    float d = 6.0f * g;
    float s_raw = amax / d;
    int sc = oracle_e4m3_encode(s_raw);
    *sc_out = (uint8_t)sc;
    if (sc == 0) {
        for (int i = 0; i < 16; i++) nib_out[i] = 0;
        return;
    }
    float den = (float)oracle_e4m3_value(sc) * g;
    for (int i = 0; i < 16; i++) {
        float q = x[i] / den;
        nib_out[i] = (uint8_t)oracle_e2m1_encode(q);
    }
}

/* Quantize a row-pitched bf16 matrix [rows x cols] (cols % 16 == 0).
 * codes: [rows][cols/2] bytes; element 2i in the low nibble and 2i+1 in the
 *        high nibble of byte i (reading: the memory order of packed FP4 in the
 *        PTX ISA and the OCP spec -- the first element in the low bits).
 * sf:    logical (unswizzled) scales [rows][cols/16]. */
void oracle_quantize(const uint16_t* x, int64_t rows, int64_t cols, int64_t ld, float g,
                     uint8_t* codes, uint8_t* sf)
{
    int64_t kb = cols / 16;
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; r++) {
        for (int64_t b = 0; b < kb; b++) {
            float xb[16];
            uint8_t nib[16];
            for (int i = 0; i < 16; i++) xb[i] = (float)oracle_bf16_value(x[r * ld + b * 16 + i]);
            quantize_block16(xb, g, &sf[r * kb + b], nib);
            for (int i = 0; i < 8; i++)
                codes[r * (cols / 2) + b * 8 + i] = (uint8_t)(nib[2 * i] | (nib[2 * i + 1] << 4));
        }
    }
}

/* Decode one element of a quantized matrix to binary64 (exact). */
double oracle_dequant_element(const uint8_t* codes, const uint8_t* sf, int64_t cols, float g,
                              int64_t r, int64_t k)
{
    uint8_t byte = codes[r * (cols / 2) + k / 2];
    int code = (k & 1) ? (byte >> 4) : (byte & 15);
    return oracle_e2m1_value(code) * oracle_e4m3_value(sf[r * (cols / 16) + k / 16]) * (double)g;
}

/* ------------------------------------------------------------------ */
/* Scale-factor layout [SFL]                                           */
/* ------------------------------------------------------------------ */

/* Rows are padded to a multiple of 128 and scale columns (K/16) to a
 * multiple of 4.  The matrix is cut into 128 x 4 tiles of 512 bytes, stored
 * row-tile-major (all K tiles of rows 0..127 first).  Inside a tile, row r
 * and column c sit at (r % 32) * 16 + (r % 128) / 32 * 4 + c % 4. */
int64_t oracle_sf_padded_rows(int64_t rows) { return (rows + 127) / 128 * 128; }
int64_t oracle_sf_padded_cols(int64_t kb) { return (kb + 3) / 4 * 4; }

int64_t oracle_sf_offset(int64_t r, int64_t c, int64_t kb)
{
    int64_t kb_pad = oracle_sf_padded_cols(kb);
    int64_t tile = (r / 128) * (kb_pad / 4) + c / 4;
    return tile * 512 + (r % 32) * 16 + ((r % 128) / 32) * 4 + (c % 4);
}

/* logical [rows][kb] -> swizzled buffer of padded_rows * padded_cols bytes;
 * padding bytes are 0. */
void oracle_sf_swizzle(const uint8_t* logical, int64_t rows, int64_t kb, uint8_t* swz)
{
    memset(swz, 0, (size_t)(oracle_sf_padded_rows(rows) * oracle_sf_padded_cols(kb)));
    for (int64_t r = 0; r < rows; r++)
        for (int64_t c = 0; c < kb; c++)
            swz[oracle_sf_offset(r, c, kb)] = logical[r * kb + c];
}

void oracle_sf_unswizzle(const uint8_t* swz, int64_t rows, int64_t kb, uint8_t* logical)
{
    for (int64_t r = 0; r < rows; r++)
        for (int64_t c = 0; c < kb; c++)
            logical[r * kb + c] = swz[oracle_sf_offset(r, c, kb)];
}

/* ------------------------------------------------------------------ */
/* Block-scaled GEMM [GLU item 3]                                      */
/* ------------------------------------------------------------------ */

/* Each product term is e2m1_a * sf_a * e2m1_w * sf_w.  2*e2m1 is an integer
 * in [-12, 12] and 512*e4m3 an integer in [0, 229376], so with
 * qa = 2*e2m1_a*512*sf_a (|qa| < 2^22) the term times 2^20 is the integer
 * qa*qw (|.| < 2^43).  Summing in int64 is exact for K < 2^20. */
static int32_t exact_operand(const uint8_t* codes, const uint8_t* sf, int64_t cols, int64_t r, int64_t k)
{
    uint8_t byte = codes[r * (cols / 2) + k / 2];
    int code = (k & 1) ? (byte >> 4) : (byte & 15);
    double v = 2.0 * oracle_e2m1_value(code) * 512.0 * oracle_e4m3_value(sf[r * (cols / 16) + k / 16]);
    return (int32_t)v;   /* exact integer */
}

/* Exact dot products, sampled: for each (m, n) pair compute
 *     dot[i]  = sum_k a[m,k] * w[n,k]          (exact value, as binary64)
 *     adot[i] = sum_k |a[m,k] * w[n,k]|
 * with a, w the decoded values WITHOUT the global scales.  sf arrays are the
 * logical (unswizzled) scales. */
void oracle_dot_sampled(const uint8_t* a_codes, const uint8_t* a_sf,
                        const uint8_t* w_codes, const uint8_t* w_sf, int64_t K,
                        const int64_t* m_idx, const int64_t* n_idx, int64_t count,
                        double* dot, double* adot)
{
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < count; i++) {
        int64_t acc = 0, aacc = 0;
        for (int64_t k = 0; k < K; k++) {
            int64_t p = (int64_t)exact_operand(a_codes, a_sf, K, m_idx[i], k) *
                        (int64_t)exact_operand(w_codes, w_sf, K, n_idx[i], k);
            acc += p;
            aacc += p < 0 ? -p : p;
        }
        dot[i] = ldexp((double)acc, -20);
        adot[i] = ldexp((double)aacc, -20);
    }
}

/* Full GEMM: out[m][n] = alpha * dot(m, n) with alpha = fp32(g_a * g_w)
 * (reading: the two global scales are folded into one binary32 factor that
 * multiplies the accumulator once).  ref (binary64, may be NULL) receives
 * alpha*dot exactly as computed in binary64; absref (may be NULL) receives
 * alpha*sum|a w|; out_bf16 (may be NULL) receives bf16_RNE(alpha*dot), plus
 * a residual if residual != NULL: bf16_RNE(res + bf16_RNE(alpha*dot)).
 * Operands are pre-decoded to exact integers once per call. */
void oracle_gemm(const uint8_t* a_codes, const uint8_t* a_sf, float g_a,
                 const uint8_t* w_codes, const uint8_t* w_sf, float g_w,
                 int64_t M, int64_t N, int64_t K,
                 const uint16_t* residual, int64_t ldr,
                 double* ref, double* absref, uint16_t* out_bf16, int64_t ldo)
{
    int32_t* qa = (int32_t*)malloc(sizeof(int32_t) * (size_t)(M * K));
    int32_t* qw = (int32_t*)malloc(sizeof(int32_t) * (size_t)(N * K));
#pragma omp parallel for schedule(static)
    for (int64_t m = 0; m < M; m++)
        for (int64_t k = 0; k < K; k++) qa[m * K + k] = exact_operand(a_codes, a_sf, K, m, k);
#pragma omp parallel for schedule(static)
    for (int64_t n = 0; n < N; n++)
        for (int64_t k = 0; k < K; k++) qw[n * K + k] = exact_operand(w_codes, w_sf, K, n, k);
    float alpha = g_a * g_w;
#pragma omp parallel for schedule(static)
    for (int64_t m = 0; m < M; m++) {
        for (int64_t n = 0; n < N; n++) {
            int64_t acc = 0, aacc = 0;
            const int32_t* pa = qa + m * K;
            const int32_t* pw = qw + n * K;
            for (int64_t k = 0; k < K; k++) {
                int64_t p = (int64_t)pa[k] * (int64_t)pw[k];
                acc += p;
                aacc += p < 0 ? -p : p;
            }
            double v = (double)alpha * ldexp((double)acc, -20);
            if (ref) ref[m * N + n] = v;
            if (absref) absref[m * N + n] = (double)alpha * ldexp((double)aacc, -20);
            if (out_bf16) {
                uint16_t y = oracle_bf16_from_double(v);
                if (residual)
                    y = oracle_bf16_from_double(oracle_bf16_value(residual[m * ldr + n]) +
                                                oracle_bf16_value(y));
                out_bf16[m * ldo + n] = y;
            }
        }
    }
    free(qa);
    free(qw);
}

/* ------------------------------------------------------------------ */
/* RMSNorm [P8 item 2, GLU item 2 "batched-row rms_norm"]              */
/* ------------------------------------------------------------------ */

/* y = bf16_RNE( fp32( fp32(x * r) * w ) ),  r = 1 / sqrt(ms + eps) in
 * binary32, ms = mean(x^2) computed in binary64 and rounded once to binary32.
 * Reading: the norm weight multiplies as stored (not 1 + w); y is rounded to
 * bf16 before it is quantized, so norm+quantize equals norm then quantize. */
void oracle_rmsnorm(const uint16_t* x, int64_t rows, int64_t cols, int64_t ldx,
                    const uint16_t* w, float eps, uint16_t* y, int64_t ldy)
{
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; r++) {
        double ss = 0.0;
        for (int64_t c = 0; c < cols; c++) {
            double v = oracle_bf16_value(x[r * ldx + c]);
            ss += v * v;
        }
        float ms = (float)(ss / (double)cols);
        float rinv = 1.0f / sqrtf(ms + eps);
        for (int64_t c = 0; c < cols; c++) {
            float t = (float)oracle_bf16_value(x[r * ldx + c]) * rinv;
            float u = t * (float)oracle_bf16_value(w[c]);
            y[r * ldy + c] = oracle_bf16_from_double((double)u);
        }
    }
}

/* ------------------------------------------------------------------ */
/* SwiGLU [GLU item 2]                                                 */
/* ------------------------------------------------------------------ */

/* s = bf16_RNE( gate * sigmoid(gate) * up ) evaluated in binary64 from bf16
 * gate and up (reading: gate and up are the bf16 values an unfused GEMM
 * would store). */
uint16_t oracle_swiglu1(uint16_t gate, uint16_t up)
{
    double gv = oracle_bf16_value(gate), uv = oracle_bf16_value(up);
    return oracle_bf16_from_double(gv / (1.0 + exp(-gv)) * uv);
}

void oracle_swiglu(const uint16_t* gate, const uint16_t* up, int64_t n, uint16_t* s)
{
    for (int64_t i = 0; i < n; i++) s[i] = oracle_swiglu1(gate[i], up[i]);
}

/* ------------------------------------------------------------------ */
/* Rotary position embedding of projection output rows [ROPE]         */
/* ------------------------------------------------------------------ */

/* y: bf16 [rows x cols] (pitch ldy), e.g. the QKV GEMM output.  The `heads`
 * heads of head_dim columns starting at column col0 are rotated; every other
 * column is copied.  In a rotated head the first head_dim - rope_dim columns
 * are copied and the last rope_dim form rope_dim/2 pairs (e, o) = (x[2i],
 * x[2i+1]); with c = cos_t[pos[t]][i], s = sin_t[pos[t]][i] (tables of pitch
 * table_ld floats):
 *   forward: e' = e*c - o*s,  o' = e*s + o*c
 *   inverse: e' = e*c + o*s,  o' = o*c - e*s
 * each product, sum and difference one binary32 operation, e' and o' then
 * rounded to bf16 (RNE).
 * Reading: the tables are inputs (the page indexes cos and sin by position
 * and does not say how they are built). */
void oracle_rope(const uint16_t* y, int64_t rows, int64_t cols, int64_t ldy, const int32_t* pos,
                 const float* cos_t, const float* sin_t, int64_t table_ld, int64_t col0, int64_t heads,
                 int64_t head_dim, int64_t rope_dim, int inverse, uint16_t* out, int64_t ldo)
{
    for (int64_t t = 0; t < rows; t++) {
        for (int64_t c = 0; c < cols; c++) out[t * ldo + c] = y[t * ldy + c];
        const float* ct = cos_t + (int64_t)pos[t] * table_ld;
        const float* st = sin_t + (int64_t)pos[t] * table_ld;
        for (int64_t h = 0; h < heads; h++) {
            const int64_t base = col0 + h * head_dim + (head_dim - rope_dim);
            for (int64_t i = 0; i < rope_dim / 2; i++) {
                const float e = (float)oracle_bf16_value(y[t * ldy + base + 2 * i]);
                const float o = (float)oracle_bf16_value(y[t * ldy + base + 2 * i + 1]);
                const float c = ct[i], s = st[i];
                const float ec = e * c, os = o * s, es = e * s, oc = o * c;
                const float e2 = inverse ? ec + os : ec - os;
                const float o2 = inverse ? oc - es : es + oc;
                out[t * ldo + base + 2 * i] = oracle_bf16_from_double((double)e2);
                out[t * ldo + base + 2 * i + 1] = oracle_bf16_from_double((double)o2);
            }
        }
    }
}

/* ------------------------------------------------------------------ */
/* MLP block: RMSNorm -> quantize -> gate/up GEMMs -> SwiGLU -> requant  */
/*            -> down GEMM (+ residual)                                 */
/* ------------------------------------------------------------------ */

/* Inputs: x [T x H] bf16 (row pitch ldx), norm weight [H], quantized weights
 * (codes + LOGICAL scales + global scale) for gate [I x H], up [I x H],
 * down [H x I].  g_inter < 0 asks for the intermediate global scale to be
 * computed from this call's SwiGLU output (per-call scale); otherwise the
 * given value is used (a scale fixed ahead of time, as [P0] fix 1 keeps a
 * warm-up scale on the device).
 * Outputs: out [T x H] bf16 (= bf16(x + bf16(down))) when add_residual, else
 * bf16(down); optionally the stages (any pointer may be NULL):
 *   g_h_out (1), h_codes [T x H/2], h_sf [T x H/16], s_bf16 [T x I],
 *   g_inter_out (1), s_codes [T x I/2], s_sf [T x I/16]. */
void oracle_mlp(const uint16_t* x, int64_t T, int64_t H, int64_t I, int64_t ldx,
                const uint16_t* norm_w, float eps,
                const uint8_t* wg_codes, const uint8_t* wg_sf, float g_wg,
                const uint8_t* wu_codes, const uint8_t* wu_sf, float g_wu,
                const uint8_t* wd_codes, const uint8_t* wd_sf, float g_wd,
                float g_inter, int add_residual,
                uint16_t* out, int64_t ldo,
                float* g_h_out, uint8_t* h_codes_out, uint8_t* h_sf_out,
                uint16_t* s_out, float* g_inter_out, uint8_t* s_codes_out, uint8_t* s_sf_out)
{
    uint16_t* h = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)(T * H));
    uint8_t* hc = (uint8_t*)malloc((size_t)(T * H / 2));
    uint8_t* hs = (uint8_t*)malloc((size_t)(T * H / 16));
    uint16_t* gate = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)(T * I));
    uint16_t* up = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)(T * I));
    uint16_t* s = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)(T * I));
    uint8_t* sc = (uint8_t*)malloc((size_t)(T * I / 2));
    uint8_t* ss = (uint8_t*)malloc((size_t)(T * I / 16));
    uint16_t* dn = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)(T * H));

    oracle_rmsnorm(x, T, H, ldx, norm_w, eps, h, H);
    float g_h = oracle_global_scale(h, T, H, H);
    oracle_quantize(h, T, H, H, g_h, hc, hs);
    oracle_gemm(hc, hs, g_h, wg_codes, wg_sf, g_wg, T, I, H, NULL, 0, NULL, NULL, gate, I);
    oracle_gemm(hc, hs, g_h, wu_codes, wu_sf, g_wu, T, I, H, NULL, 0, NULL, NULL, up, I);
    oracle_swiglu(gate, up, T * I, s);
    float gi = g_inter < 0.0f ? oracle_global_scale(s, T, I, I) : g_inter;
    oracle_quantize(s, T, I, I, gi, sc, ss);
    oracle_gemm(sc, ss, gi, wd_codes, wd_sf, g_wd, T, H, I, NULL, 0, NULL, NULL, dn, H);
    for (int64_t t = 0; t < T; t++)
        for (int64_t c = 0; c < H; c++) {
            uint16_t v = dn[t * H + c];
            if (add_residual)
                v = oracle_bf16_from_double(oracle_bf16_value(x[t * ldx + c]) + oracle_bf16_value(v));
            out[t * ldo + c] = v;
        }

    if (g_h_out) *g_h_out = g_h;
    if (h_codes_out) memcpy(h_codes_out, hc, (size_t)(T * H / 2));
    if (h_sf_out) memcpy(h_sf_out, hs, (size_t)(T * H / 16));
    if (s_out) memcpy(s_out, s, sizeof(uint16_t) * (size_t)(T * I));
    if (g_inter_out) *g_inter_out = gi;
    if (s_codes_out) memcpy(s_codes_out, sc, (size_t)(T * I / 2));
    if (s_sf_out) memcpy(s_sf_out, ss, (size_t)(T * I / 16));
    free(h); free(hc); free(hs); free(gate); free(up); free(s); free(sc); free(ss); free(dn);
}

int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
