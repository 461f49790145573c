/*
 * Muon optimizer step -- CPU ORACLE.  TEST INFRASTRUCTURE ONLY.
 *
 * Only the test suite, the smoke check and the benchmark's CPU-baseline /
 * reference legs load this file's library.  The product (the CUDA library
 * under muon_newton_schulz_step_gb300/) never calls it and shares no code,
 * header, table or helper with it.
 *
 * What it computes: the per-matrix Muon step over whole matrices held on one
 * rank, as described in "How PyTorch Scaled a Near-1T MoE on Europe's Public
 * Supercomputer", section "Three optimizations that changed the economics",
 * FlexShard bullet (Muon's Newton-Schulz update works on full matrices; whole
 * experts are placed on one rank, so the orthogonalisation is local), with one
 * optimizer state per matrix ("Domyn is training a 1T-parameter MoE on
 * Europe's Jupiter supercomputer...", section "What moved the number": Muon
 * keeps one state where Adam keeps two).  The pages give none of the formulas;
 * the readings taken here are:
 *
 *   momentum      M' = fma(mu, M, g)                (fp32, one rounding)
 *   Nesterov      U  = fma(mu, M', g)               (fp32, one rounding)
 *   orientation   if rows > cols, work on U^T so that r = min <= k = max
 *   normalise     d = sqrt(sum U^2) (fp64) + eps;  sigma = (float)(1/d);
 *                 X0 = bf16(U *f32 sigma)
 *   Newton-Schulz for t in 1..steps, with (a, b, c) = (3.4445, -4.7750, 2.0315):
 *                 A  = bf16( X X^T )                 fp32 accumulation
 *                 B  = bf16( b*A + c*(A A) )         fp32 accumulation / epilogue
 *                 X  = bf16( a*X + B X )             fp32 accumulation / epilogue
 *   update        dcy = (float)(1 - lr*wd), s = (float)(lr*0.2*sqrt(max(m,n)))
 *                 (both in double, rounded once);
 *                 W' = round_W( fma(-s, O, dcy *f32 W) )
 *
 * Every product of two bf16 values is exact in fp32, so the only freedom in
 * the bf16-emulating mode is the order of the fp32 sums: this file sums each
 * output element over p in ascending order, one thread per output row, so the
 * result does not depend on the thread count.  A second mode does the same
 * steps in fp64 with no rounding at all (used to check the algorithm against
 * the closed form U p^5(s) V^T).
 *
 * Build:  gcc -O3 -fopenmp -ffp-contract=off -shared -fPIC  (see build.py).
 * -ffp-contract=off keeps every a*b+c above as a rounded product and a rounded
 * sum; the explicit fmaf calls are the only fused operations.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ---------------------------------------------------------------- bf16 --- */

/* Round an IEEE binary32 value to bfloat16 (the top 16 bits of binary32),
 * round-to-nearest, ties-to-even, written from the IEEE definition: look at
 * the 16 dropped bits; above half -> round up, exactly half -> round to the
 * even neighbour.  A carry out of the mantissa moves into the exponent, which
 * is the correct behaviour (including overflow to infinity).  NaN stays a
 * (quiet) NaN. */
uint16_t oracle_bf16_rne(float x)
{
    uint32_t u;
    memcpy(&u, &x, sizeof u);
    if ((u & 0x7f800000u) == 0x7f800000u && (u & 0x007fffffu) != 0u)
        return (uint16_t)((u >> 16) | 0x0040u);
    uint32_t hi = u >> 16;
    uint32_t lo = u & 0xffffu;
    if (lo > 0x8000u || (lo == 0x8000u && (hi & 1u)))
        hi += 1u;
    return (uint16_t)hi;
}

float oracle_bf16_to_f32(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* x rounded to the nearest bf16 value, returned as fp32 (exactly representable) */
static float rb(float x) { return oracle_bf16_to_f32(oracle_bf16_rne(x)); }

void oracle_bf16_rne_array(const float* x, uint16_t* out, int64_t n)
{
    for (int64_t e = 0; e < n; ++e) out[e] = oracle_bf16_rne(x[e]);
}

/* ---------------------------------------------------------------- e4m3 --- */

/* Round an IEEE binary32 value to FP8 E4M3 (1 sign bit, 4 exponent bits with
 * bias 7, 3 mantissa bits; no infinities; largest finite value 448 = 1.75 *
 * 2^8; S.1111.111 is NaN), written from that definition: round to nearest,
 * ties to even, on the grid of the value's binade (spacing 2^(e-3) for
 * 2^e <= |x| < 2^(e+1), e >= -6; spacing 2^-9 below 2^-6, the subnormals).
 * Magnitudes that round above 448 saturate to 448 (the saturating
 * conversion); NaN stays NaN.  Returns the 8-bit code. */
uint8_t oracle_e4m3_rne(float x)
{
    if (isnan(x)) return 0x7f;
    const uint8_t sign = signbit(x) ? 0x80 : 0x00;
    double a = fabs((double)x);
    if (a == 0.0) return sign;
    int e = (int)floor(log2(a));
    if (ldexp(1.0, e) > a) --e;              /* exact binade of a */
    if (ldexp(1.0, e + 1) <= a) ++e;
    if (e < -6) e = -6;                       /* subnormal grid */
    const double q = ldexp(1.0, e - 3);       /* spacing of the grid */
    double m = a / q;                         /* exact: a power-of-two division */
    double r = floor(m);
    const double frac = m - r;
    if (frac > 0.5 || (frac == 0.5 && fmod(r, 2.0) != 0.0)) r += 1.0;
    double v = r * q;
    if (v >= 448.0) return (uint8_t)(sign | 0x7e);     /* saturate to 448 */
    /* encode v: normal if v >= 2^-6 */
    if (v < ldexp(1.0, -6)) return (uint8_t)(sign | (uint8_t)(v / ldexp(1.0, -9)));
    int ev = (int)floor(log2(v));
    if (ldexp(1.0, ev) > v) --ev;
    if (ldexp(1.0, ev + 1) <= v) ++ev;
    const int mant = (int)(v / ldexp(1.0, ev - 3)) - 8;
    return (uint8_t)(sign | ((ev + 7) << 3) | mant);
}

float oracle_e4m3_to_f32(uint8_t v)
{
    const int sign = v & 0x80, ex = (v >> 3) & 0xf, mant = v & 7;
    if (ex == 0xf && mant == 7) return NAN;
    double a = ex == 0 ? ldexp((double)mant, -9) : ldexp(1.0 + mant / 8.0, ex - 7);
    return (float)(sign ? -a : a);
}

void oracle_e4m3_rne_array(const float* x, uint8_t* out, int64_t n)
{
    for (int64_t e = 0; e < n; ++e) out[e] = oracle_e4m3_rne(x[e]);
}

/* Scale of the FP8 Gram operands: X * 2^8, a fixed power of two (exact).
 * Every element of every iterate is at most its largest singular value:
 * X0 has Frobenius norm 1, and each iteration maps a singular value s in
 * [0, 1.21] to p(s) = a s + b s^3 + c s^5 <= 1.2024 (the quintic's maximum,
 * at s ~ 0.5545), so |X| stays below 1.21 and |X| * 2^8 below 310, inside
 * E4M3's range (448).  A larger value would saturate (RNE, saturating). */
#define ORACLE_FP8_SCALE_EXP 8

/* ------------------------------------------------------------ momentum --- */

/* Heavy-ball momentum with an optional Nesterov look-ahead, one fp32 fma each:
 * M'[e] = fma(mu, M[e], g[e]);  U[e] = fma(mu, M'[e], g[e])  (or U = M'). */
void oracle_momentum(const float* g, float* M, float* U, int64_t n, float mu, int nesterov)
{
    for (int64_t e = 0; e < n; ++e) {
        const float mp = fmaf(mu, M[e], g[e]);
        M[e] = mp;
        U[e] = nesterov ? fmaf(mu, mp, g[e]) : mp;
    }
}

/* ---------------------------------------------- gradient accumulation --- */

/* Sum of K stacked gradients (bf16 bits or fp32), each n elements, in fp32:
 * g = G_0, then g = g + G_j for j = 1 .. K-1, every add rounded once (this is
 * "sending bf16 over the wire and summing in fp32 locally" from "Training a
 * trillion-parameter AI on the GPUs powering Europe's fastest supercomputer"). */
void oracle_grad_sum(const void* G, int g_bf16, int64_t n, int K, float* g)
{
    for (int64_t e = 0; e < n; ++e) {
        float acc = 0.0f;
        for (int j = 0; j < K; ++j) {
            const int64_t idx = (int64_t)j * n + e;
            const float v = g_bf16 ? oracle_bf16_to_f32(((const uint16_t*)G)[idx]) : ((const float*)G)[idx];
            acc = (j == 0) ? v : acc + v;
        }
        g[e] = acc;
    }
}

/* ------------------------------------------------------ plain products --- */

/* Order of the fp32 running sums.  The pages fix none; ascending p is the
 * oracle's reading.  Descending p is an equally valid reading, selectable only
 * to measure how far a legal change of summation order alone moves a result
 * (the conditioning of an input), never to compare against the GPU. */
static int g_sum_descending = 0;

void oracle_set_sum_order(int descending) { g_sum_descending = descending != 0; }

/* C (M x N) = A (M x K) * B (K x N), all row-major fp32.  Each C[i][j] is an
 * fp32 running sum over p = 0, 1, ..., K-1 (or K-1, ..., 0 in the descending
 * order) of the fp32 product A[i][p]*B[p][j]. */
static void mm_f32(const float* A, const float* B, float* C, int M, int K, int N)
{
    const int desc = g_sum_descending;
#pragma omp parallel for schedule(static)
    for (int i = 0; i < M; ++i) {
        float* c = C + (size_t)i * N;
        for (int j = 0; j < N; ++j) c[j] = 0.0f;
        const float* a = A + (size_t)i * K;
        for (int q = 0; q < K; ++q) {
            const int p = desc ? K - 1 - q : q;
            const float aip = a[p];
            const float* b = B + (size_t)p * N;
            for (int j = 0; j < N; ++j) {
                const float prod = aip * b[j];
                c[j] = c[j] + prod;
            }
        }
    }
}

/* The same product in fp64, no rounding beyond fp64's own. */
static void mm_f64(const double* A, const double* B, double* C, int M, int K, int N)
{
#pragma omp parallel for schedule(static)
    for (int i = 0; i < M; ++i) {
        double* c = C + (size_t)i * N;
        for (int j = 0; j < N; ++j) c[j] = 0.0;
        const double* a = A + (size_t)i * K;
        for (int p = 0; p < K; ++p) {
            const double aip = a[p];
            const double* b = B + (size_t)p * N;
            for (int j = 0; j < N; ++j) c[j] = c[j] + aip * b[j];
        }
    }
}

/* ------------------------------------------------------ Newton-Schulz --- */

/* Newton-Schulz orthogonalisation of one m x n fp32 matrix U (row-major),
 * emulating bf16 storage of X, A and B with fp32 accumulation.  Output O is
 * m x n fp32 holding bf16-exact values.  Returns 0, or -1 on a bad argument /
 * allocation failure. */
/* Gram product of the FP8 variant (see oracle_ns_bf16_sched_fp8). */
static int g_fp8_gram = 0;

int oracle_ns_bf16_sched(const float* U, int m, int n, int steps,
                         const float* abc, double eps, float* O)
{
    if (m <= 0 || n <= 0 || steps < 0) return -1;
    const int trans = m > n;
    const int r = trans ? n : m;
    const int k = trans ? m : n;
    const size_t rk = (size_t)r * k, rr = (size_t)r * r;

    float* X  = (float*)malloc(rk * sizeof(float));
    float* XT = (float*)malloc(rk * sizeof(float));
    float* A  = (float*)malloc(rr * sizeof(float));
    float* Bm = (float*)malloc(rr * sizeof(float));
    float* S  = (float*)malloc((rk > rr ? rk : rr) * sizeof(float));
    if (!X || !XT || !A || !Bm || !S) {
        free(X); free(XT); free(A); free(Bm); free(S);
        return -1;
    }

    /* orientation: X holds U (r x k), transposed when the matrix is tall */
    for (int i = 0; i < r; ++i)
        for (int j = 0; j < k; ++j)
            X[(size_t)i * k + j] = trans ? U[(size_t)j * n + i] : U[(size_t)i * n + j];

    /* Frobenius normalisation */
    double ss = 0.0;
    for (size_t e = 0; e < rk; ++e) ss += (double)X[e] * (double)X[e];
    const double d = sqrt(ss) + eps;
    const float sigma = (float)(1.0 / d);
    for (size_t e = 0; e < rk; ++e) X[e] = rb(X[e] * sigma);

    for (int t = 0; t < steps; ++t) {
        const float a = abc[3 * t], b = abc[3 * t + 1], c = abc[3 * t + 2];
        /* A = X X^T */
        if (!g_fp8_gram) {
            for (int i = 0; i < r; ++i)
                for (int j = 0; j < k; ++j)
                    XT[(size_t)j * r + i] = X[(size_t)i * k + j];
            mm_f32(X, XT, S, r, k, r);
            for (size_t e = 0; e < rr; ++e) A[e] = rb(S[e]);
        } else {
            /* FP8 variant: A = bf16( 2^-2s * sum_p q(2^s X[i][p]) q(2^s X[j][p]) ),
             * q = E4M3 rounding, s = ORACLE_FP8_SCALE_EXP; products of two E4M3
             * values are exact in fp32, the sum runs in fp32 */
            const int sx = ORACLE_FP8_SCALE_EXP;
            for (int i = 0; i < r; ++i)
                for (int j = 0; j < k; ++j) {
                    const float qv = oracle_e4m3_to_f32(oracle_e4m3_rne(ldexpf(X[(size_t)i * k + j], sx)));
                    XT[(size_t)j * r + i] = qv;
                }
            float* XQ = (float*)malloc(rk * sizeof(float));
            if (!XQ) { free(X); free(XT); free(A); free(Bm); free(S); return -1; }
            for (int i = 0; i < r; ++i)
                for (int j = 0; j < k; ++j) XQ[(size_t)i * k + j] = XT[(size_t)j * r + i];
            mm_f32(XQ, XT, S, r, k, r);
            free(XQ);
            for (size_t e = 0; e < rr; ++e) A[e] = rb(ldexpf(S[e], -2 * sx));
        }

        /* B = b A + c A A */
        mm_f32(A, A, S, r, r, r);
        for (size_t e = 0; e < rr; ++e) {
            const float lin = b * A[e];
            const float quad = c * S[e];
            Bm[e] = rb(lin + quad);
        }

        /* X = a X + B X */
        mm_f32(Bm, X, S, r, r, k);
        for (size_t e = 0; e < rk; ++e) {
            const float lin = a * X[e];
            X[e] = rb(lin + S[e]);
        }
    }

    for (int i = 0; i < r; ++i)
        for (int j = 0; j < k; ++j) {
            const float v = X[(size_t)i * k + j];
            if (trans) O[(size_t)j * n + i] = v; else O[(size_t)i * n + j] = v;
        }

    free(X); free(XT); free(A); free(Bm); free(S);
    return 0;
}

/* The FP8 variant of the Newton-Schulz iteration: identical except that the
 * Gram product's operands are X rounded to FP8 E4M3 after the exact scaling by
 * 2^8, A = bf16(2^-16 sum_p q(2^8 X) q(2^8 X)^T) in fp32 accumulation.  The
 * polynomial and the update stay in bf16. */
int oracle_ns_bf16_sched_fp8(const float* U, int m, int n, int steps,
                             const float* abc, double eps, float* O)
{
    g_fp8_gram = 1;
    const int rc = oracle_ns_bf16_sched(U, m, n, steps, abc, eps, O);
    g_fp8_gram = 0;
    return rc;
}

/* Newton-Schulz with one (a, b, c) triple used at every step. */
int oracle_ns_bf16(const float* U, int m, int n, int steps,
                   float a, float b, float c, double eps, float* O)
{
    if (steps < 0) return -1;
    float* abc = (float*)malloc((size_t)(steps > 0 ? steps : 1) * 3 * sizeof(float));
    if (!abc) return -1;
    for (int t = 0; t < steps; ++t) { abc[3 * t] = a; abc[3 * t + 1] = b; abc[3 * t + 2] = c; }
    const int rc = oracle_ns_bf16_sched(U, m, n, steps, abc, eps, O);
    free(abc);
    return rc;
}

/* The same algorithm entirely in fp64 with no rounding to bf16 (X0 = U/d);
 * abc holds one (a, b, c) triple per step. */
int oracle_ns_f64_sched(const double* U, int m, int n, int steps,
                        const double* abc, double eps, double* O)
{
    if (m <= 0 || n <= 0 || steps < 0) return -1;
    const int trans = m > n;
    const int r = trans ? n : m;
    const int k = trans ? m : n;
    const size_t rk = (size_t)r * k, rr = (size_t)r * r;

    double* X  = (double*)malloc(rk * sizeof(double));
    double* XT = (double*)malloc(rk * sizeof(double));
    double* A  = (double*)malloc(rr * sizeof(double));
    double* Bm = (double*)malloc(rr * sizeof(double));
    double* S  = (double*)malloc((rk > rr ? rk : rr) * sizeof(double));
    if (!X || !XT || !A || !Bm || !S) {
        free(X); free(XT); free(A); free(Bm); free(S);
        return -1;
    }

    for (int i = 0; i < r; ++i)
        for (int j = 0; j < k; ++j)
            X[(size_t)i * k + j] = trans ? U[(size_t)j * n + i] : U[(size_t)i * n + j];

    double ss = 0.0;
    for (size_t e = 0; e < rk; ++e) ss += X[e] * X[e];
    const double d = sqrt(ss) + eps;
    for (size_t e = 0; e < rk; ++e) X[e] = X[e] / d;

    for (int t = 0; t < steps; ++t) {
        const double a = abc[3 * t], b = abc[3 * t + 1], c = abc[3 * t + 2];
        for (int i = 0; i < r; ++i)
            for (int j = 0; j < k; ++j)
                XT[(size_t)j * r + i] = X[(size_t)i * k + j];
        mm_f64(X, XT, A, r, k, r);
        mm_f64(A, A, S, r, r, r);
        for (size_t e = 0; e < rr; ++e) Bm[e] = b * A[e] + c * S[e];
        mm_f64(Bm, X, S, r, r, k);
        for (size_t e = 0; e < rk; ++e) X[e] = a * X[e] + S[e];
    }

    for (int i = 0; i < r; ++i)
        for (int j = 0; j < k; ++j) {
            const double v = X[(size_t)i * k + j];
            if (trans) O[(size_t)j * n + i] = v; else O[(size_t)i * n + j] = v;
        }

    free(X); free(XT); free(A); free(Bm); free(S);
    return 0;
}

int oracle_ns_f64(const double* U, int m, int n, int steps,
                  double a, double b, double c, double eps, double* O)
{
    if (steps < 0) return -1;
    double* abc = (double*)malloc((size_t)(steps > 0 ? steps : 1) * 3 * sizeof(double));
    if (!abc) return -1;
    for (int t = 0; t < steps; ++t) { abc[3 * t] = a; abc[3 * t + 1] = b; abc[3 * t + 2] = c; }
    const int rc = oracle_ns_f64_sched(U, m, n, steps, abc, eps, O);
    free(abc);
    return rc;
}

/* -------------------------------------------------------- weight update --- */

/* Host-side scalars of the decoupled-weight-decay update, computed in double
 * and rounded to fp32 once: dcy = 1 - lr*wd,  s = lr * 0.2 * sqrt(max(m, n)). */
void oracle_update_scalars(float lr, float wd, int m, int n, float* dcy, float* s)
{
    const int mx = m > n ? m : n;
    *dcy = (float)(1.0 - (double)lr * (double)wd);
    *s = (float)((double)lr * 0.2 * sqrt((double)mx));
}

/* W' = fma(-s, O, dcy*W) with W in fp32. */
void oracle_weight_update_f32(float* W, const float* O, int64_t n, float dcy, float s)
{
    for (int64_t e = 0; e < n; ++e) {
        const float decayed = dcy * W[e];
        W[e] = fmaf(-s, O[e], decayed);
    }
}

/* W' = bf16(fma(-s, O, dcy*W)) with W held as bf16 bit patterns. */
void oracle_weight_update_bf16(uint16_t* W, const float* O, int64_t n, float dcy, float s)
{
    for (int64_t e = 0; e < n; ++e) {
        const float decayed = dcy * oracle_bf16_to_f32(W[e]);
        W[e] = oracle_bf16_rne(fmaf(-s, O[e], decayed));
    }
}

/* ---------------------------------------------------------------- AdamW --- */

/* AdamW for the parameters Muon does not cover ("Domyn is training a
 * 1T-parameter MoE...", table "The model and the machine": Muon for about
 * 99.5% of parameters, AdamW for the rest).  Decoupled weight decay, bias
 * correction; host scalars in double rounded once to fp32:
 *   b1c = 1 - beta1, b2c = 1 - beta2, dcy = 1 - lr*wd,
 *   step_size = lr / (1 - beta1^t), inv_sqrt_bc2 = 1 / sqrt(1 - beta2^t)
 * per element, every operation one IEEE fp32 rounding:
 *   m' = fma(beta1, m, b1c*g)
 *   v' = fma(beta2, v, b2c*(g*g))
 *   denom = sqrt(v') * inv_sqrt_bc2 + eps
 *   p' = round_P( fma(-step_size, m' / denom, dcy * p) )                  */
void oracle_adamw_scalars(float lr, float beta1, float beta2, float wd, int step, float* out5)
{
    const double t = (double)step;
    out5[0] = (float)(1.0 - (double)beta1);
    out5[1] = (float)(1.0 - (double)beta2);
    out5[2] = (float)(1.0 - (double)lr * (double)wd);
    out5[3] = (float)((double)lr / (1.0 - pow((double)beta1, t)));
    out5[4] = (float)(1.0 / sqrt(1.0 - pow((double)beta2, t)));
}

void oracle_adamw(void* P, int p_bf16, const void* G, int g_bf16, float* Mo, float* V, int64_t n,
                  float lr, float beta1, float beta2, float eps, float wd, int step)
{
    float s[5];
    oracle_adamw_scalars(lr, beta1, beta2, wd, step, s);
    const float b1c = s[0], b2c = s[1], dcy = s[2], step_size = s[3], inv_sqrt_bc2 = s[4];
    for (int64_t e = 0; e < n; ++e) {
        const float g = g_bf16 ? oracle_bf16_to_f32(((const uint16_t*)G)[e]) : ((const float*)G)[e];
        const float p = p_bf16 ? oracle_bf16_to_f32(((const uint16_t*)P)[e]) : ((float*)P)[e];
        const float gm = b1c * g;
        const float m = fmaf(beta1, Mo[e], gm);
        const float gg = g * g;
        const float gv = b2c * gg;
        const float v = fmaf(beta2, V[e], gv);
        const float root = sqrtf(v);
        const float scaled = root * inv_sqrt_bc2;
        const float denom = scaled + eps;
        const float ratio = m / denom;
        const float decayed = dcy * p;
        const float np = fmaf(-step_size, ratio, decayed);
        Mo[e] = m;
        V[e] = v;
        if (p_bf16) ((uint16_t*)P)[e] = oracle_bf16_rne(np);
        else ((float*)P)[e] = np;
    }
}

/* ---------------------------------------------------------- full step --- */

/* One Muon step on one m x n matrix.
 *   W: fp32 (w_bf16 = 0) or bf16 bits (w_bf16 = 1), updated in place
 *   G: fp32 (g_bf16 = 0) or bf16 bits (g_bf16 = 1)
 *   M: fp32 momentum, updated in place
 *   O_out: optional m x n fp32 copy of the orthogonalised update (bf16-exact)
 * Returns 0 or -1. */
int oracle_muon_step(void* W, int w_bf16, const void* G, int g_bf16, float* M,
                     int m, int n, float lr, float mu, float wd, int nesterov,
                     int steps, float a, float b, float c, double eps, float* O_out)
{
    if (m <= 0 || n <= 0) return -1;
    const int64_t mn = (int64_t)m * n;
    float* g = (float*)malloc((size_t)mn * sizeof(float));
    float* U = (float*)malloc((size_t)mn * sizeof(float));
    float* O = (float*)malloc((size_t)mn * sizeof(float));
    if (!g || !U || !O) { free(g); free(U); free(O); return -1; }

    for (int64_t e = 0; e < mn; ++e)
        g[e] = g_bf16 ? oracle_bf16_to_f32(((const uint16_t*)G)[e]) : ((const float*)G)[e];
    oracle_momentum(g, M, U, mn, mu, nesterov);
    int rc = oracle_ns_bf16(U, m, n, steps, a, b, c, eps, O);
    if (rc == 0) {
        float dcy, s;
        oracle_update_scalars(lr, wd, m, n, &dcy, &s);
        if (w_bf16) oracle_weight_update_bf16((uint16_t*)W, O, mn, dcy, s);
        else        oracle_weight_update_f32((float*)W, O, mn, dcy, s);
        if (O_out) memcpy(O_out, O, (size_t)mn * sizeof(float));
    }
    free(g); free(U); free(O);
    return rc;
}

int oracle_num_threads(void)
{
#ifdef _OPENMP
    extern int omp_get_max_threads(void);
    return omp_get_max_threads();
#else
    return 1;
#endif
}
