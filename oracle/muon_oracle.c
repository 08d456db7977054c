/*
 * Oracle for the Muon optimizer step and the AdamW step.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is a plain, slow, deliberately
 * unoptimised CPU restatement of what the GPU library computes.  Only the
 * test suite, the smoke check and the benchmark's CPU-baseline leg may load
 * it.  It shares no code, header, table or helper with the CUDA library, and
 * it never reads anything the CUDA library produced.
 *
 * Sources, cited by page title and section:
 *   [OPT]  "LLM training series, part 2: optimizers (SGD -> Adam -> AdamW ->
 *          Muon)", mhpq.cn article.  Section numbers are the article's own.
 *   [K2]   "Kimi K2 ... what is worth noting" (Zhihu answer by toothacher17).
 *          Section numbers are the answer's own.
 * Quantities the pages leave open (the quintic coefficients, the Nesterov
 * form, the 0.2*sqrt(max(m,n)) update scale, the 1e-7 norm epsilon) are the
 * values this library is specified to use; each reading is stated where used.
 *
 * Arithmetic conventions (the same ones the library documents):
 *   - every scalar the method names (lr, mu, beta, ...) is an IEEE fp32 value;
 *   - element-wise formulas are evaluated as separately rounded fp32
 *     operations in the order written next to them (build with
 *     -ffp-contract=off so no multiply-add is fused);
 *   - every matrix product is accumulated in fp64 in ascending k order, then
 *     rounded once to fp32; bf16 rounding is round-to-nearest-even of that
 *     fp32 value (see oracle_bf16_from_f32).
 *   - variants exist only to measure how far equally faithful bf16
 *     evaluations of the step lie apart (the iteration is not unique once
 *     it is rounded): products accumulated in fp32 instead of fp64, either
 *     one rounded-to-nearest addition per product (ACC_FP32) or blocks of 16
 *     products added to the fp32 sum with one round-toward-zero each
 *     (ACC_FP32_RZ16, the way tensor-core fp32 accumulation behaves in
 *     measurement); and the cast to bf16 taken after the normalisation
 *     instead of before it (cast_after_scale).  The pages fix none of these
 *     choices.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------------ */
/* bf16 encoding                                                             */
/* ------------------------------------------------------------------------ */

/* bf16 keeps the top 16 bits of an fp32 word (sign, 8 exponent bits, 7
 * mantissa bits).  Round-to-nearest-even by definition: look at the 16
 * dropped bits; above half -> round up, below half -> round down, exactly
 * half -> round to the candidate whose last kept bit is 0.  NaN stays NaN
 * (quiet bit forced), +-inf stays inf. */
uint16_t oracle_bf16_from_f32(float x)
{
    uint32_t bits;
    memcpy(&bits, &x, sizeof bits);
    uint32_t exponent = (bits >> 23) & 0xffu;
    uint32_t mantissa = bits & 0x7fffffu;
    if (exponent == 0xffu) {
        if (mantissa != 0)
            return (uint16_t)((bits >> 16) | 0x40u);
        return (uint16_t)(bits >> 16);
    }
    uint32_t kept = bits >> 16;
    uint32_t dropped = bits & 0xffffu;
    if (dropped > 0x8000u || (dropped == 0x8000u && (kept & 1u)))
        kept += 1u; /* a carry into the exponent is the correct result */
    return (uint16_t)kept;
}

float oracle_f32_from_bf16(uint16_t h)
{
    uint32_t bits = (uint32_t)h << 16;
    float x;
    memcpy(&x, &bits, sizeof x);
    return x;
}

static float bf16_round(float x)
{
    return oracle_f32_from_bf16(oracle_bf16_from_f32(x));
}

void oracle_bf16_encode(const float* x, uint16_t* out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = oracle_bf16_from_f32(x[i]);
}

/* ------------------------------------------------------------------------ */
/* Plain matrix product, fp64 accumulation                                   */
/* ------------------------------------------------------------------------ */

/* C[i][j] = sum_{k=0}^{K-1} A[i][k] * B[k][j], A is MxK, B is KxN, all
 * row-major fp64.  Each C[i][j] is summed in ascending k with one fp64
 * rounding per multiply and per add.  The loops run i, k, j only so the j
 * loop reads B row-wise; that does not change any element's summation
 * order.  Rows are independent and may run on several threads. */
static void matmul_f64(const double* A, const double* B, double* C,
                       int64_t M, int64_t K, int64_t N)
{
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < M; ++i) {
        double* c = C + i * N;
        for (int64_t j = 0; j < N; ++j)
            c[j] = 0.0;
        for (int64_t k = 0; k < K; ++k) {
            double a = A[i * K + k];
            const double* b = B + k * N;
            for (int64_t j = 0; j < N; ++j)
                c[j] += a * b[j];
        }
    }
}

/* The same product with each C[i][j] accumulated in fp32 instead: in
 * ascending k, every product a*b rounded to fp32 and every partial sum
 * rounded to fp32 (for bf16 operands the products are exact in fp32; only
 * the additions round).  The result is stored as the fp64 value of that
 * fp32 sum. */
static void matmul_f32acc(const double* A, const double* B, double* C,
                          int64_t M, int64_t K, int64_t N)
{
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < M; ++i) {
        float* c = (float*)malloc(sizeof(float) * (N > 0 ? N : 1));
        for (int64_t j = 0; j < N; ++j)
            c[j] = 0.0f;
        for (int64_t k = 0; k < K; ++k) {
            const float a = (float)A[i * K + k];
            const double* b = B + k * N;
            for (int64_t j = 0; j < N; ++j) {
                const float prod = a * (float)b[j];
                c[j] = c[j] + prod;
            }
        }
        for (int64_t j = 0; j < N; ++j)
            C[i * N + j] = (double)c[j];
        free(c);
    }
}

/* x rounded to fp32 toward zero: the nearest-rounded fp32 value, moved one
 * step towards zero when it lies farther from zero than x. */
static float f32_toward_zero(double x)
{
    float f = (float)x;
    if (fabs((double)f) > fabs(x))
        f = nextafterf(f, 0.0f);
    return f;
}

/* The same product accumulated block-wise: the products of each run of 16
 * consecutive k (ascending; the last run may be shorter) are summed in
 * fp64, and each run's sum is added to the fp32 accumulator with one
 * rounding toward zero, acc = rz32(acc + run).  For bf16 operands the fp64
 * run sums are exact unless a run's products span more than 37 binades. */
static void matmul_f32rz16(const double* A, const double* B, double* C,
                           int64_t M, int64_t K, int64_t N)
{
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < M; ++i) {
        float* c = (float*)malloc(sizeof(float) * (N > 0 ? N : 1));
        double* run = (double*)malloc(sizeof(double) * (N > 0 ? N : 1));
        for (int64_t j = 0; j < N; ++j)
            c[j] = 0.0f;
        for (int64_t k0 = 0; k0 < K; k0 += 16) {
            const int64_t k1 = k0 + 16 < K ? k0 + 16 : K;
            for (int64_t j = 0; j < N; ++j)
                run[j] = 0.0;
            for (int64_t k = k0; k < k1; ++k) {
                const double a = A[i * K + k];
                const double* b = B + k * N;
                for (int64_t j = 0; j < N; ++j)
                    run[j] += a * b[j];
            }
            for (int64_t j = 0; j < N; ++j)
                c[j] = f32_toward_zero((double)c[j] + run[j]);
        }
        for (int64_t j = 0; j < N; ++j)
            C[i * N + j] = (double)c[j];
        free(run);
        free(c);
    }
}

/* Accumulation modes of the products (see the header). */
enum { ACC_FP64 = 0, ACC_FP32 = 1, ACC_FP32_RZ16 = 2 };

static void matmul(const double* A, const double* B, double* C,
                   int64_t M, int64_t K, int64_t N, int acc)
{
    if (acc == ACC_FP32)
        matmul_f32acc(A, B, C, M, K, N);
    else if (acc == ACC_FP32_RZ16)
        matmul_f32rz16(A, B, C, M, K, N);
    else
        matmul_f64(A, B, C, M, K, N);
}

/* C = A B (M x K times K x N, row-major fp64 arrays), accumulated as `acc`
 * says: 0 fp64, 1 fp32 one rounding per addition, 2 fp32 round-toward-zero
 * per 16-product block. */
void oracle_matmul(const double* A, const double* B, double* C,
                   int64_t M, int64_t K, int64_t N, int acc)
{
    matmul(A, B, C, M, K, N, acc);
}

static void transpose_f64(const double* X, double* XT, int64_t R, int64_t C)
{
    for (int64_t r = 0; r < R; ++r)
        for (int64_t c = 0; c < C; ++c)
            XT[c * R + r] = X[r * C + c];
}

/* ------------------------------------------------------------------------ */
/* Newton-Schulz orthogonalisation                                           */
/* ------------------------------------------------------------------------ */

/* One odd matrix polynomial applied `steps` times to a wide X (rows <= cols),
 * step s with its own coefficients (a, b, c) = coeffs[3s .. 3s+2]:
 *     A  = X X^T
 *     B  = b A + c A A
 *     X <- a X + B X
 * [OPT] section 4.2 gives the iteration's purpose and the cubic member
 * X <- (3X - X X^T X)/2, i.e. (a,b,c) = (1.5, -0.5, 0); the library's
 * default is the quintic (a,b,c) = (3.4445, -4.7750, 2.0315), 5 steps.
 *
 * X is rows x cols, row-major, overwritten with the result.  The iteration's
 * input is x_scale * X: the scale is applied inside the first step (below),
 * never to a stored X, so X keeps the values it was given (bf16 values when
 * emulating).
 * emulate_bf16 != 0: the GPU's storage points are reproduced: A, B and the
 *   new X are each rounded fp64 -> fp32 -> bf16 once per step, and the
 *   epilogues are fp32 with s = x_scale on the first step, s = 1 after:
 *       A = bf16( fl32(fl32(s*s) * float(X X^T)) )
 *       B = bf16( fl32(b*A) + fl32(c*float(A A)) )
 *       X = bf16( fl32(fl32(a*s)*X) + fl32(s*float(B X)) )
 *   (a factor of 1 is exact, so later steps are the plain iteration).  With
 *   no steps the result is bf16( fl32(x_scale * X) ).
 * emulate_bf16 == 0: everything stays in fp64 (used to check the iteration
 *   against its singular-value closed form).
 * acc != 0 (with emulate_bf16 only): the three products are accumulated
 *   in fp32 (1: matmul_f32acc, 2: matmul_f32rz16) instead of fp64; the
 *   spread variants. */
int oracle_newton_schulz_ex(double* X, int64_t rows, int64_t cols, int steps,
                            const float* coeffs, int emulate_bf16, float x_scale, int acc)
{
    if (acc < 0 || acc > 2 || (acc && !emulate_bf16))
        return 1;
    if (rows <= 0 || cols <= 0 || steps < 0 || rows > cols || (steps > 0 && !coeffs))
        return 1;
    if (steps == 0) {
        for (int64_t i = 0; i < rows * cols; ++i)
            X[i] = emulate_bf16 ? bf16_round(x_scale * (float)X[i]) : (double)x_scale * X[i];
        return 0;
    }
    double* XT = (double*)malloc(sizeof(double) * rows * cols);
    double* A = (double*)malloc(sizeof(double) * rows * rows);
    double* AA = (double*)malloc(sizeof(double) * rows * rows);
    double* Bm = (double*)malloc(sizeof(double) * rows * rows);
    double* BX = (double*)malloc(sizeof(double) * rows * cols);
    if (!XT || !A || !AA || !Bm || !BX) {
        free(XT); free(A); free(AA); free(Bm); free(BX);
        return 2;
    }
    for (int s = 0; s < steps; ++s) {
        const float a = coeffs[3 * s], b = coeffs[3 * s + 1], c = coeffs[3 * s + 2];
        const float xs = s == 0 ? x_scale : 1.0f;  /* input scale, first step only */
        /* A = (xs X)(xs X)^T */
        transpose_f64(X, XT, rows, cols);
        matmul(X, XT, A, rows, cols, rows, acc);
        if (emulate_bf16) {
            const float xs2 = xs * xs;
            for (int64_t i = 0; i < rows * rows; ++i)
                A[i] = bf16_round(xs2 * (float)A[i]);
        } else {
            for (int64_t i = 0; i < rows * rows; ++i)
                A[i] *= (double)xs * (double)xs;
        }
        /* B = b A + c A A */
        matmul(A, A, AA, rows, rows, rows, acc);
        for (int64_t i = 0; i < rows * rows; ++i) {
            if (emulate_bf16) {
                float t1 = b * (float)A[i];
                float t2 = c * (float)AA[i];
                Bm[i] = bf16_round(t1 + t2);
            } else {
                Bm[i] = (double)b * A[i] + (double)c * AA[i];
            }
        }
        /* X = a (xs X) + B (xs X) */
        matmul(Bm, X, BX, rows, rows, cols, acc);
        const float axs = a * xs;
        for (int64_t i = 0; i < rows * cols; ++i) {
            if (emulate_bf16) {
                float t1 = axs * (float)X[i];
                float t2 = xs * (float)BX[i];
                X[i] = bf16_round(t1 + t2);
            } else {
                X[i] = (double)a * (double)xs * X[i] + (double)xs * BX[i];
            }
        }
    }
    free(XT); free(A); free(AA); free(Bm); free(BX);
    return 0;
}

int oracle_newton_schulz_scaled(double* X, int64_t rows, int64_t cols, int steps,
                                const float* coeffs, int emulate_bf16, float x_scale)
{
    return oracle_newton_schulz_ex(X, rows, cols, steps, coeffs, emulate_bf16, x_scale, 0);
}

/* The iteration on X itself (input scale 1). */
int oracle_newton_schulz_table(double* X, int64_t rows, int64_t cols, int steps,
                               const float* coeffs, int emulate_bf16)
{
    return oracle_newton_schulz_scaled(X, rows, cols, steps, coeffs, emulate_bf16, 1.0f);
}

/* The same iteration with one coefficient triple for every step. */
int oracle_newton_schulz(double* X, int64_t rows, int64_t cols, int steps,
                         float a, float b, float c, int emulate_bf16)
{
    if (steps < 0 || steps > 100)
        return 1;
    float table[300];
    for (int s = 0; s < steps; ++s) {
        table[3 * s] = a;
        table[3 * s + 1] = b;
        table[3 * s + 2] = c;
    }
    return oracle_newton_schulz_table(X, rows, cols, steps, table, emulate_bf16);
}

/* ------------------------------------------------------------------------ */
/* Muon step for one matrix                                                  */
/* ------------------------------------------------------------------------ */

typedef struct {
    float lr;           /* learning rate                                    */
    float weight_decay; /* decoupled weight decay                           */
    float momentum;     /* mu                                               */
    int nesterov;       /* 1: Nesterov look-ahead, 0: plain EMA momentum    */
    int ns_steps;       /* Newton-Schulz steps                              */
    float ns_a, ns_b, ns_c;
    float norm_eps;     /* added to the Frobenius norm                      */
    float rms_scale;    /* update scale = rms_scale * sqrt(max(rows, cols)) */
    int scale_mode;     /* 0: rms_scale * sqrt(max(rows, cols));
                           1: max(1, sqrt(rows / cols))                     */
    int skip_nonfinite; /* used by the multi-matrix step (Python side)      */
    float max_grad_norm;/* used by the multi-matrix step (Python side)      */
    int reserved;
    const float* ns_coeffs; /* NULL, or 3 * ns_steps per-step coefficients  */
} oracle_muon_hparams;

/* Steps 1-2 of the Muon step, element by element, in place on M.  With
 * scale_g != 0 the gradient is first multiplied by g_scale in fp32 (the
 * global-norm clip factor of the multi-matrix step):
 *  1. momentum, an exponential moving average of the gradient
 *     ([OPT] section 2.1):   M = fl(fl(mu*M) + fl((1-mu)*G))
 *  2. Nesterov look-ahead, read as the same average taken one step further:
 *        u = fl(fl((1-mu)*G) + fl(mu*M))        (nesterov = 1)
 *        u = M                                   (nesterov = 0)
 * (1-mu) is computed in fp32.  u may be NULL. */
void oracle_momentum_scaled(const float* G, float* M, float* u, int64_t n, float mu, int nesterov,
                            float g_scale, int scale_g)
{
    const float one_minus_mu = 1.0f - mu;
    for (int64_t i = 0; i < n; ++i) {
        const float g = scale_g ? g_scale * G[i] : G[i];
        float gterm = one_minus_mu * g;
        float mnew = mu * M[i] + gterm;
        M[i] = mnew;
        if (u)
            u[i] = nesterov ? gterm + mu * mnew : mnew;
    }
}

void oracle_momentum(const float* G, float* M, float* u, int64_t n, float mu, int nesterov)
{
    oracle_momentum_scaled(G, M, u, n, mu, nesterov, 1.0f, 0);
}

/* Steps 3-4: Frobenius normalisation and bf16 rounding.
 *  3. ||u||_F summed in fp64 in element order; s = float(1/(sqrt(sum u^2)+eps))
 *  4. X0 = bf16(u) written wide (min x max): transposed when rows > cols so
 *     that NS works on the smaller Gram matrix X X^T.
 * The normalised NS input is s * X0: the pages say the iteration runs in
 * bf16 on the normalised matrix but not where the cast falls; here the
 * look-ahead is cast once and s is applied in fp32 inside the first NS step
 * (oracle_newton_schulz_scaled), the GPU path's rounding points.
 * X0 is a (min x max) fp64 array of bf16 values.  Returns s. */
float oracle_normalize(const float* u, int64_t rows, int64_t cols, float eps, double* X0)
{
    const int64_t n = rows * cols;
    const int transposed = rows > cols;
    const int64_t np = transposed ? rows : cols;
    double ss = 0.0;
    for (int64_t i = 0; i < n; ++i)
        ss += (double)u[i] * (double)u[i];
    const float s = (float)(1.0 / (sqrt(ss) + (double)eps));
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t c = 0; c < cols; ++c) {
            double x0 = bf16_round(u[r * cols + c]);
            if (transposed)
                X0[c * np + r] = x0;
            else
                X0[r * np + c] = x0;
        }
    return s;
}

/* Steps 3-4 under the other reading of where the cast falls: the
 * normalised look-ahead itself is cast, X0 = bf16(fl32(u * s)) (wide, as
 * above), and the NS iteration then runs on X0 unscaled.  s is the same
 * fp32 value oracle_normalize returns; so is the return value. */
float oracle_normalize_cast_after(const float* u, int64_t rows, int64_t cols, float eps, double* X0)
{
    const float s = oracle_normalize(u, rows, cols, eps, X0);
    const int transposed = rows > cols;
    const int64_t np = transposed ? rows : cols;
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t c = 0; c < cols; ++c) {
            const float scaled = u[r * cols + c] * s;
            double x0 = bf16_round(scaled);
            if (transposed)
                X0[c * np + r] = x0;
            else
                X0[r * np + c] = x0;
        }
    return s;
}

/* The update's scale factor, computed in fp64 and rounded to fp32:
 *   mode 0: rms_scale * sqrt(max(rows, cols)) -- the update RMS matches
 *           AdamW's 0.2-0.4 ([K2] section 3.1);
 *   mode 1: max(1, sqrt(d_out / d_in)) = max(1, sqrt(rows / cols)) for an
 *           (out, in) weight -- the per-matrix learning-rate adjustment of
 *           the muP view ([K2] section 3.2). */
float oracle_update_scale(int64_t rows, int64_t cols, float rms_scale, int scale_mode)
{
    if (scale_mode == 1) {
        double r = sqrt((double)rows / (double)cols);
        return (float)(r > 1.0 ? r : 1.0);
    }
    const int64_t np = rows > cols ? rows : cols;
    return (float)((double)rms_scale * sqrt((double)np));
}

/* Step 7: decoupled weight decay and the RMS-matched update ([OPT] section
 * 3.1 for the decoupled form, [K2] section 3.1 for matching the update RMS
 * of AdamW).  Both terms use the old W:
 *    scale = oracle_update_scale(rows, cols, rms_scale, scale_mode)
 *    W = fl(W - fl(lr * fl(fl(wd*W) + fl(scale*O))))
 * O is the NS output in the wide orientation (min x max, float values). */
void oracle_final_update(float* W, const float* O, int64_t rows, int64_t cols,
                         float lr, float weight_decay, float rms_scale, int scale_mode)
{
    const int transposed = rows > cols;
    const int64_t np = transposed ? rows : cols;
    const float scale = oracle_update_scale(rows, cols, rms_scale, scale_mode);
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t c = 0; c < cols; ++c) {
            float o = transposed ? O[c * np + r] : O[r * np + c];
            float w = W[r * cols + c];
            float decay = weight_decay * w;
            float step = scale * o;
            float delta = lr * (decay + step);
            W[r * cols + c] = w - delta;
        }
}

/* Per-matrix statistics of a step, for monitoring (the update does not use
 * them):
 *   u_norm     = sqrt(sum u^2), the fp64 sum in element order: the norm that
 *                step 3 divides by
 *   update_rms = sqrt(sum fl(scale * o)^2 / (rows * cols)): each product and
 *                square rounded to fp32, summed in fp64; scale as in step 7.
 *                This is the RMS of the RMS-matched update before lr and
 *                decay, which [K2] section 3.1 sets to match AdamW's 0.2-0.4.
 * u: rows x cols; O: the wide NS output (min x max), rows * cols values. */
void oracle_step_stats(const float* u, const float* O, int64_t rows, int64_t cols,
                       float rms_scale, int scale_mode, double* u_norm, double* update_rms)
{
    const int64_t n = rows * cols;
    double su = 0.0, so = 0.0;
    for (int64_t i = 0; i < n; ++i)
        su += (double)u[i] * (double)u[i];
    const float scale = oracle_update_scale(rows, cols, rms_scale, scale_mode);
    for (int64_t i = 0; i < n; ++i) {
        const float v = scale * O[i];
        const float sq = v * v;
        so += (double)sq;
    }
    *u_norm = sqrt(su);
    *update_rms = sqrt(so / (double)n);
}

/* One Muon step on one rows x cols matrix, in place on W and M:
 * oracle_momentum (on g_scale * G when scale_g != 0), oracle_normalize, NS
 * (bf16 emulation; per-step coefficients when hp->ns_coeffs is set) on the
 * wide matrix, oracle_final_update.
 *   W   fp32 master weight (rows x cols, row-major), updated in place
 *   G   gradient, fp32 values (a bf16 gradient is passed already widened:
 *       the widening is exact)
 *   M   fp32 momentum, updated in place
 *   acc               how the NS products accumulate: 0 fp64, 1 fp32
 *                     (one rounding per addition), 2 fp32 round-toward-
 *                     zero per 16-product block
 *   cast_after_scale  X0 = bf16(u * s) and NS runs on it unscaled
 *                     (oracle_normalize_cast_after), instead of X0 =
 *                     bf16(u) with s applied inside the first NS step
 *   X0  optional out: the bf16 NS input before any in-step scale (wide,
 *       float values)
 *   O   optional out: the NS output (wide, float values)
 * The two flags select the spread variants; (0, 0) is the library's
 * arithmetic.  Returns 0 on success. */
int oracle_muon_step_matrix_ex(float* W, const float* G, float* M,
                               int64_t rows, int64_t cols,
                               const oracle_muon_hparams* hp,
                               float g_scale, int scale_g,
                               int acc, int cast_after_scale,
                               float* X0_out, float* O_out)
{
    if (rows <= 0 || cols <= 0 || !hp)
        return 1;
    const int64_t n = rows * cols;
    const int64_t mp = rows > cols ? cols : rows;
    const int64_t np = rows > cols ? rows : cols;
    float* u = (float*)malloc(sizeof(float) * n);
    double* X = (double*)malloc(sizeof(double) * n);
    float* O = (float*)malloc(sizeof(float) * n);
    if (!u || !X || !O) {
        free(u); free(X); free(O);
        return 2;
    }
    oracle_momentum_scaled(G, M, u, n, hp->momentum, hp->nesterov, g_scale, scale_g);
    const float s = cast_after_scale ? oracle_normalize_cast_after(u, rows, cols, hp->norm_eps, X)
                                     : oracle_normalize(u, rows, cols, hp->norm_eps, X);
    if (X0_out)
        for (int64_t i = 0; i < n; ++i)
            X0_out[i] = (float)X[i];
    float table[300];
    const float* coeffs = hp->ns_coeffs;
    if (!coeffs) {
        if (hp->ns_steps < 0 || hp->ns_steps > 100) {
            free(u); free(X); free(O);
            return 11;
        }
        for (int k = 0; k < hp->ns_steps; ++k) {
            table[3 * k] = hp->ns_a;
            table[3 * k + 1] = hp->ns_b;
            table[3 * k + 2] = hp->ns_c;
        }
        coeffs = table;
    }
    int rc = oracle_newton_schulz_ex(X, mp, np, hp->ns_steps, coeffs, 1, cast_after_scale ? 1.0f : s, acc);
    if (rc) {
        free(u); free(X); free(O);
        return 10 + rc;
    }
    for (int64_t i = 0; i < n; ++i)
        O[i] = (float)X[i];
    if (O_out)
        memcpy(O_out, O, sizeof(float) * n);
    oracle_final_update(W, O, rows, cols, hp->lr, hp->weight_decay, hp->rms_scale, hp->scale_mode);
    free(u); free(X); free(O);
    return 0;
}

/* The step as the library computes it: fp64 products, the look-ahead cast
 * before the normalisation. */
int oracle_muon_step_matrix_scaled(float* W, const float* G, float* M,
                                   int64_t rows, int64_t cols,
                                   const oracle_muon_hparams* hp,
                                   float g_scale, int scale_g,
                                   float* X0_out, float* O_out)
{
    return oracle_muon_step_matrix_ex(W, G, M, rows, cols, hp, g_scale, scale_g, 0, 0, X0_out, O_out);
}

int oracle_muon_step_matrix(float* W, const float* G, float* M,
                            int64_t rows, int64_t cols,
                            const oracle_muon_hparams* hp,
                            float* X0_out, float* O_out)
{
    return oracle_muon_step_matrix_scaled(W, G, M, rows, cols, hp, 1.0f, 0, X0_out, O_out);
}

/* Statistics of all gradients of one multi-matrix step ([OPT] section 5.4:
 * an Inf guard that skips the step, and clipping by the global norm):
 * *sumsq = sum of g^2 over every element of every matrix, in fp64, matrix by
 * matrix in element order; *nonfinite = number of NaN or +-inf elements. */
void oracle_grad_stats(const float* const* G, const int64_t* n, int64_t count,
                       double* sumsq, int64_t* nonfinite)
{
    double s = 0.0;
    int64_t bad = 0;
    for (int64_t k = 0; k < count; ++k)
        for (int64_t i = 0; i < n[k]; ++i) {
            const double g = (double)G[k][i];
            s += g * g;
            if (!isfinite(G[k][i]))
                ++bad;
        }
    *sumsq = s;
    *nonfinite = bad;
}

/* The clip factor: min(1, max_norm / (sqrt(sumsq) + 1e-6)) in fp64, rounded
 * to fp32 (a NaN ratio gives 1). */
float oracle_clip_factor(double sumsq, float max_norm)
{
    const double c = (double)max_norm / (sqrt(sumsq) + 1e-6);
    return (float)(c < 1.0 ? c : 1.0);
}

/* ------------------------------------------------------------------------ */
/* AdamW                                                                     */
/* ------------------------------------------------------------------------ */

typedef struct {
    float lr, beta1, beta2, eps, weight_decay;
} oracle_adamw_hparams;

/* AdamW on flat fp32 buffers, step t >= 1, in place on p, m, v.
 * [OPT] section 2.3 gives Adam with bias correction and section 3.1 the
 * decoupled weight decay:
 *   m = b1 m + (1-b1) g;  v = b2 v + (1-b2) g^2
 *   m_hat = m / (1-b1^t); v_hat = v / (1-b2^t)
 *   p = p - lr * m_hat / (sqrt(v_hat) + eps) - lr * wd * p
 * The bias-correction denominators are computed once in fp64 and rounded to
 * fp32; everything else is separately rounded fp32 in this order:
 *   m    = fl(fl(b1*m) + fl((1-b1)*g))
 *   v    = fl(fl(b2*v) + fl((1-b2)*fl(g*g)))
 *   upd  = fl( fl(m/bc1) / fl(sqrt(fl(v/bc2)) + eps) )
 *   p    = fl(p - fl(lr * fl(upd + fl(wd*p))))
 * with (1-b1), (1-b2) computed in fp32.  Returns 0 on success. */
int oracle_adamw_step(float* p, const float* g, float* m, float* v, int64_t n,
                      const oracle_adamw_hparams* hp, int64_t t)
{
    if (!hp || t < 1 || n < 0)
        return 1;
    const float bc1 = (float)(1.0 - pow((double)hp->beta1, (double)t));
    const float bc2 = (float)(1.0 - pow((double)hp->beta2, (double)t));
    const float one_minus_b1 = 1.0f - hp->beta1;
    const float one_minus_b2 = 1.0f - hp->beta2;
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) {
        float gi = g[i];
        float mi = hp->beta1 * m[i] + one_minus_b1 * gi;
        float g2 = gi * gi;
        float vi = hp->beta2 * v[i] + one_minus_b2 * g2;
        float m_hat = mi / bc1;
        float v_hat = vi / bc2;
        float den = sqrtf(v_hat) + hp->eps;
        float upd = m_hat / den;
        float decay = hp->weight_decay * p[i];
        p[i] = p[i] - hp->lr * (upd + decay);
        m[i] = mi;
        v[i] = vi;
    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Plan: grouping, orientation and chunking                                  */
/* ------------------------------------------------------------------------ */

/* Per-matrix workspace bytes of the library, restated from its documented
 * layout (not from its code): two wide X buffers (m' x ld(n') bf16), the A
 * and B Gram buffers (m' x ld(m') bf16), each padded to 256 bytes, plus an
 * 8 KiB per-matrix record; ld(x) = x rounded up to a multiple of 8. */
static int64_t round_up(int64_t x, int64_t q) { return (x + q - 1) / q * q; }

int64_t oracle_ws_bytes_per_matrix(int64_t mp, int64_t np)
{
    int64_t x = round_up(2 * mp * round_up(np, 8), 256);
    int64_t g = round_up(2 * mp * round_up(mp, 8), 256);
    return 2 * x + 2 * g + 8192;
}

typedef struct {
    int32_t mat_idx, transposed, group_id, slot, chunk_id, pad_;
    int64_t mp, np;
} oracle_plan_entry;

/* The plan orders matrices by (m', n') ascending with m' = min(rows, cols),
 * n' = max(rows, cols), ties broken by the caller's index; transposed is
 * rows > cols.  group_id numbers the distinct (m', n') pairs in that order.
 * Matrices are packed into chunks in plan order: a new chunk starts when
 * adding the next matrix's workspace would exceed ws_bytes.  slot counts the
 * matrices of one group within one chunk.  The ordering is written out as an
 * insertion sort so that stability is evident.  Returns 0 on success, 3 when
 * a single matrix needs more than ws_bytes. */
int oracle_plan(const int64_t* rows, const int64_t* cols, int64_t count,
                int64_t ws_bytes, oracle_plan_entry* out)
{
    if (count < 0 || (count > 0 && (!rows || !cols || !out)))
        return 1;
    int64_t* order = (int64_t*)malloc(sizeof(int64_t) * (count ? count : 1));
    if (!order)
        return 2;
    for (int64_t i = 0; i < count; ++i) {
        if (rows[i] <= 0 || cols[i] <= 0) {
            free(order);
            return 1;
        }
        order[i] = i;
    }
    for (int64_t i = 1; i < count; ++i) {
        int64_t cur = order[i];
        int64_t cm = rows[cur] < cols[cur] ? rows[cur] : cols[cur];
        int64_t cn = rows[cur] < cols[cur] ? cols[cur] : rows[cur];
        int64_t j = i - 1;
        while (j >= 0) {
            int64_t o = order[j];
            int64_t om = rows[o] < cols[o] ? rows[o] : cols[o];
            int64_t on = rows[o] < cols[o] ? cols[o] : rows[o];
            if (om > cm || (om == cm && on > cn)) {
                order[j + 1] = order[j];
                --j;
            } else {
                break;
            }
        }
        order[j + 1] = cur;
    }
    int32_t group = -1, chunk = 0, slot = 0;
    int64_t prev_m = -1, prev_n = -1, used = 0;
    for (int64_t k = 0; k < count; ++k) {
        int64_t i = order[k];
        int64_t mp = rows[i] < cols[i] ? rows[i] : cols[i];
        int64_t np = rows[i] < cols[i] ? cols[i] : rows[i];
        int64_t need = oracle_ws_bytes_per_matrix(mp, np);
        if (need > ws_bytes) {
            free(order);
            return 3;
        }
        int new_group = (mp != prev_m || np != prev_n);
        if (new_group)
            ++group;
        if (k > 0 && used + need > ws_bytes) {
            ++chunk;
            used = 0;
            slot = 0;
        } else if (new_group) {
            slot = 0;
        }
        out[k].mat_idx = (int32_t)i;
        out[k].transposed = rows[i] > cols[i];
        out[k].group_id = group;
        out[k].slot = slot;
        out[k].chunk_id = chunk;
        out[k].pad_ = 0;
        out[k].mp = mp;
        out[k].np = np;
        ++slot;
        used += need;
        prev_m = mp;
        prev_n = np;
    }
    free(order);
    return 0;
}

int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
