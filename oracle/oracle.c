/*
 * oracle.c -- plain, slow, obviously-correct CPU reference for the layout-folding
 * hot path.  TEST INFRASTRUCTURE ONLY: nothing on the product path may link,
 * load or call this file; only the test-suite, the smoke check and the bench's
 * CPU-baseline leg do.  It shares no code with the CUDA library.
 *
 * Arithmetic is fp64 over inputs widened exactly from bf16 (or fp32), with
 * every reduction summed sequentially in its natural index order.  OpenMP only
 * distributes independent output rows over cores; it never changes the order of
 * any sum.
 *
 * Sources (web pages, cited by title and section):
 *  [P1] "Strength reduction: fold transpose into a subsequent GEMM call"
 *       (lightning-thunder issue 1252) -- the Feature program and its trace.
 *  [P2] "Feature request: Schedule a small matmul op as a reduction (or
 *       pointwise) op" (NVIDIA/Fuser issue 3646) -- the T19 matmul and its
 *       broadcast/mul/squeeze rewrite.
 *  [P3] "Improve the Inductor generated kernel for the pattern of output1 =
 *       pointwise(intput); output2 = transpose(output1)" (pytorch issue
 *       130015) -- the float8 cast and its column-major copy (Examples).
 *  [P4] "Allow reductions in matmul epilogues" (NVIDIA/Fuser issue 2213) --
 *       the fused matmul + cross-entropy fusion definition.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* bf16 -> fp64, exact: a bf16 value is the top 16 bits of an IEEE binary32. */
static double bf16_to_f64(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* fp32 -> bf16 with round-to-nearest, ties to even (the IEEE default rounding
 * applied to an 8-bit significand).  NaN stays a quiet NaN. */
static uint16_t f32_to_bf16_rne(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7fffffffu) > 0x7f800000u)
        return (uint16_t)((u >> 16) | 0x0040u);
    uint32_t lsb = (u >> 16) & 1u;
    u += 0x7fffu + lsb;
    return (uint16_t)(u >> 16);
}

int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void oracle_set_num_threads(int n)
{
#ifdef _OPENMP
    if (n > 0)
        omp_set_num_threads(n);
#else
    (void)n;
#endif
}

uint16_t oracle_bf16_round(float f) { return f32_to_bf16_rne(f); }

/*
 * NT GEMM [P1, Feature: `torch.matmul(x, weight.t())`, and the "so-called NT
 * GEMM" remark]:  out[m,n] = sum_k X[m,k] * W[n,k], with X [M,K] and W [N,K]
 * both row-major (K contiguous).  The weight is read in its stored layout.
 */
void oracle_gemm_nt(const uint16_t *x, const uint16_t *w, int64_t M, int64_t N,
                    int64_t K, double *out)
{
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t m = 0; m < M; ++m) {
        const uint16_t *xr = x + m * K;
        for (int64_t n = 0; n < N; ++n) {
            const uint16_t *wr = w + n * K;
            double acc = 0.0;
            for (int64_t k = 0; k < K; ++k)
                acc += bf16_to_f64(xr[k]) * bf16_to_f64(wr[k]);
            out[m * N + n] = acc;
        }
    }
}

/* Same definition restricted to a list of rows of X (for shapes whose full
 * product is too slow here): out[r,n] = sum_k X[rows[r],k] * W[n,k]. */
void oracle_gemm_nt_rows(const uint16_t *x, const uint16_t *w, const int64_t *rows,
                         int64_t R, int64_t N, int64_t K, double *out)
{
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t r = 0; r < R; ++r) {
        const uint16_t *xr = x + rows[r] * K;
        for (int64_t n = 0; n < N; ++n) {
            const uint16_t *wr = w + n * K;
            double acc = 0.0;
            for (int64_t k = 0; k < K; ++k)
                acc += bf16_to_f64(xr[k]) * bf16_to_f64(wr[k]);
            out[r * N + n] = acc;
        }
    }
}

/* The materialised transpose that the traced program runs as its own fusion
 * [P1, trace: `prims.transpose(weight, (1, 0))`]:  wt[k,n] = W[n,k]. */
void oracle_transpose_bf16(const uint16_t *w, int64_t N, int64_t K, uint16_t *wt)
{
    for (int64_t n = 0; n < N; ++n)
        for (int64_t k = 0; k < K; ++k)
            wt[k * N + n] = w[n * K + k];
}

/* The GEMM the trace then runs on the transposed copy [P1, trace:
 * `prims.matmul(t7, t)`]:  out[m,n] = sum_k X[m,k] * Wt[k,n], Wt [K,N]. */
void oracle_gemm_nn(const uint16_t *x, const uint16_t *wt, int64_t M, int64_t N,
                    int64_t K, double *out)
{
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t m = 0; m < M; ++m) {
        const uint16_t *xr = x + m * K;
        for (int64_t n = 0; n < N; ++n) {
            double acc = 0.0;
            for (int64_t k = 0; k < K; ++k)
                acc += bf16_to_f64(xr[k]) * bf16_to_f64(wt[k * N + n]);
            out[m * N + n] = acc;
        }
    }
}

/*
 * The contraction with either operand in either stored layout [P1, Feature:
 * the transposed weight folded into the GEMM; P4, the matmul scheduler's
 * canonicalisation of operand layouts to one (M, N, K) contraction]:
 *   out[m,n] = sum_k X(m,k) * W(n,k)
 *   X(m,k) = x[m*K + k] (x_mn == 0: X stored [M,K]) or x[k*M + m] (x_mn == 1: stored [K,M])
 *   W(n,k) = w[n*K + k] (w_mn == 0: W stored [N,K]) or w[k*N + n] (w_mn == 1: stored [K,N])
 * fp64, k summed in order.  `rows` (may be NULL) restricts it to R listed
 * rows m: out is then [R, N].
 */
void oracle_gemm_layout(const uint16_t *x, int x_mn, const uint16_t *w, int w_mn, int64_t M, int64_t N,
                        int64_t K, const int64_t *rows, int64_t R, double *out)
{
    const int64_t nrows = rows ? R : M;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t r = 0; r < nrows; ++r) {
        const int64_t m = rows ? rows[r] : r;
        for (int64_t n = 0; n < N; ++n) {
            double acc = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                const uint16_t xv = x_mn ? x[k * M + m] : x[m * K + k];
                const uint16_t wv = w_mn ? w[k * N + n] : w[n * K + k];
                acc += bf16_to_f64(xv) * bf16_to_f64(wv);
            }
            out[r * N + n] = acc;
        }
    }
}

/*
 * The same contraction over a batch of strided views [P1: the projection's
 * input is itself a view of a larger tensor; the matmul page's operands are
 * batched and permuted views]: for b < batch,
 *   out[b][m][n] = sum_k X_b(m,k) * W_b(n,k)
 *   X_b(m,k) = x[b*sx + m*ldx + k] (x_mn == 0) or x[b*sx + k*ldx + m] (x_mn == 1)
 *   W_b(n,k) = w[b*sw + n*ldw + k] (w_mn == 0) or w[b*sw + k*ldw + n] (w_mn == 1)
 * (sw == 0: one W for every batch).  fp64, k in order; out is [batch, M, N].
 */
void oracle_gemm_batched(const uint16_t *x, int x_mn, int64_t ldx, int64_t sx, const uint16_t *w, int w_mn,
                         int64_t ldw, int64_t sw, int64_t batch, int64_t M, int64_t N, int64_t K, double *out)
{
#pragma omp parallel for collapse(2) schedule(dynamic, 1)
    for (int64_t b = 0; b < batch; ++b)
        for (int64_t m = 0; m < M; ++m) {
            const uint16_t *xb = x + b * sx;
            const uint16_t *wb = w + b * sw;
            for (int64_t n = 0; n < N; ++n) {
                double acc = 0.0;
                for (int64_t k = 0; k < K; ++k) {
                    const uint16_t xv = x_mn ? xb[k * ldx + m] : xb[m * ldx + k];
                    const uint16_t wv = w_mn ? wb[k * ldw + n] : wb[n * ldw + k];
                    acc += bf16_to_f64(xv) * bf16_to_f64(wv);
                }
                out[(b * M + m) * N + n] = acc;
            }
        }
}

/*
 * Row-wise cross-entropy over logits z [M,N] (fp64) [P4, fusion example]:
 *   mx   = max_n z[m,n]                      ("allreduce log sum exp in N")
 *   e    = exp(z - mx),  sumexp = sum_n e
 *   lse  = log(sumexp) + mx
 *   loss = lse - z[m, L[m]]                  (the "xent = lse - y_i*onehot(L)_i"
 *                                             comment; see the reading below)
 *   grad = e / sumexp - onehot(L)            ("yhatminusy")
 * Reading: the example's code sums (lse - where(onehot, z, 0)) over N, which
 * would give N*lse - z_L; its comment and the standard cross-entropy give
 * lse - z_L, and only that form gives ln N for equal logits, so it is taken.
 * A label outside [0,N) makes that row's loss NaN (the page defines no
 * ignore-index); its grad row is then the softmax alone.
 * lse_or_null / grad_or_null may be NULL.
 */
void oracle_xent_logits(const double *z, const int32_t *labels, int64_t M, int64_t N,
                        double *loss, double *lse_or_null, double *grad_or_null)
{
#pragma omp parallel for schedule(dynamic, 4)
    for (int64_t m = 0; m < M; ++m) {
        const double *zr = z + m * N;
        double mx = -INFINITY;
        for (int64_t n = 0; n < N; ++n)
            if (zr[n] > mx)
                mx = zr[n];
        double sumexp = 0.0;
        for (int64_t n = 0; n < N; ++n)
            sumexp += exp(zr[n] - mx);
        double lse = log(sumexp) + mx;
        int64_t L = labels[m];
        int valid = (L >= 0 && L < N);
        loss[m] = valid ? lse - zr[L] : NAN;
        if (lse_or_null)
            lse_or_null[m] = lse;
        if (grad_or_null) {
            double *g = grad_or_null + m * N;
            for (int64_t n = 0; n < N; ++n)
                g[n] = exp(zr[n] - mx) / sumexp - ((valid && n == L) ? 1.0 : 0.0);
        }
    }
}

/*
 * Brute-force cross-entropy on small inputs: loss = -log(exp(z_L) / sum_n exp(z_n))
 * in long double, with no max subtraction (the textbook definition the fused
 * form must reproduce).  Only meaningful while exp(z) stays in range.
 */
void oracle_xent_bruteforce(const double *z, const int32_t *labels, int64_t M, int64_t N,
                            double *loss)
{
    for (int64_t m = 0; m < M; ++m) {
        const double *zr = z + m * N;
        long double den = 0.0L;
        for (int64_t n = 0; n < N; ++n)
            den += expl((long double)zr[n]);
        int64_t L = labels[m];
        if (L < 0 || L >= N) {
            loss[m] = NAN;
            continue;
        }
        long double p = expl((long double)zr[L]) / den;
        loss[m] = (double)(-logl(p));
    }
}

/* GEMM + cross-entropy from bf16 inputs: z = X W^T (oracle_gemm_nt) followed
 * by oracle_xent_logits, for a list of rows of X.  z_or_null receives the fp64
 * logits [R,N] if given; the caller owns every buffer. */
void oracle_xent_rows(const uint16_t *x, const uint16_t *w, const int32_t *labels,
                      const int64_t *rows, int64_t R, int64_t N, int64_t K,
                      double *z, double *loss, double *lse_or_null, double *grad_or_null)
{
    oracle_gemm_nt_rows(x, w, rows, R, N, K, z);
    /* labels are indexed by the original row */
    int32_t lab_small[1];
    for (int64_t r = 0; r < R; ++r) {
        lab_small[0] = labels[rows[r]];
        oracle_xent_logits(z + r * N, lab_small, 1, N, loss + r,
                           lse_or_null ? lse_or_null + r : NULL,
                           grad_or_null ? grad_or_null + r * N : NULL);
    }
}

/*
 * K=1 matmul as broadcast-multiply-squeeze [P2, the T19 matmul of a [64,1]
 * and a [1,4096] operand and its proposed rewrite broadcast(T15) *
 * broadcast(T18), squeezed]:  out[i,j] = a[i] * b[j], one fp32 multiply
 * (the single rounding of the exact product), no accumulation.
 */
void oracle_matmul_k1(const float *a, const float *b, int64_t M, int64_t N, float *out)
{
    for (int64_t i = 0; i < M; ++i)
        for (int64_t j = 0; j < N; ++j) {
            double p = (double)a[i] * (double)b[j];  /* exact in fp64 */
            out[i * N + j] = (float)p;               /* one rounding to fp32 */
        }
}

/* The same product for bf16 operands of a K=1 NT GEMM: X [M,1], W [N,1],
 * out[i,j] = bf16_rn(x[i] * w[j]) -- the bf16 x bf16 product is exact in fp64
 * (and in fp32), so this is the single rounding of the exact result. */
void oracle_matmul_k1_bf16(const uint16_t *x, const uint16_t *w, int64_t M, int64_t N,
                           uint16_t *out)
{
    for (int64_t i = 0; i < M; ++i)
        for (int64_t j = 0; j < N; ++j) {
            double p = bf16_to_f64(x[i]) * bf16_to_f64(w[j]);
            out[i * N + j] = f32_to_bf16_rne((float)p);
        }
}

/*
 * The RoPE segment around the K=1 matmul [P2, the kernel_math listing of the
 * Mistral forward, T3 .. T26], one step per tensor:
 *   T13[i]    = float(T3[i])             inv_freq, bf16 -> fp32 (exact)
 *   T18[s]    = float(T4[s])             position id, int64 -> fp32 (round to nearest)
 *   T19[i,s]  = T13[i] * T18[s]          the K=1 matmul: one fp32 multiply
 *   T20[s,i]  = T19[i,s]                 permute to [S, H]
 *   T21[s,c]  = c <  H ? T20[s,c]   : 0  pad H zeros on the right
 *   T22[s,c]  = c >= H ? T20[s,c-H] : 0  pad H zeros on the left
 *   T23[s,c]  = c < H ? T21[s,c] : T22[s,c]   cat of the padded halves (2H columns)
 *   T24[s,c]  = cosf(T23[s,c])           fp32 cosine: cos of the fp32 argument,
 *                                        rounded to fp32 (here from fp64 libm)
 *   T26[s,c]  = bf16(T24[s,c])           round to nearest even
 * cos_out is T26 as [S, 2H] row-major.  sin_out (may be NULL) is the same chain
 * with sinf in place of cosf: the listing prints only the cosine branch; the
 * segment's second [4096,128] output, T31, is read as the sine (the RoPE module
 * returns the cosine and the sine of the same angles).
 */
void oracle_rope_cos_sin(const uint16_t *inv_freq, const int64_t *pos, int64_t H, int64_t S,
                         uint16_t *cos_out, uint16_t *sin_out)
{
    for (int64_t s = 0; s < S; ++s) {
        float t18 = (float)pos[s];
        for (int64_t c = 0; c < 2 * H; ++c) {
            float t21 = 0.0f, t22 = 0.0f;
            if (c < H)
                t21 = (float)(bf16_to_f64(inv_freq[c]) * (double)t18);       /* T20[s,c] */
            else
                t22 = (float)(bf16_to_f64(inv_freq[c - H]) * (double)t18);   /* T20[s,c-H] */
            float t23 = c < H ? t21 : t22;
            cos_out[s * 2 * H + c] = f32_to_bf16_rne((float)cos((double)t23));
            if (sin_out)
                sin_out[s * 2 * H + c] = f32_to_bf16_rne((float)sin((double)t23));
        }
    }
}

/*
 * fp32 -> float8 E4M3 ("fn" variant: 1 sign bit, 4 exponent bits with bias 7,
 * 3 mantissa bits, no infinities, S.1111.111 is NaN, largest finite 448),
 * round to nearest, ties to even, by the definition: find the representable
 * neighbours of |f| and pick the nearer one (the even mantissa on a tie).
 * Inputs are clamped to +-448 by the caller; NaN maps to 0x7F.
 */
uint8_t oracle_f32_to_e4m3(float f)
{
    if (f != f)
        return 0x7F;
    uint8_t sign = (f < 0.0f || (f == 0.0f && 1.0f / f < 0.0f)) ? 0x80 : 0x00;
    double a = fabs((double)f);
    if (a == 0.0)
        return sign;
    /* value of code c (c in 0..126, positive): subnormal for exponent field 0 */
    double best = 0.0;
    int best_code = 0;
    for (int c = 0; c <= 126; ++c) {
        int e = c >> 3, m = c & 7;
        double v = e == 0 ? ldexp((double)m, -9) : ldexp(1.0 + m / 8.0, e - 7);
        if (v <= a) {
            best = v;
            best_code = c;
        }
    }
    if (best_code == 126) /* at or above 448 */
        return (uint8_t)(sign | 126);
    {
        int c_hi = best_code + 1;
        int e = c_hi >> 3, m = c_hi & 7;
        double hi = e == 0 ? ldexp((double)m, -9) : ldexp(1.0 + m / 8.0, e - 7);
        double dlo = a - best, dhi = hi - a;
        int code = best_code;
        if (dhi < dlo || (dhi == dlo && (c_hi & 1) == 0))
            code = c_hi;
        return (uint8_t)(sign | code);
    }
}

/*
 * The float8 training cast of "Improve the Inductor generated kernel for the
 * pattern of output1 = pointwise(intput); output2 = transpose(output1)"
 * (pytorch issue 130015), Examples: x = input * scale (bf16 times an fp32
 * scale: one fp32 multiply), clamped to [-448, 448], converted to E4M3; the
 * page returns the result both as is ([M,K] row-major) and as
 * t().contiguous().t() -- the same values stored column-major, i.e. the
 * [K,M] row-major array out_t[k*M + m] = out[m*K + k].
 */
void oracle_fp8_cast_dual(const uint16_t *x, int64_t M, int64_t K, float scale, uint8_t *out, uint8_t *out_t)
{
    for (int64_t m = 0; m < M; ++m)
        for (int64_t k = 0; k < K; ++k) {
            float v = (float)(bf16_to_f64(x[m * K + k]) * (double)scale); /* exact product, one rounding */
            if (v > 448.0f)
                v = 448.0f;
            if (v < -448.0f)
                v = -448.0f;
            uint8_t q = oracle_f32_to_e4m3(v);
            out[m * K + k] = q;
            out_t[k * M + m] = q;
        }
}
