/*
 * ns_oracle.c -- plain fp64 CPU oracle for batched quintic Newton-Schulz.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing on the product path may link, load or
 * call this file: only the tests, the smoke check and the benchmark's CPU
 * baseline leg use it. It shares no code, header or constant generator with
 * the CUDA library.
 *
 * What it computes, per matrix (no blocking, no fusion, no reordering beyond
 * the definition; every sum runs over its index in increasing order):
 *
 *   1. s = ||X||_F                          (plain sum of squares, then sqrt)
 *   2. X <- X / (s + eps)
 *   3. if M > N: W = X^T (so W is m x n with m = min(M,N)); else W = X
 *   4. repeat `steps` times:
 *        A = W W^T                 (m x m)
 *        B = b*A + c*(A A)         (m x m)
 *        W = a*W + B W             (m x n)
 *   5. write W back, transposed again if step 3 transposed.
 *
 * Sources. The three pages ("Fix megabatch_orthogonalize_async hang on empty
 * FSDP2 shards"; "Balance LayerWise optimizer shards by Newton-Schulz cost,
 * not parameter size"; the xtuner Muon remainder-strategy PR) all run this
 * iteration inside Muon, NorMuon and Dion2 but never print it. Its form, the
 * coefficients (a,b,c) = (3.4445, -4.7750, 2.0315), the default of 5 steps,
 * eps = 1e-7 and the rule of working on the transpose when M > N are the
 * standard quintic Newton-Schulz iteration of Muon. The zero-row property it
 * must preserve is stated in the first page's "Fix" section; the cost
 * max(M,N)*min(M,N)^2 is item 1 of the second page's "Changes" section.
 *
 * Build: gcc -O2 -ffp-contract=off -fopenmp -shared -fPIC ns_oracle.c -lm
 * (OpenMP only splits independent output rows across threads; the order of
 * every individual sum is unchanged. Contraction into FMA is off so x86 and
 * Arm hosts give the same bits.)
 *
 * Compile-time switch NS_ORACLE_MUTATION=k plants one deliberate mistake so
 * the tests can show that the pins catch it; the default (0) is the oracle.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifndef NS_ORACLE_MUTATION
#define NS_ORACLE_MUTATION 0
#endif

/* Newton-Schulz cost of one M x N matrix: max(M,N) * min(M,N)^2
 * (second page, "Changes" item 1). Returns -1 for negative dims. */
int64_t ns_oracle_cost(int64_t M, int64_t N)
{
    if (M < 0 || N < 0) return -1;
    int64_t hi = M > N ? M : N;
    int64_t lo = M > N ? N : M;
    return hi * lo * lo;
}

/* Frobenius norm: square root of the plain row-major sum of squares. */
double ns_oracle_frobenius(const double *X, int64_t M, int64_t N)
{
    double acc = 0.0;
    for (int64_t i = 0; i < M * N; ++i) {
#if NS_ORACLE_MUTATION == 5
        acc += fabs(X[i]);              /* planted: 1-norm instead of sum of squares */
#else
        acc += X[i] * X[i];
#endif
    }
    return sqrt(acc);
}

/* C = P Q for P (r x q), Q (q x s), all row-major. Each C[i][j] is the sum
 * over k = 0..q-1 of P[i][k]*Q[k][j], accumulated in increasing k. */
static void matmul(const double *P, const double *Q, int64_t r, int64_t q, int64_t s, double *C)
{
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < r; ++i) {
        double *crow = C + i * s;
        for (int64_t j = 0; j < s; ++j) crow[j] = 0.0;
        for (int64_t k = 0; k < q; ++k) {
            const double p = P[i * q + k];
            const double *qrow = Q + k * s;
            for (int64_t j = 0; j < s; ++j) crow[j] += p * qrow[j];
        }
    }
}

/* A = W W^T for W m x n, row-major; A is m x m: A[i][j] is the sum over
 * k = 0..n-1 of W[i][k]*W[j][k] in increasing k, computed as W times an
 * explicit copy of W^T (Wt, n x m) so the same product routine serves. */
static void gram(const double *W, int64_t m, int64_t n, double *Wt, double *A)
{
    for (int64_t i = 0; i < m; ++i)
        for (int64_t k = 0; k < n; ++k)
#if NS_ORACLE_MUTATION == 3
            Wt[k * m + i] = W[((i + 1) % m) * n + k];  /* planted: wrong row of the second operand */
#else
            Wt[k * m + i] = W[i * n + k];
#endif
    matmul(W, Wt, m, n, m, A);
}

/*
 * In-place Newton-Schulz on one row-major M x N fp64 matrix.
 *
 * orient: 0 = the specification's rule (work on X^T when M > N),
 *         1 = never transpose, 2 = always transpose.
 * Orientations 1 and 2 exist only so the tests can check the identity
 * X p(X^T X) = p(X X^T) X (the two orientations agree in exact arithmetic).
 *
 * Returns 0, or -1 for bad arguments, -2 if memory ran out.
 */
int ns_oracle_orthogonalize_sched(double *X, int64_t M, int64_t N, int steps,
                                  const double *table, double eps, int orient);

int ns_oracle_orthogonalize(double *X, int64_t M, int64_t N, int steps,
                            double a, double b, double c, double eps, int orient)
{
    if (steps < 0) return -1;
    double *table = (double *)malloc(sizeof(double) * 3 * (size_t)(steps > 0 ? steps : 1));
    if (!table) return -2;
    for (int it = 0; it < steps; ++it) {
        table[3 * it] = a; table[3 * it + 1] = b; table[3 * it + 2] = c;
    }
    int rc = ns_oracle_orthogonalize_sched(X, M, N, steps, table, eps, orient);
    free(table);
    return rc;
}

/*
 * As ns_oracle_orthogonalize, with the coefficients of step `it` in
 * table[3*it .. 3*it+2] = (a, b, c), so every step may use its own triple.
 */
int ns_oracle_orthogonalize_sched(double *X, int64_t M, int64_t N, int steps,
                                  const double *table, double eps, int orient)
{
    if (!X && M * N > 0) return -1;
    if (M < 0 || N < 0 || steps < 0 || orient < 0 || orient > 2) return -1;
    if (steps > 0 && !table) return -1;
    if (M == 0 || N == 0) return 0;

    const double s = ns_oracle_frobenius(X, M, N);
#if NS_ORACLE_MUTATION == 6
    const double denom = s * s + eps;            /* planted: squared norm */
#else
    const double denom = s + eps;
#endif
    int transpose = (orient == 0) ? (M > N) : (orient == 2);
    const int64_t m = transpose ? N : M;
    const int64_t n = transpose ? M : N;

    double *W = (double *)malloc(sizeof(double) * (size_t)(m * n));
    double *W2 = (double *)malloc(sizeof(double) * (size_t)(m * n));
    double *A = (double *)malloc(sizeof(double) * (size_t)(m * m));
    double *AA = (double *)malloc(sizeof(double) * (size_t)(m * m));
    double *Wt = (double *)malloc(sizeof(double) * (size_t)(m * n));
    if (!W || !W2 || !A || !AA || !Wt) {
        free(W); free(W2); free(A); free(AA); free(Wt);
        return -2;
    }

    /* step 2 + 3: normalise (divide by s + eps) and orient */
    for (int64_t i = 0; i < M; ++i)
        for (int64_t j = 0; j < N; ++j) {
            const double v = X[i * N + j] / denom;
            if (transpose) W[j * n + i] = v; else W[i * n + j] = v;
        }

    int nsteps = steps;
#if NS_ORACLE_MUTATION == 7
    if (nsteps > 0) nsteps -= 1;                 /* planted: one step short */
#endif
    for (int it = 0; it < nsteps; ++it) {
        const double a = table[3 * it], b = table[3 * it + 1], c = table[3 * it + 2];
        gram(W, m, n, Wt, A);                    /* A = W W^T */
        matmul(A, A, m, m, m, AA);               /* AA = A A */
        for (int64_t i = 0; i < m * m; ++i) {    /* B = b A + c A^2, kept in A */
#if NS_ORACLE_MUTATION == 1
            A[i] = b * A[i];                     /* planted: c*A^2 term dropped */
#elif NS_ORACLE_MUTATION == 2
            A[i] = -b * A[i] + c * AA[i];        /* planted: wrong sign of b */
#else
            A[i] = b * A[i] + c * AA[i];
#endif
        }
        matmul(A, W, m, m, n, W2);               /* W2 = B W */
        for (int64_t i = 0; i < m * n; ++i) {    /* W = a W + B W */
#if NS_ORACLE_MUTATION == 4
            W[i] = a * W[i] - W2[i];             /* planted: wrong sign of BW */
#else
            W[i] = a * W[i] + W2[i];
#endif
        }
    }

    for (int64_t i = 0; i < M; ++i)
        for (int64_t j = 0; j < N; ++j)
            X[i * N + j] = transpose ? W[j * n + i] : W[i * n + j];

    free(W); free(W2); free(A); free(AA); free(Wt);
    return 0;
}

/* Batched form: count matrices, each row-major, laid out back to back in X
 * (matrix i starts at offsets[i] doubles). Same arguments as above. */
int ns_oracle_orthogonalize_batched(double *X, const int64_t *offsets, const int64_t *shapes,
                                    int count, int steps, double a, double b, double c,
                                    double eps)
{
    if (count < 0) return -1;
    for (int i = 0; i < count; ++i) {
        int rc = ns_oracle_orthogonalize(X + offsets[i], shapes[2 * i], shapes[2 * i + 1],
                                         steps, a, b, c, eps, 0);
        if (rc) return rc;
    }
    return 0;
}
