/*
 * muon_oracle.c -- plain fp64 CPU oracle of one Muon optimizer step.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file.  It exists so that the GPU library can be checked against a
 * slow, obviously correct restatement of the method; only tests/,
 * __graft_entry__.smoke() and the CPU-baseline leg of bench.py use it.  It
 * shares no code, header, table or helper with the CUDA path.
 *
 * What it computes, and where the pages define it:
 *   "Cara Melatih ChatGPT Sendiri dengan Budget 50 Dolar" (apidog.com),
 *   section "2. Pengoptimal Muon (nanochat/optim.py)", and its Thai
 *   translation on dev.to, section "2. ตัวปรับปรุง Muon":
 *     - the name MomentUm Orthogonalized by Newton-Schulz (momentum first),
 *     - 2-D matrices go to Muon (the optimizer split table on the dev.to page),
 *     - the quintic Newton-Schulz loop with one (a, b, c) row per iteration:
 *       a Gram matrix, a polynomial b*A + c*A*A, and an axpy a*X + (product).
 *   The pages leave open the momentum form, the normalisation, the orientation
 *   and the weight-update scale; the readings taken here are:
 *     momentum, mode 0 (default): m' = beta*m + g ; u = nesterov ? g + beta*m' : m'
 *     momentum, mode 1 (EMA):     m' = beta*m + (1-beta)*g ;
 *                                 u = nesterov ? (1-beta)*g + beta*m' : m'
 *     X0 = u / (||u||_F + eps), with the long side kept as columns
 *       (a stored r x c matrix with r > c is transposed first);
 *     per iteration k with (a, b, c) = row k:  A = X X^T,  B = b A + c A A,
 *       X = a X + B X      (equal in exact arithmetic to the pages' X^T X form,
 *       since X p(X^T X) = p(X X^T) X);
 *     O = X, transposed back to r x c;  p' = p - lr * sqrt(max(1, r/c)) * O.
 *
 * Precision: everything in double; m' and p' are rounded to float only where
 * they are stored, as the optimizer state is float.
 *
 * All matrices are dense row-major.  Matrix products are the textbook triple
 * loop (row i, then k, then j), blocked only so the cache holds a slice of the
 * right operand; every C[i][j] still sums over k in ascending order.
 */
#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* C (M x N) = A (M x K) * B (K x N), all row-major. */
static void mat_mul(int M, int N, int K, const double* A, const double* B, double* C) {
    const int RB = 8, KB = 128;
#pragma omp parallel for schedule(static)
    for (int ib = 0; ib < M; ib += RB) {
        int ie = ib + RB < M ? ib + RB : M;
        for (int i = ib; i < ie; ++i) memset(C + (size_t)i * N, 0, sizeof(double) * (size_t)N);
        for (int kb = 0; kb < K; kb += KB) {
            int ke = kb + KB < K ? kb + KB : K;
            for (int i = ib; i < ie; ++i) {
                double* Ci = C + (size_t)i * N;
                for (int k = kb; k < ke; ++k) {
                    const double a = A[(size_t)i * K + k];
                    const double* Bk = B + (size_t)k * N;
                    for (int j = 0; j < N; ++j) Ci[j] += a * Bk[j];
                }
            }
        }
    }
}

/* T (cols x rows) = S^T for S (rows x cols). */
static void transpose(int rows, int cols, const double* S, double* T) {
#pragma omp parallel for schedule(static)
    for (int i = 0; i < rows; ++i)
        for (int j = 0; j < cols; ++j) T[(size_t)j * rows + i] = S[(size_t)i * cols + j];
}

int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void oracle_set_num_threads(int n) {
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

/*
 * Momentum (the "MomentUm" of the name; form chosen as stated above).
 * g, m: n_elem floats.  m_out receives m' rounded to float; u_out receives the
 * update direction in double (computed from the unrounded m').
 */
void oracle_momentum(long n_elem, const float* g, const float* m, double beta, int nesterov,
                     int mode, float* m_out, double* u_out) {
#pragma omp parallel for schedule(static)
    for (long e = 0; e < n_elem; ++e) {
        const double gd = (double)g[e], md = (double)m[e];
        double mn, u;
        if (mode == 1) {
            mn = beta * md + (1.0 - beta) * gd;
            u = nesterov ? (1.0 - beta) * gd + beta * mn : mn;
        } else {
            mn = beta * md + gd;
            u = nesterov ? gd + beta * mn : mn;
        }
        m_out[e] = (float)mn;
        u_out[e] = u;
    }
}

/* Frobenius norm of n doubles, summed in index order. */
double oracle_frobenius(long n, const double* x) {
    double s = 0.0;
    for (long e = 0; e < n; ++e) s += x[e] * x[e];
    return sqrt(s);
}

/*
 * The quintic Newton-Schulz loop on an already oriented and normalised
 * X (rows x cols), in place: for k in 0..K-1 with (a, b, c) = coeffs[3k..3k+2]:
 *   A = X X^T ; B = b A + c (A A) ; X = a X + B X.
 * Returns 0, or -1 if memory could not be allocated.
 */
int oracle_newton_schulz(int rows, int cols, double* X, int K, const double* coeffs) {
    const size_t rc = (size_t)rows * cols, rr = (size_t)rows * rows;
    double* XT = (double*)malloc(sizeof(double) * rc);
    double* A = (double*)malloc(sizeof(double) * rr);
    double* AA = (double*)malloc(sizeof(double) * rr);
    double* BX = (double*)malloc(sizeof(double) * rc);
    if (!XT || !A || !AA || !BX) {
        free(XT); free(A); free(AA); free(BX);
        return -1;
    }
    for (int k = 0; k < K; ++k) {
        const double a = coeffs[3 * k], b = coeffs[3 * k + 1], c = coeffs[3 * k + 2];
        transpose(rows, cols, X, XT);
        mat_mul(rows, rows, cols, X, XT, A);          /* A = X X^T            */
        mat_mul(rows, rows, rows, A, A, AA);          /* A A                  */
        for (size_t e = 0; e < rr; ++e) A[e] = b * A[e] + c * AA[e];  /* B   */
        mat_mul(rows, cols, rows, A, X, BX);          /* B X                  */
        for (size_t e = 0; e < rc; ++e) X[e] = a * X[e] + BX[e];
    }
    free(XT); free(A); free(AA); free(BX);
    return 0;
}

/*
 * Orthogonalised update of one stored r x c direction u (double):
 * orient (transpose when r > c), divide by (||u||_F + eps), run K
 * Newton-Schulz iterations, orient back.  O is r x c.
 * Returns 0, or -1 on allocation failure.
 */
int oracle_orthogonalize(int r, int c, const double* u, int K, const double* coeffs, double eps,
                         double* O) {
    const size_t rc = (size_t)r * c;
    const int tall = r > c;
    const int rows = tall ? c : r, cols = tall ? r : c;
    double* X = (double*)malloc(sizeof(double) * rc);
    if (!X) return -1;
    if (tall) transpose(r, c, u, X);
    else memcpy(X, u, sizeof(double) * rc);
    /* the norm is taken on the oriented copy (same value, one summation order) */
    const double s = 1.0 / (oracle_frobenius((long)rc, X) + eps);
    for (size_t e = 0; e < rc; ++e) X[e] *= s;
    if (oracle_newton_schulz(rows, cols, X, K, coeffs) != 0) {
        free(X);
        return -1;
    }
    if (tall) transpose(rows, cols, X, O);
    else memcpy(O, X, sizeof(double) * rc);
    free(X);
    return 0;
}

/* Update scale of a stored r x c matrix: sqrt(max(1, r / c)). */
static double oracle_aspect_scale(int r, int c) {
    const double ratio = (double)r / (double)c;
    return sqrt(ratio > 1.0 ? ratio : 1.0);
}

/*
 * One full Muon step on one stored r x c matrix.
 * Inputs p, g, m (float, r x c).  Outputs: p_out (p', float), m_out (m',
 * float) and, if O_out is not NULL, the orthogonalised update O (double).
 * Returns 0, or -1 on allocation failure.
 */
int oracle_muon_matrix(int r, int c, const float* p, const float* g, const float* m, double lr,
                       double beta, int nesterov, int mode, int K, const double* coeffs, double eps,
                       float* p_out, float* m_out, double* O_out) {
    const size_t rc = (size_t)r * c;
    double* u = (double*)malloc(sizeof(double) * rc);
    double* O = O_out ? O_out : (double*)malloc(sizeof(double) * rc);
    if (!u || !O) {
        free(u);
        if (!O_out) free(O);
        return -1;
    }
    oracle_momentum((long)rc, g, m, beta, nesterov, mode, m_out, u);
    int rcode = oracle_orthogonalize(r, c, u, K, coeffs, eps, O);
    if (rcode == 0) {
        const double scale = lr * oracle_aspect_scale(r, c);
        for (size_t e = 0; e < rc; ++e) p_out[e] = (float)((double)p[e] - scale * O[e]);
    }
    free(u);
    if (!O_out) free(O);
    return rcode;
}

/*
 * AdamW for the parameters the optimizer split sends away from Muon (the
 * dev.to page's table in section "2. ตัวปรับปรุง Muon": embeddings, lm_head
 * and scalar parameters go to AdamW).  The pages give no formula; the reading
 * is decoupled weight decay with bias-corrected moments, step t >= 1:
 *   p  <- p (1 - lr wd)
 *   m  <- beta1 m + (1 - beta1) g
 *   v  <- beta2 v + (1 - beta2) g^2
 *   p  <- p - (lr / (1 - beta1^t)) m / (sqrt(v / (1 - beta2^t)) + eps)
 * Everything in double; p, m, v are rounded to float where they are stored.
 */
void oracle_adamw(long n_elem, float* p, const float* g, float* m, float* v, double lr, double beta1,
                  double beta2, double eps, double weight_decay, int step) {
    const double bc1 = 1.0 - pow(beta1, (double)step);
    const double bc2 = 1.0 - pow(beta2, (double)step);
#pragma omp parallel for schedule(static)
    for (long e = 0; e < n_elem; ++e) {
        double pd = (double)p[e] * (1.0 - lr * weight_decay);
        const double gd = (double)g[e];
        const double md = beta1 * (double)m[e] + (1.0 - beta1) * gd;
        const double vd = beta2 * (double)v[e] + (1.0 - beta2) * gd * gd;
        pd -= (lr / bc1) * md / (sqrt(vd / bc2) + eps);
        p[e] = (float)pd;
        m[e] = (float)md;
        v[e] = (float)vd;
    }
}

/*
 * NorMuon variance scaling of an orthogonalised update O (stored r x c layout),
 * as the apidog.com page's section "2. Pengoptimal Muon" (paragraph "Reduksi
 * Varians NorMuon") and the dev.to page's "NorMuon variance scaling" sketch
 * it: after orthogonalisation the update is normalised per neuron.  The
 * sketch leaves red_dim, the second-moment state, step_size and v_norm_new
 * undefined; the reading taken here:
 *   a neuron is a stored row (an output unit): v_mean_i = mean_j O_ij^2
 *   V_i   <- beta2 V_i + (1 - beta2) v_mean_i      (state across steps, float)
 *   step_i = 1 / sqrt(V_i + eps)
 *   v_norm     = sqrt(sum_i v_mean_i)
 *   v_norm_new = sqrt(sum_i v_mean_i step_i^2)     (the same statistic of O * step)
 *   O'_ij = O_ij step_i v_norm / max(v_norm_new, 1e-10)
 * which keeps ||O'||_F = ||O||_F.  V is rounded to float where it is stored.
 * O is overwritten by O'.  All sums in index order.
 */
void oracle_normuon_scale(int r, int c, double* O, float* V, double beta2, double eps) {
    double* vm = (double*)malloc(sizeof(double) * (size_t)r);
    double* st = (double*)malloc(sizeof(double) * (size_t)r);
    if (!vm || !st) {
        free(vm);
        free(st);
        return;
    }
    double s_old = 0.0, s_new = 0.0;
    for (int i = 0; i < r; ++i) {
        double s = 0.0;
        for (int j = 0; j < c; ++j) s += O[(size_t)i * c + j] * O[(size_t)i * c + j];
        vm[i] = s / (double)c;
        const double Vn = beta2 * (double)V[i] + (1.0 - beta2) * vm[i];
        V[i] = (float)Vn;
        st[i] = 1.0 / sqrt(Vn + eps);
        s_old += vm[i];
        s_new += vm[i] * st[i] * st[i];
    }
    const double v_norm = sqrt(s_old);
    const double v_norm_new = sqrt(s_new);
    const double ratio = v_norm / (v_norm_new > 1e-10 ? v_norm_new : 1e-10);
    for (int i = 0; i < r; ++i)
        for (int j = 0; j < c; ++j) O[(size_t)i * c + j] *= st[i] * ratio;
    free(vm);
    free(st);
}

/*
 * One Muon step with NorMuon scaling: as oracle_muon_matrix, with O replaced
 * by its NorMuon-scaled O' before the update p' = p - lr sqrt(max(1, r/c)) O'.
 * V (r floats) is the per-row second-moment state, updated in place.
 */
int oracle_normuon_matrix(int r, int c, const float* p, const float* g, const float* m, double lr, double beta,
                          int nesterov, int mode, int K, const double* coeffs, double eps, float* V,
                          double beta2, double eps2, float* p_out, float* m_out, double* O_out) {
    const size_t rc = (size_t)r * c;
    double* u = (double*)malloc(sizeof(double) * rc);
    double* O = O_out ? O_out : (double*)malloc(sizeof(double) * rc);
    if (!u || !O) {
        free(u);
        if (!O_out) free(O);
        return -1;
    }
    oracle_momentum((long)rc, g, m, beta, nesterov, mode, m_out, u);
    int rcode = oracle_orthogonalize(r, c, u, K, coeffs, eps, O);
    if (rcode == 0) {
        oracle_normuon_scale(r, c, O, V, beta2, eps2);
        const double scale = lr * oracle_aspect_scale(r, c);
        for (size_t e = 0; e < rc; ++e) p_out[e] = (float)((double)p[e] - scale * O[e]);
    }
    free(u);
    if (!O_out) free(O);
    return rcode;
}
