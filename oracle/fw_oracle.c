/*
 * fw_oracle.c -- plain, slow, fp64 CPU oracle for the causal fast-weight
 * memory recurrence.  TEST INFRASTRUCTURE ONLY: this file is built and called
 * by the test suite, by the package's smoke check and by the benchmark's CPU
 * baseline leg.  No product code path links, loads or calls it, and it shares
 * no code, header or constant with the CUDA library.
 *
 * Everything is computed in double precision, one token at a time, exactly in
 * the order the pages state the rule.  Chains (one (batch, head) pair each)
 * are independent; the only parallelism is a pthread pool over chains.
 *
 * Sources (page title, section):
 *  - "Fast Weight Attention for Continual Learning" (paper reading), §3.2 and
 *    §4.2: instantaneous ridge loss l_t(S) = 1/2 |S^T x_t - y_t|^2
 *    + (lambda_t/2)|S|_F^2 and its one normalised gradient step (Falcon-1)
 *        S_t = (1 - eta_t lambda_t) S_{t-1} + eta_t x_t r_t^T,
 *        r_t = y_t - S_{t-1}^T x_t,
 *        eta_t = beta_t / (|x_t|^2 + lambda_t + eps).
 *  - same page, §1.4 and §4.1: read after write (o_t = S_t^T q_t), the
 *    shifted training pair (x_t, y_t) = (phi(k_{t-1}), v_t), and the boundary
 *    x_1 := 0, eta_1 := 0 (the first token's write is a no-op).
 *  - same page, §4.2: Falcon-2, a step per value channel j,
 *        eta_{j,t} = beta_{j,t} / (|x_t|^2 + lambda_t + eps),
 *    with the residual r_t and the feature x_t shared: column j of S takes
 *    its own scalar write S[:,j] = (1 - eta_{j,t} lambda_t) S[:,j]
 *    + eta_{j,t} x_t r_{t,j}.
 *  - same page, §4.3: the inner-product family (Falcon-1A): the loss
 *    -<S^T x_t, y_t> + (lambda/2)|S|^2 gives the additive write
 *        S_t = (1 - eta_t lambda_t) S_{t-1} + eta_t x_t y_t^T
 *    (no residual); the normalised step is kept as a write-size stabiliser.
 *  - same page, §3.3 and §4.1: the 2 x 2 design read-after-write /
 *    read-before-write x same-step pair / shifted pair.
 *  - same page, §4.2: Falcon-3, one minibatch gradient step on the average
 *    loss of the last W causal pairs (the window), with the step set by the
 *    window's exact smoothness,
 *        S_t = (1 - eta_t lambda_t) S_{t-1}
 *              + (eta_t / B_t) sum_{j in window} x_j (y_j - S_{t-1}^T x_j)^T,
 *        eta_t = beta_t / (mu_t + lambda_t + eps),
 *        mu_t = lambda_max((1/B_t) sum_{j in window} x_j x_j^T);
 *    §4.3: Falcon-3A, the same window, step and decay with the additive
 *    write (y_j in place of the residual).
 *  - "Attention is also an FFN" blog, §2.1 and §4.1: plain linear attention
 *    S_i = S_{i-1} + phi(k_i) v_i^T, y_i = phi(q_i)^T S_i, with the feature
 *    map phi(x) = elu(x) + 1, and the state kept in floating point.
 *
 * Readings where the pages leave a step open:
 *  - phi is applied to the key only in Falcon-1 mode (the read uses q_t as
 *    is); in linear-attention mode it is applied to both q and k, never to v.
 *  - gamma_t = 1 - eta_t lambda_t is used as is, without a clamp; it can be
 *    zero or negative when lambda_t is large against |x_t|^2.
 *  - a decode step has no notion of position: it applies the formula with
 *    the key it is given (a caller starting a sequence passes beta = 0).
 *  - an optional k_init replaces the zero pair of the first token (so that a
 *    prefill can continue a previous one); then eta_1 follows the formula.
 *  - Falcon-1A takes Falcon-1's eta_t, pairing and boundary; only the write
 *    drops the residual (r_t := y_t).  Falcon-2A is Falcon-2 with that
 *    additive write.
 *  - Falcon-2 keeps lambda_t shared by the channels (the page gives only beta
 *    a channel index) and Falcon-1's pairing and boundary.
 *  - read-before-write (no formula printed): o_t = S_{t-1}^T q_t, the read
 *    taken before token t's write.
 *  - same-step pair (no formula printed): x_t = phi(k_t) for every t; the
 *    first token then has a pair of its own (no boundary rule, k_init unused).
 *  - Falcon-3's window at token t holds the pairs t-W+1 .. t that exist: the
 *    first token's shifted pair does not (x_1 := 0 is no pair), nor do pairs
 *    before the sequence; B_t counts the pairs that do, and eta_t := 0 when
 *    there are none.  With W = 1 this is exactly Falcon-1.  A window carried
 *    in from an earlier call supplies the pairs before this call's first
 *    token.  mu_t is found from the B_t x B_t Gram matrix of the window's
 *    keys, whose nonzero eigenvalues are those of the d_k x d_k window
 *    covariance (X X^T and X^T X share them), by cyclic Jacobi rotations
 *    (Golub and Van Loan, the symmetric Schur decomposition) run to
 *    convergence.
 *  - Falcon-3's lambda_t and beta_t are one per token (the window variant of
 *    the scalar step).
 *
 * Layouts (all contiguous, row-major, double):
 *   q, k   [nc][T][dk]     v, o   [nc][T][dv]     beta, lam [nc][T]
 *   beta of Falcon-2 / 2A: [nc][T][dv]
 *   S0, S  [nc][dk][dv]    k_init [nc][dk]
 *   Falcon-3 window carry: x [nc][W-1][dk], y [nc][W-1][dv] (oldest first,
 *   phi already applied to x), n [nc] = how many of the newest slots hold a
 *   pair; slots that hold none are ignored on input and zero on output.
 * S[i][j] is key row i, value column j; reads are o_j = sum_i S[i][j] q_i.
 */
#include <math.h>
#include <pthread.h>
#include <stdlib.h>
#include <string.h>

enum { ORC_PHI_IDENTITY = 0, ORC_PHI_ELU1 = 1 };
enum { ORC_FALCON1 = 0, ORC_LINATTN = 1, ORC_FALCON1A = 2, ORC_FALCON2 = 3, ORC_FALCON2A = 4,
       ORC_FALCON3 = 5, ORC_FALCON3A = 6 };
enum { ORC_RBW = 1, ORC_SAME_PAIR = 2 };

/* elu(z) + 1: z + 1 for z > 0, exp(z) for z <= 0 (blog §4.1). */
static double orc_phi(int phi, double z)
{
    if (phi == ORC_PHI_ELU1) return z > 0.0 ? z + 1.0 : exp(z);
    return z;
}

/* S^T q into out (a read of the state as it stands). */
static void read_state(int dk, int dv, const double *S, const double *q, double *out)
{
    int i, j;
    for (j = 0; j < dv; ++j) {
        double c = 0.0;
        for (i = 0; i < dk; ++i) c += S[(size_t)i * dv + j] * q[i];
        out[j] = c;
    }
}

/* One Falcon-1 / Falcon-1A chain (inner == 1: no residual), token by token.
 * chan == 1: Falcon-2 / 2A, beta is [T][dv] and every value channel takes its
 * own step and decay; eta_v, gamma_v are dv scratch values. */
static void falcon1_chain(long T, int dk, int dv, const double *q, const double *k,
                          const double *v, const double *beta, const double *lam,
                          const double *S0, const double *k_init, int phi, double eps,
                          int inner, int chan, int flags, double *o, double *S, double *x,
                          double *r, double *eta_v, double *gamma_v)
{
    long t;
    int i, j;
    const int rbw = (flags & ORC_RBW) != 0, same = (flags & ORC_SAME_PAIR) != 0;
    if (S0) memcpy(S, S0, sizeof(double) * (size_t)dk * dv);
    else memset(S, 0, sizeof(double) * (size_t)dk * dv);

    for (t = 0; t < T; ++t) {
        double n = 0.0;
        const double *kprev = same ? k + t * dk : (t > 0) ? k + (t - 1) * dk : k_init;
        if (rbw) read_state(dk, dv, S, q + t * dk, o + t * dv);   /* read before write */
        if (kprev) {
            for (i = 0; i < dk; ++i) x[i] = orc_phi(phi, kprev[i]);
            for (i = 0; i < dk; ++i) n += x[i] * x[i];
        } else {
            for (i = 0; i < dk; ++i) x[i] = 0.0; /* x_1 := 0, eta_1 := 0 */
        }
        for (j = 0; j < dv; ++j) {
            const double b = chan ? beta[t * dv + j] : beta[t];
            eta_v[j] = kprev ? b / (n + lam[t] + eps) : 0.0;
            gamma_v[j] = 1.0 - eta_v[j] * lam[t];
        }
        /* residual against the state before the write (Falcon-1A: the target) */
        for (j = 0; j < dv; ++j) {
            double a = 0.0;
            if (!inner)
                for (i = 0; i < dk; ++i) a += S[(size_t)i * dv + j] * x[i];
            r[j] = v[t * dv + j] - a;
        }
        /* the write, column by column */
        for (i = 0; i < dk; ++i)
            for (j = 0; j < dv; ++j)
                S[(size_t)i * dv + j] = gamma_v[j] * S[(size_t)i * dv + j] + eta_v[j] * x[i] * r[j];
        if (!rbw) read_state(dk, dv, S, q + t * dk, o + t * dv);   /* read after write */
    }
}

/* One plain linear-attention chain: S += phi(k_t) v_t^T, o_t = S^T phi(q_t)
 * (read before the write with ORC_RBW). */
static void linattn_chain(long T, int dk, int dv, const double *q, const double *k,
                          const double *v, const double *S0, int phi, int flags,
                          double *o, double *S, double *x, double *qt)
{
    long t;
    int i, j;
    const int rbw = (flags & ORC_RBW) != 0;
    if (S0) memcpy(S, S0, sizeof(double) * (size_t)dk * dv);
    else memset(S, 0, sizeof(double) * (size_t)dk * dv);
    for (t = 0; t < T; ++t) {
        for (i = 0; i < dk; ++i) x[i] = orc_phi(phi, k[t * dk + i]);
        for (i = 0; i < dk; ++i) qt[i] = orc_phi(phi, q[t * dk + i]);
        if (rbw) read_state(dk, dv, S, qt, o + t * dv);
        for (i = 0; i < dk; ++i)
            for (j = 0; j < dv; ++j)
                S[(size_t)i * dv + j] += x[i] * v[t * dv + j];
        if (!rbw) read_state(dk, dv, S, qt, o + t * dv);
    }
}

/* One decode step of one state (in place); qt is scratch for phi(q).  beta
 * points at this state's step size (Falcon-2 / 2A: dv of them). */
static void step_one(int mode, int flags, int dk, int dv, const double *q, const double *kp,
                     const double *v, const double *beta, double lam, int phi, double eps,
                     double *S, double *o, double *x, double *r, double *qt)
{
    int i, j;
    const int rbw = (flags & ORC_RBW) != 0;
    if (mode == ORC_LINATTN) {
        for (i = 0; i < dk; ++i) x[i] = orc_phi(phi, kp[i]);
        for (i = 0; i < dk; ++i) qt[i] = orc_phi(phi, q[i]);
        if (rbw) read_state(dk, dv, S, qt, o);
        for (i = 0; i < dk; ++i)
            for (j = 0; j < dv; ++j) S[(size_t)i * dv + j] += x[i] * v[j];
        if (!rbw) read_state(dk, dv, S, qt, o);
        return;
    }
    {
        const int chan = (mode == ORC_FALCON2 || mode == ORC_FALCON2A);
        const int inner = (mode == ORC_FALCON1A || mode == ORC_FALCON2A);
        double n = 0.0;
        for (i = 0; i < dk; ++i) x[i] = orc_phi(phi, kp[i]);
        for (i = 0; i < dk; ++i) n += x[i] * x[i];
        if (rbw) read_state(dk, dv, S, q, o);
        for (j = 0; j < dv; ++j) {
            double a = 0.0;
            if (!inner)
                for (i = 0; i < dk; ++i) a += S[(size_t)i * dv + j] * x[i];
            r[j] = v[j] - a;
        }
        for (j = 0; j < dv; ++j) {
            const double eta = (chan ? beta[j] : beta[0]) / (n + lam + eps);
            const double gamma = 1.0 - eta * lam;
            for (i = 0; i < dk; ++i)
                S[(size_t)i * dv + j] = gamma * S[(size_t)i * dv + j] + eta * x[i] * r[j];
        }
        if (!rbw) read_state(dk, dv, S, q, o);
    }
}

/* ---- Falcon-3 / 3A: the sliding window --------------------------------- */

/* Largest eigenvalue of the symmetric n x n matrix A (row-major, destroyed):
 * cyclic Jacobi sweeps, each rotation J chosen so that (J^T A J)_pq = 0, until
 * the off-diagonal mass is negligible; the diagonal then holds the spectrum. */
static double sym_max_eig(int n, double *A)
{
    int sweep, p, q, k;
    double best;
    for (sweep = 0; sweep < 100; ++sweep) {
        double off = 0.0, diag = 0.0;
        for (p = 0; p < n; ++p)
            for (q = 0; q < n; ++q) {
                if (p == q) diag += A[p * n + q] * A[p * n + q];
                else off += A[p * n + q] * A[p * n + q];
            }
        if (off <= 1e-32 * diag || off == 0.0) break;
        for (p = 0; p < n - 1; ++p)
            for (q = p + 1; q < n; ++q) {
                const double apq = A[p * n + q];
                double tau, t, c, s;
                if (apq == 0.0) continue;
                tau = (A[q * n + q] - A[p * n + p]) / (2.0 * apq);
                t = (tau >= 0.0 ? 1.0 : -1.0) / (fabs(tau) + sqrt(1.0 + tau * tau));
                c = 1.0 / sqrt(1.0 + t * t);
                s = t * c;
                for (k = 0; k < n; ++k) { /* A <- A J (columns p, q) */
                    const double akp = A[k * n + p], akq = A[k * n + q];
                    A[k * n + p] = c * akp - s * akq;
                    A[k * n + q] = s * akp + c * akq;
                }
                for (k = 0; k < n; ++k) { /* A <- J^T A (rows p, q) */
                    const double apk = A[p * n + k], aqk = A[q * n + k];
                    A[p * n + k] = c * apk - s * aqk;
                    A[q * n + k] = s * apk + c * aqk;
                }
            }
    }
    best = A[0];
    for (p = 1; p < n; ++p)
        if (A[p * n + p] > best) best = A[p * n + p];
    return best;
}

/* One Falcon-3 / 3A write of S (dk x dv) with the nb pairs (wx[j], wy[j]) of
 * the window (nb may be 0: no write).  Returns mu_t (0 without pairs).
 * G (nb*nb) and r (nb*dv) are scratch. */
static double window_write(int dk, int dv, int nb, const double *const *wx,
                           const double *const *wy, double beta, double lam, double eps,
                           int inner, double *S, double *G, double *r)
{
    int a, b, i, j;
    double mu, eta, gamma, c;
    if (nb == 0) return 0.0; /* eta_t = 0: S is left as it is */
    for (a = 0; a < nb; ++a)
        for (b = 0; b < nb; ++b) {
            double g = 0.0;
            for (i = 0; i < dk; ++i) g += wx[a][i] * wx[b][i];
            G[a * nb + b] = g / nb; /* window-average covariance, Gram form */
        }
    mu = sym_max_eig(nb, G);
    eta = beta / (mu + lam + eps);
    gamma = 1.0 - eta * lam;
    c = eta / nb;
    /* residuals against the state before the write (Falcon-3A: the targets) */
    for (a = 0; a < nb; ++a)
        for (j = 0; j < dv; ++j) {
            double s = 0.0;
            if (!inner)
                for (i = 0; i < dk; ++i) s += S[(size_t)i * dv + j] * wx[a][i];
            r[a * dv + j] = wy[a][j] - s;
        }
    for (i = 0; i < dk; ++i)
        for (j = 0; j < dv; ++j) {
            double upd = 0.0;
            for (a = 0; a < nb; ++a) upd += wx[a][i] * r[a * dv + j];
            S[(size_t)i * dv + j] = gamma * S[(size_t)i * dv + j] + c * upd;
        }
    return mu;
}

/* Pair m of a Falcon-3 prefill (m < 0: from the carried window) into x, y.
 * Returns 1 if the pair exists, else 0 (x, y zero). */
static int window_pair(long m, int W, int dk, int dv, const double *k, const double *v,
                       const double *k_init, const double *cx, const double *cy, int cn,
                       int phi, int same, double *x, double *y)
{
    int i, have = 0;
    const double *kp = NULL;
    if (m < 0) {
        const long slot = m + W - 1;
        if (cx && slot >= W - 1 - cn) {
            memcpy(x, cx + slot * dk, sizeof(double) * dk);
            memcpy(y, cy + slot * dv, sizeof(double) * dv);
            return 1;
        }
    } else {
        kp = same ? k + m * dk : (m > 0) ? k + (m - 1) * dk : k_init;
        if (kp) {
            for (i = 0; i < dk; ++i) x[i] = orc_phi(phi, kp[i]);
            memcpy(y, v + m * dv, sizeof(double) * dv);
            have = 1;
        }
    }
    if (!have) {
        memset(x, 0, sizeof(double) * dk);
        memset(y, 0, sizeof(double) * dv);
    }
    return have;
}

/* One Falcon-3 / 3A chain; scratch px (W*dk), py (W*dv), G (W*W), r (W*dv). */
static void falcon3_chain(long T, int dk, int dv, int W, const double *q, const double *k,
                          const double *v, const double *beta, const double *lam,
                          const double *S0, const double *k_init, const double *cx,
                          const double *cy, int cn, int phi, double eps, int inner, int flags,
                          double *o, double *S, double *ox, double *oy, int *on, double *mu,
                          double *px, double *py, double *G, double *r)
{
    long t;
    int j;
    const int rbw = (flags & ORC_RBW) != 0, same = (flags & ORC_SAME_PAIR) != 0;
    const double *wx[64], *wy[64];
    if (S0) memcpy(S, S0, sizeof(double) * (size_t)dk * dv);
    else memset(S, 0, sizeof(double) * (size_t)dk * dv);
    for (t = 0; t < T; ++t) {
        int nb = 0;
        double m;
        for (j = 0; j < W; ++j) /* pairs t-W+1 .. t */
            if (window_pair(t - W + 1 + j, W, dk, dv, k, v, k_init, cx, cy, cn, phi, same,
                            px + (size_t)nb * dk, py + (size_t)nb * dv)) {
                wx[nb] = px + (size_t)nb * dk;
                wy[nb] = py + (size_t)nb * dv;
                ++nb;
            }
        if (rbw) read_state(dk, dv, S, q + t * dk, o + t * dv);
        m = window_write(dk, dv, nb, wx, wy, beta[t], lam[t], eps, inner, S, G, r);
        if (mu) mu[t] = m;
        if (!rbw) read_state(dk, dv, S, q + t * dk, o + t * dv);
    }
    if (ox) { /* the window after token T: pairs T-W+1 .. T-1 */
        int n = 0;
        for (j = 0; j < W - 1; ++j)
            n += window_pair(T - (W - 1) + j, W, dk, dv, k, v, k_init, cx, cy, cn, phi, same,
                             ox + (size_t)j * dk, oy + (size_t)j * dv);
        *on = n;
    }
}

/* One Falcon-3 / 3A decode step (in place on S): the window is the carried
 * pairs plus the new pair (phi(k_prev), y); the carry moves on by one. */
static void step3_one(int dk, int dv, int W, int inner, int flags, const double *q,
                      const double *kp, const double *y, double beta, double lam, int phi,
                      double eps, double *S, const double *cx, const double *cy, int cn,
                      double *o, double *ox, double *oy, int *on, double *px, double *G,
                      double *r)
{
    int i, j, nb = 0;
    const int rbw = (flags & ORC_RBW) != 0;
    const double *wx[64], *wy[64];
    for (j = 0; j < W - 1; ++j)
        if (cx && j >= W - 1 - cn) {
            wx[nb] = cx + (size_t)j * dk;
            wy[nb] = cy + (size_t)j * dv;
            ++nb;
        }
    for (i = 0; i < dk; ++i) px[i] = orc_phi(phi, kp[i]);
    wx[nb] = px;
    wy[nb] = y;
    ++nb;
    if (rbw) read_state(dk, dv, S, q, o);
    window_write(dk, dv, nb, wx, wy, beta, lam, eps, inner, S, G, r);
    if (!rbw) read_state(dk, dv, S, q, o);
    if (ox) {
        for (j = 0; j < W - 2; ++j) { /* slot j <- slot j + 1 */
            const int have = cx && (j + 1 >= W - 1 - cn);
            for (i = 0; i < dk; ++i) ox[(size_t)j * dk + i] = have ? cx[(size_t)(j + 1) * dk + i] : 0.0;
            for (i = 0; i < dv; ++i) oy[(size_t)j * dv + i] = have ? cy[(size_t)(j + 1) * dv + i] : 0.0;
        }
        if (W > 1) {
            memcpy(ox + (size_t)(W - 2) * dk, px, sizeof(double) * dk);
            memcpy(oy + (size_t)(W - 2) * dv, y, sizeof(double) * dv);
        }
        *on = (cn + 1 < W - 1) ? cn + 1 : W - 1;
    }
}

/* ---- thread pool over independent chains ------------------------------- */

typedef struct {
    int kind; /* 0 prefill falcon1 / 1a / 2 / 2a, 1 prefill linattn, 2 step,
                 3 prefill falcon3 / 3a, 4 falcon3 / 3a step */
    long nc, T;
    int dk, dv, phi, mode, flags;
    double eps;
    const double *q, *k, *v, *beta, *lam, *S0, *k_init;
    double *o, *S;
    /* Falcon-3 / 3A */
    int W;
    const double *cx, *cy;
    const int *cn;
    double *ox, *oy, *mu_t;
    int *on;
    long next;
    pthread_mutex_t mu;
} orc_job;

static void *orc_worker(void *arg)
{
    orc_job *J = (orc_job *)arg;
    int dk = J->dk, dv = J->dv;
    const int W = J->W > 0 ? J->W : 1;
    double *x = (double *)malloc(sizeof(double) * (size_t)(dk + dv + dk + 2 * dv));
    double *r = x + dk, *qt = r + dv, *eta_v = qt + dk, *gamma_v = eta_v + dv;
    double *px = (double *)malloc(sizeof(double) * (size_t)(W * (dk + 2 * dv) + W * W));
    double *py = px + (size_t)W * dk, *r3 = py + (size_t)W * dv, *G = r3 + (size_t)W * dv;
    const int inner3 = (J->mode == ORC_FALCON3A);
    const int chan = (J->mode == ORC_FALCON2 || J->mode == ORC_FALCON2A);
    const long bstride = chan ? (long)dv : 1;
    for (;;) {
        long c;
        pthread_mutex_lock(&J->mu);
        c = J->next++;
        pthread_mutex_unlock(&J->mu);
        if (c >= J->nc) break;
        if (J->kind == 0) {
            falcon1_chain(J->T, dk, dv, J->q + c * J->T * dk, J->k + c * J->T * dk,
                          J->v + c * J->T * dv, J->beta + c * J->T * bstride, J->lam + c * J->T,
                          J->S0 ? J->S0 + (size_t)c * dk * dv : NULL,
                          J->k_init ? J->k_init + (size_t)c * dk : NULL, J->phi, J->eps,
                          J->mode == ORC_FALCON1A || J->mode == ORC_FALCON2A, chan, J->flags,
                          J->o + c * J->T * dv, J->S + (size_t)c * dk * dv, x, r, eta_v, gamma_v);
        } else if (J->kind == 1) {
            linattn_chain(J->T, dk, dv, J->q + c * J->T * dk, J->k + c * J->T * dk,
                          J->v + c * J->T * dv, J->S0 ? J->S0 + (size_t)c * dk * dv : NULL,
                          J->phi, J->flags, J->o + c * J->T * dv, J->S + (size_t)c * dk * dv,
                          x, qt);
        } else if (J->kind == 3) {
            const size_t cs = (size_t)(W - 1);
            falcon3_chain(J->T, dk, dv, W, J->q + c * J->T * dk, J->k + c * J->T * dk,
                          J->v + c * J->T * dv, J->beta + c * J->T, J->lam + c * J->T,
                          J->S0 ? J->S0 + (size_t)c * dk * dv : NULL,
                          J->k_init ? J->k_init + (size_t)c * dk : NULL,
                          J->cx ? J->cx + c * cs * dk : NULL, J->cy ? J->cy + c * cs * dv : NULL,
                          J->cn ? J->cn[c] : 0, J->phi, J->eps, inner3, J->flags,
                          J->o + c * J->T * dv, J->S + (size_t)c * dk * dv,
                          J->ox ? J->ox + c * cs * dk : NULL, J->oy ? J->oy + c * cs * dv : NULL,
                          J->on ? J->on + c : NULL, J->mu_t ? J->mu_t + c * J->T : NULL,
                          px, py, G, r3);
        } else if (J->kind == 4) {
            const size_t cs = (size_t)(W - 1);
            step3_one(dk, dv, W, inner3, J->flags, J->q + (size_t)c * dk, J->k + (size_t)c * dk,
                      J->v + (size_t)c * dv, J->beta[c], J->lam[c], J->phi, J->eps,
                      J->S + (size_t)c * dk * dv, J->cx ? J->cx + c * cs * dk : NULL,
                      J->cy ? J->cy + c * cs * dv : NULL, J->cn ? J->cn[c] : 0,
                      J->o + (size_t)c * dv, J->ox ? J->ox + c * cs * dk : NULL,
                      J->oy ? J->oy + c * cs * dv : NULL, J->on ? J->on + c : NULL, px, G, r3);
        } else {
            step_one(J->mode, J->flags, dk, dv, J->q + (size_t)c * dk, J->k + (size_t)c * dk,
                     J->v + (size_t)c * dv, J->beta ? J->beta + c * bstride : NULL,
                     J->lam ? J->lam[c] : 0.0, J->phi, J->eps,
                     J->S + (size_t)c * dk * dv, J->o + (size_t)c * dv, x, r, qt);
        }
    }
    free(x);
    free(px);
    return NULL;
}

static void orc_run(orc_job *J, int nthreads)
{
    int i;
    pthread_t th[256];
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    if (nthreads > J->nc) nthreads = (int)(J->nc > 0 ? J->nc : 1);
    J->next = 0;
    pthread_mutex_init(&J->mu, NULL);
    if (nthreads == 1) {
        orc_worker(J);
    } else {
        for (i = 0; i < nthreads; ++i) pthread_create(&th[i], NULL, orc_worker, J);
        for (i = 0; i < nthreads; ++i) pthread_join(th[i], NULL);
    }
    pthread_mutex_destroy(&J->mu);
}

/* ---- exported entry points --------------------------------------------- */

/* Falcon-1 / 1A / 2 / 2A prefill (mode ORC_FALCON1, ORC_FALCON1A, ORC_FALCON2,
 * ORC_FALCON2A; beta is [nc][T][dv] for the last two) over nc independent
 * chains; flags: ORC_RBW, ORC_SAME_PAIR.  S0, k_init may be NULL. */
void orc_falcon1(long nc, long T, int dk, int dv, const double *q, const double *k,
                 const double *v, const double *beta, const double *lam, const double *S0,
                 const double *k_init, int phi, double eps, int mode, int flags, double *o,
                 double *S_T, int nthreads)
{
    orc_job J;
    memset(&J, 0, sizeof(J));
    J.kind = 0; J.nc = nc; J.T = T; J.dk = dk; J.dv = dv; J.phi = phi; J.eps = eps;
    J.mode = mode; J.flags = flags;
    J.q = q; J.k = k; J.v = v; J.beta = beta; J.lam = lam; J.S0 = S0; J.k_init = k_init;
    J.o = o; J.S = S_T;
    orc_run(&J, nthreads);
}

/* Plain linear-attention prefill over nc chains (flags: ORC_RBW).  S0 may be NULL. */
void orc_linattn(long nc, long T, int dk, int dv, const double *q, const double *k,
                 const double *v, const double *S0, int phi, int flags, double *o,
                 double *S_T, int nthreads)
{
    orc_job J;
    memset(&J, 0, sizeof(J));
    J.kind = 1; J.nc = nc; J.T = T; J.dk = dk; J.dv = dv; J.phi = phi; J.flags = flags;
    J.q = q; J.k = k; J.v = v; J.S0 = S0; J.o = o; J.S = S_T;
    orc_run(&J, nthreads);
}

/* One decode step for ns independent states (flags: ORC_RBW; beta is [ns][dv]
 * for ORC_FALCON2 / ORC_FALCON2A); S is updated in place. */
void orc_step(long ns, int dk, int dv, int mode, int flags, const double *q,
              const double *k_prev, const double *v, const double *beta, const double *lam,
              int phi, double eps, double *S, double *o, int nthreads)
{
    orc_job J;
    memset(&J, 0, sizeof(J));
    J.kind = 2; J.nc = ns; J.T = 1; J.dk = dk; J.dv = dv; J.mode = mode; J.phi = phi;
    J.flags = flags;
    J.eps = eps; J.q = q; J.k = k_prev; J.v = v; J.beta = beta; J.lam = lam;
    J.o = o; J.S = S;
    orc_run(&J, nthreads);
}

/* Falcon-3 / 3A prefill (mode ORC_FALCON3, ORC_FALCON3A) with a window of W
 * pairs (1 <= W <= 64) over nc chains; flags: ORC_RBW, ORC_SAME_PAIR.
 * S0, k_init, the carried window (cx, cy, cn), the window after the last token
 * (ox, oy, on) and mu [nc][T] (the mu_t of every token) may be NULL. */
void orc_falcon3(long nc, long T, int dk, int dv, int W, const double *q, const double *k,
                 const double *v, const double *beta, const double *lam, const double *S0,
                 const double *k_init, const double *cx, const double *cy, const int *cn,
                 int phi, double eps, int mode, int flags, double *o, double *S_T, double *ox,
                 double *oy, int *on, double *mu, int nthreads)
{
    orc_job J;
    memset(&J, 0, sizeof(J));
    J.kind = 3; J.nc = nc; J.T = T; J.dk = dk; J.dv = dv; J.W = W; J.phi = phi; J.eps = eps;
    J.mode = mode; J.flags = flags;
    J.q = q; J.k = k; J.v = v; J.beta = beta; J.lam = lam; J.S0 = S0; J.k_init = k_init;
    J.cx = cx; J.cy = cy; J.cn = cn; J.ox = ox; J.oy = oy; J.on = on; J.mu_t = mu;
    J.o = o; J.S = S_T;
    orc_run(&J, nthreads);
}

/* One Falcon-3 / 3A decode step for ns states (flags: ORC_RBW); S is updated
 * in place; the carried window (cx, cy, cn; NULL = empty) moves on into
 * (ox, oy, on) (NULL = not wanted). */
void orc_step3(long ns, int dk, int dv, int W, int mode, int flags, const double *q,
               const double *k_prev, const double *v, const double *beta, const double *lam,
               int phi, double eps, double *S, const double *cx, const double *cy,
               const int *cn, double *o, double *ox, double *oy, int *on, int nthreads)
{
    orc_job J;
    memset(&J, 0, sizeof(J));
    J.kind = 4; J.nc = ns; J.T = 1; J.dk = dk; J.dv = dv; J.W = W; J.mode = mode; J.phi = phi;
    J.flags = flags; J.eps = eps;
    J.q = q; J.k = k_prev; J.v = v; J.beta = beta; J.lam = lam;
    J.cx = cx; J.cy = cy; J.cn = cn; J.ox = ox; J.oy = oy; J.on = on;
    J.o = o; J.S = S;
    orc_run(&J, nthreads);
}
