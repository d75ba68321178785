/*
 * la_oracle.c -- plain fp64 CPU oracle for causal kernelised linear attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file: only the test-suite, the smoke check and the CPU-baseline
 * leg of the benchmark use it.  It shares no code, header, table or helper
 * with the CUDA library; inputs arrive as fp64 arrays holding exactly the
 * values the GPU reads (bf16 / fp32 upcast without rounding).
 *
 * What it computes, and where the pages define it:
 *
 *   phi(x) = elu(x) + 1 with alpha = 1, evaluated as max(x,0) + exp(min(x,0))
 *     ("Linear Attention Kernel", section "Choice of phi";
 *      "Efficient Attention Variants", section 10, feature map of the
 *      verification program).
 *
 *   causal recurrence, write-then-read (the j <= t mask):
 *     S_t = S_{t-1} + phi(k_t) v_t^T,  z_t = z_{t-1} + phi(k_t),
 *     o_t = phi(q_t)^T S_t / phi(q_t)^T z_t,  S_0 = 0, z_0 = 0
 *     ("Efficient Attention Variants", section 5, prefix-sum recurrence;
 *      "Linear Attention Kernel", section "Recurrent form").
 *
 *   non-causal reassociation: S = sum_j phi(k_j) v_j^T, z = sum_j phi(k_j),
 *     o_i = phi(q_i)^T S / phi(q_i)^T z
 *     ("Efficient Attention Variants", section 4;
 *      "Linear Attention Kernel", section "Rewrite: associativity").
 *
 *   scalar decay (RetNet): S_t = gamma S_{t-1} + k_t v_t^T, o_t = q_t^T S_t,
 *     no feature map and no normaliser
 *     ("Efficient Attention Variants", section 7.1 RetNet).
 *
 *   per-key-channel decay (GLA form): S_t = diag(alpha_t) S_{t-1} + k_t v_t^T,
 *     alpha_t in (0,1]^d scales row i of the state (key feature i) and is
 *     broadcast along the value channels
 *     ("Efficient Attention Variants", section 7.2 GLA; "Linear Attention and
 *      SSM", list of phi choices, RWKV-5/6 state M_s = diag(w) M_{s-1} + ...).
 *
 *   initial state: every recurrence may start from a given (S_0, z_0) instead
 *     of zero -- the state is the whole summary of the prefix, so a sequence
 *     can be processed in pieces ("Efficient Attention Variants", sections 1
 *     and 5: a fixed-size state replaces the history).
 *
 *   positive random features (Performer): with x = u / d^(1/4) and Gaussian
 *     rows w_1..w_r (passed in, drawn by the caller),
 *     phi(u)_j = exp(w_j^T x - |x|^2 / 2) / sqrt(r), whose inner products
 *     estimate exp(q^T k / sqrt(d)) without bias
 *     ("Efficient Attention Variants", section 6 Performer).
 *
 *   explicit N x N masked kernel matrix (the object the method avoids), used
 *     only as a brute-force cross-check on tiny inputs:
 *     A_ij = phi(q_i)^T phi(k_j) * L_ij,  O = A V / rowsum(A)
 *     ("Efficient Attention Variants", section 10, dense evaluation;
 *      "Linear Attention and SSM", eq. attn-linssm-ssd, structured mask L).
 *
 * Readings where the pages are silent (each also listed in the design notes):
 *   - feature_map ORC_FM_IDENTITY_NORM uses phi = identity with the
 *     normaliser, so that the hand-worked example of "Efficient Attention
 *     Variants" section 5.1 (which gives phi(k_j), phi(q_3) directly) can be
 *     reproduced.
 *   - feature_map ORC_FM_NONE is phi = identity without normaliser (RetNet).
 *   - a decay gamma combined with a normalised map decays z with the same
 *     gamma, i.e. the mask L_ij = gamma^(i-j) multiplies numerator and
 *     denominator alike.
 *   - no 1/sqrt(d) scaling anywhere: the linear forms on the pages have none
 *     (the random-feature map scales by d^(-1/4) itself, as its page does).
 *   - per-channel decay with a normalised map decays z_i with alpha_t,i, as
 *     the scalar case decays z with gamma.
 *   - an initial state is continued exactly as if its prefix had been run
 *     through the recurrence; the non-causal form takes none.
 *
 * Planted-mistake hooks (ORC_PLANT_*) exist only so that the test-suite can
 * build deliberately wrong variants of this file and check that its pins
 * reject each of them.  The normal build defines none of them.
 */
#include <math.h>
#include <pthread.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

enum { ORC_FM_ELU1 = 0, ORC_FM_IDENTITY_NORM = 1, ORC_FM_NONE = 2 };

enum { ORC_OK = 0, ORC_ERR_ARG = 1, ORC_ERR_NONPOSITIVE_DEN = 2 };

/* ---------------------------------------------------------------- phi ---- */

static double orc_phi1(double x, int fm)
{
    if (fm != ORC_FM_ELU1)
        return x;
#ifdef ORC_PLANT_PHI_NO_PLUS_ONE
    return x > 0.0 ? x : exp(x) - 1.0;
#else
    /* elu(x) + 1 = max(x,0) + exp(min(x,0)); no large positive exponent. */
    return (x > 0.0 ? x : 0.0) + exp(x < 0.0 ? x : 0.0);
#endif
}

/* Elementwise feature map, exported so that tests can compare it with an
 * independent library ELU. */
void orc_phi(const double* x, double* y, long n, int fm)
{
    for (long i = 0; i < n; ++i)
        y[i] = orc_phi1(x[i], fm);
}

static int orc_normalised(int fm) { return fm == ORC_FM_ELU1 || fm == ORC_FM_IDENTITY_NORM; }

static int orc_check_dims(long B, long H, long N, long d, long dv, int fm)
{
    if (B < 1 || H < 1 || N < 0 || d < 1 || dv < 1)
        return ORC_ERR_ARG;
    if (fm != ORC_FM_ELU1 && fm != ORC_FM_IDENTITY_NORM && fm != ORC_FM_NONE)
        return ORC_ERR_ARG;
    return ORC_OK;
}

/* ------------------------------------------------- one (b,h) sequence ---- */

/*
 * Token-by-token recurrence over one sequence, starting from the state (S, z)
 * it is given and leaving the final state there.  S is d x dv row-major
 * (S[i*dv + c] pairs key feature i with value channel c), z has d entries.
 * out (N x dv) may be NULL when only the state is wanted.
 * Returns ORC_ERR_NONPOSITIVE_DEN if a normalised read met den <= 0 (the
 * output of that row is then num/den as computed, possibly inf/nan).
 */
static int orc_seq_recurrence(const double* q, const double* k, const double* v, double* out,
                              double* S, double* z, long N, long d, long dv, int fm, double gamma,
                              const double* alpha, double* f, double* g, double* num)
{
    int rc = ORC_OK;
    const int norm = orc_normalised(fm);
    for (long t = 0; t < N; ++t) {
        for (long i = 0; i < d; ++i) {
            f[i] = orc_phi1(k[t * d + i], fm);
            if (q)
                g[i] = orc_phi1(q[t * d + i], fm);
        }
#ifdef ORC_PLANT_READ_BEFORE_WRITE
        if (out) {
            for (long c = 0; c < dv; ++c) {
                double s = 0.0;
                for (long i = 0; i < d; ++i)
                    s += g[i] * S[i * dv + c];
                num[c] = s;
            }
            double den = 0.0;
            for (long i = 0; i < d; ++i)
                den += g[i] * z[i];
            for (long c = 0; c < dv; ++c)
                out[t * dv + c] = norm ? num[c] / den : num[c];
        }
#endif
        /* write: S <- a S + phi(k_t) v_t^T ; z <- a z + phi(k_t), with a the
         * scalar gamma or, per row i of the state, alpha_t,i */
        for (long i = 0; i < d; ++i) {
            if (alpha)
                gamma = alpha[t * d + i];
            for (long c = 0; c < dv; ++c) {
#ifdef ORC_PLANT_GLA_ALONG_VALUES
                if (alpha)
                    gamma = alpha[t * d + (c % d)];
#endif
#ifdef ORC_PLANT_DECAY_AFTER_WRITE
                S[i * dv + c] = gamma * (S[i * dv + c] + f[i] * v[t * dv + c]);
#elif defined(ORC_PLANT_TRANSPOSED_UPDATE)
                /* pairs feature i with the wrong value channel when d != dv */
                S[i * dv + c] = gamma * S[i * dv + c] + f[c % d] * v[t * dv + (i % dv)];
#else
                S[i * dv + c] = gamma * S[i * dv + c] + f[i] * v[t * dv + c];
#endif
            }
#ifdef ORC_PLANT_Z_NO_DECAY
            z[i] = z[i] + f[i];
#else
            z[i] = gamma * z[i] + f[i];
#endif
        }
#ifndef ORC_PLANT_READ_BEFORE_WRITE
        /* read: o_t = phi(q_t)^T S_t / phi(q_t)^T z_t */
        if (out) {
            for (long c = 0; c < dv; ++c) {
                double s = 0.0;
                for (long i = 0; i < d; ++i)
                    s += g[i] * S[i * dv + c];
                num[c] = s;
            }
            double den = 0.0;
            for (long i = 0; i < d; ++i)
                den += g[i] * z[i];
#ifdef ORC_PLANT_DROP_NORMALISER
            den = 1.0;
#endif
            if (norm && !(den > 0.0))
                rc = ORC_ERR_NONPOSITIVE_DEN;
            for (long c = 0; c < dv; ++c)
                out[t * dv + c] = norm ? num[c] / den : num[c];
        }
#endif
    }
    return rc;
}

/* Non-causal form over one sequence: reduce the whole sequence first, then
 * let every query read the same S, z. */
static int orc_seq_noncausal(const double* q, const double* k, const double* v, double* out,
                             long N, long d, long dv, int fm, double* S, double* z, double* f,
                             double* g, double* num)
{
    int rc = ORC_OK;
    const int norm = orc_normalised(fm);
    memset(S, 0, sizeof(double) * d * dv);
    memset(z, 0, sizeof(double) * d);
    orc_seq_recurrence(NULL, k, v, NULL, S, z, N, d, dv, fm, 1.0, NULL, f, g, num);
    for (long t = 0; t < N; ++t) {
        for (long i = 0; i < d; ++i)
            g[i] = orc_phi1(q[t * d + i], fm);
        double den = 0.0;
        for (long i = 0; i < d; ++i)
            den += g[i] * z[i];
        if (norm && !(den > 0.0))
            rc = ORC_ERR_NONPOSITIVE_DEN;
        for (long c = 0; c < dv; ++c) {
            double s = 0.0;
            for (long i = 0; i < d; ++i)
                s += g[i] * S[i * dv + c];
            out[t * dv + c] = norm ? s / den : s;
        }
    }
    return rc;
}

/* ------------------------------------------- threads over (b,h) slices ---- */

enum { JOB_FORWARD = 0, JOB_STATE = 1, JOB_DECODE = 2 };

typedef struct {
    int kind;
    const double *q, *k, *v;
    double *out, *S, *z;
    const double* gamma;
    const double* alpha;   /* [B,H,N,d] per-channel decay, or NULL */
    const double *S0, *z0; /* [B,H,d,dv], [B,H,d] initial state, or NULL */
    long B, H, N, d, dv;
    int fm, causal, init_from_state;
    long next; /* shared work counter */
    pthread_mutex_t lock;
    int rc;
} orc_job;

static void* orc_worker(void* arg)
{
    orc_job* J = (orc_job*)arg;
    const long d = J->d, dv = J->dv, N = J->N;
    double* S = J->kind == JOB_FORWARD ? (double*)malloc(sizeof(double) * d * dv) : NULL;
    double* z = J->kind == JOB_FORWARD ? (double*)malloc(sizeof(double) * d) : NULL;
    double* f = (double*)malloc(sizeof(double) * d);
    double* g = (double*)malloc(sizeof(double) * d);
    double* num = (double*)malloc(sizeof(double) * dv);
    for (;;) {
        pthread_mutex_lock(&J->lock);
        long s = J->next++;
        pthread_mutex_unlock(&J->lock);
        if (s >= J->B * J->H)
            break;
        const long h = s % J->H;
        const double gamma = J->gamma ? J->gamma[h] : 1.0;
        const double* alpha = J->alpha ? J->alpha + s * N * d : NULL;
        int rc = ORC_OK;
        if (J->kind == JOB_FORWARD) {
            const double* q = J->q + s * N * d;
            const double* k = J->k + s * N * d;
            const double* v = J->v + s * N * dv;
            double* o = J->out + s * N * dv;
            if (J->causal) {
                if (J->S0) {
                    memcpy(S, J->S0 + s * d * dv, sizeof(double) * d * dv);
#ifdef ORC_PLANT_IGNORE_Z0
                    memset(z, 0, sizeof(double) * d);
#else
                    memcpy(z, J->z0 + s * d, sizeof(double) * d);
#endif
                } else {
                    memset(S, 0, sizeof(double) * d * dv);
                    memset(z, 0, sizeof(double) * d);
                }
                rc = orc_seq_recurrence(q, k, v, o, S, z, N, d, dv, J->fm, gamma, alpha, f, g,
                                        num);
            } else {
                rc = orc_seq_noncausal(q, k, v, o, N, d, dv, J->fm, S, z, f, g, num);
            }
        } else if (J->kind == JOB_STATE) {
            double* Ss = J->S + s * d * dv;
            double* zs = J->z + s * d;
            if (!J->init_from_state) {
                memset(Ss, 0, sizeof(double) * d * dv);
                memset(zs, 0, sizeof(double) * d);
            }
            rc = orc_seq_recurrence(NULL, J->k + s * N * d, J->v + s * N * dv, NULL, Ss, zs, N, d,
                                    dv, J->fm, gamma, alpha, f, g, num);
        } else { /* JOB_DECODE: one token per sequence, state in place */
            rc = orc_seq_recurrence(J->q + s * d, J->k + s * d, J->v + s * dv, J->out + s * dv,
                                    J->S + s * d * dv, J->z + s * d, 1, d, dv, J->fm, gamma,
                                    alpha, f, g, num);
        }
        if (rc != ORC_OK) {
            pthread_mutex_lock(&J->lock);
            J->rc = rc;
            pthread_mutex_unlock(&J->lock);
        }
    }
    free(S);
    free(z);
    free(f);
    free(g);
    free(num);
    return NULL;
}

static int orc_run(orc_job* J, int nthreads)
{
    long work = J->B * J->H;
    if (nthreads <= 0)
        nthreads = (int)sysconf(_SC_NPROCESSORS_ONLN);
    if (nthreads < 1)
        nthreads = 1;
    if (nthreads > work)
        nthreads = (int)work;
    J->next = 0;
    J->rc = ORC_OK;
    pthread_mutex_init(&J->lock, NULL);
    if (nthreads <= 1) {
        orc_worker(J);
    } else {
        pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * nthreads);
        for (int i = 0; i < nthreads; ++i)
            pthread_create(&th[i], NULL, orc_worker, J);
        for (int i = 0; i < nthreads; ++i)
            pthread_join(th[i], NULL);
        free(th);
    }
    pthread_mutex_destroy(&J->lock);
    return J->rc;
}

/* ------------------------------------------------------- public entry ---- */

/*
 * Forward over B*H independent sequences.
 *   q, k : [B,H,N,d]   v, out : [B,H,N,dv]   gamma : [H] or NULL (= 1)
 *   alpha : [B,H,N,d] per-channel decay or NULL (not together with gamma)
 *   S0, z0 : [B,H,d,dv], [B,H,d] state before the first token, or NULL (= 0);
 *            both or neither
 *   causal = 1: recurrence (write then read); causal = 0: reassociation.
 * Decay or an initial state with causal = 0 is not defined by the pages and
 * is rejected.  nthreads <= 0 uses every online core.
 */
int orc_forward(const double* q, const double* k, const double* v, double* out, long B, long H,
                long N, long d, long dv, int causal, int fm, const double* gamma,
                const double* alpha, const double* S0, const double* z0, int nthreads)
{
    if (orc_check_dims(B, H, N, d, dv, fm) != ORC_OK || (gamma && alpha) || (!S0 != !z0))
        return ORC_ERR_ARG;
    if (!causal && (gamma || alpha || S0))
        return ORC_ERR_ARG;
    orc_job J;
    memset(&J, 0, sizeof J);
    J.kind = JOB_FORWARD;
    J.q = q, J.k = k, J.v = v, J.out = out, J.gamma = gamma;
    J.alpha = alpha, J.S0 = S0, J.z0 = z0;
    J.B = B, J.H = H, J.N = N, J.d = d, J.dv = dv, J.fm = fm, J.causal = causal;
    return orc_run(&J, nthreads);
}

/*
 * State after a prefix: S [B,H,d,dv], z [B,H,d] (alpha: [B,H,N,d] or NULL).
 * With init_from_state = 0
 * the recurrence starts at S_0 = 0, z_0 = 0 (the arrays are overwritten);
 * with init_from_state = 1 it continues from the values passed in.
 */
int orc_state(const double* k, const double* v, double* S, double* z, long B, long H, long N,
              long d, long dv, int fm, const double* gamma, const double* alpha,
              int init_from_state, int nthreads)
{
    if (orc_check_dims(B, H, N, d, dv, fm) != ORC_OK || (gamma && alpha))
        return ORC_ERR_ARG;
    orc_job J;
    memset(&J, 0, sizeof J);
    J.kind = JOB_STATE;
    J.k = k, J.v = v, J.S = S, J.z = z, J.gamma = gamma, J.alpha = alpha;
    J.B = B, J.H = H, J.N = N, J.d = d, J.dv = dv, J.fm = fm;
    J.init_from_state = init_from_state;
    return orc_run(&J, nthreads);
}

/*
 * One decode step for B*H sequences: q, k [B,H,d], v, out [B,H,dv], alpha
 * [B,H,d] or NULL; S, z are updated in place (write, then read), exactly one iteration of the causal
 * recurrence.
 */
int orc_decode_step(double* S, double* z, const double* q, const double* k, const double* v,
                    double* out, long B, long H, long d, long dv, int fm, const double* gamma,
                    const double* alpha, int nthreads)
{
    if (orc_check_dims(B, H, 1, d, dv, fm) != ORC_OK || (gamma && alpha))
        return ORC_ERR_ARG;
    orc_job J;
    memset(&J, 0, sizeof J);
    J.kind = JOB_DECODE;
    J.q = q, J.k = k, J.v = v, J.out = out, J.S = S, J.z = z, J.gamma = gamma;
    J.alpha = alpha;
    J.B = B, J.H = H, J.N = 1, J.d = d, J.dv = dv, J.fm = fm;
    return orc_run(&J, nthreads);
}

/*
 * Brute force over one sequence with the explicit N x N kernel matrix:
 *   A_ij = phi(q_i)^T phi(k_j) * L_ij,  L_ij = gamma^(i-j) for j <= i
 *   (causal) or 1 for all j (non-causal, gamma must be 1),
 *   O = A V / rowsum(A) for normalised maps, O = A V otherwise.
 * weights (N x N) may be NULL; if given it receives A (divided by its row
 * sums for normalised maps), the per-token attention weights.
 * Memory O(N^2): for tiny inputs only.
 */
int orc_dense(const double* q, const double* k, const double* v, double* out, double* weights,
              long N, long d, long dv, int causal, int fm, double gamma)
{
    if (orc_check_dims(1, 1, N, d, dv, fm) != ORC_OK || (!causal && gamma != 1.0))
        return ORC_ERR_ARG;
    int rc = ORC_OK;
    const int norm = orc_normalised(fm);
    double* A = (double*)malloc(sizeof(double) * (N ? N : 1) * (N ? N : 1));
    double* fq = (double*)malloc(sizeof(double) * (N ? N : 1) * d);
    double* fk = (double*)malloc(sizeof(double) * (N ? N : 1) * d);
    orc_phi(q, fq, N * d, fm);
    orc_phi(k, fk, N * d, fm);
    for (long i = 0; i < N; ++i) {
        double rowsum = 0.0;
        for (long j = 0; j < N; ++j) {
            double a = 0.0;
            for (long c = 0; c < d; ++c)
                a += fq[i * d + c] * fk[j * d + c];
            double mask = 1.0;
            if (causal)
                mask = j <= i ? pow(gamma, (double)(i - j)) : 0.0;
            A[i * N + j] = a * mask;
            rowsum += A[i * N + j];
        }
        if (norm && !(rowsum > 0.0))
            rc = ORC_ERR_NONPOSITIVE_DEN;
        for (long c = 0; c < dv; ++c) {
            double s = 0.0;
            for (long j = 0; j < N; ++j)
                s += A[i * N + j] * v[j * dv + c];
            out[i * dv + c] = norm ? s / rowsum : s;
        }
        if (weights)
            for (long j = 0; j < N; ++j)
                weights[i * N + j] = norm ? A[i * N + j] / rowsum : A[i * N + j];
    }
    free(A);
    free(fq);
    free(fk);
    return rc;
}

/*
 * Positive random features of n vectors u (rows of x, each d long) with r
 * Gaussian rows w (r x d, drawn by the caller):
 *   x' = u / d^(1/4),  y_j = exp(w_j^T x' - |x'|^2 / 2) / sqrt(r)
 * so that y(q)^T y(k) estimates exp(q^T k / sqrt(d)) without bias
 * ("Efficient Attention Variants", section 6).  y is n x r.
 */
void orc_favor(const double* x, const double* w, double* y, long n, long d, long r)
{
    const double s = 1.0 / pow((double)d, 0.25);
    const double inv_sqrt_r = 1.0 / sqrt((double)r);
    for (long t = 0; t < n; ++t) {
        double nrm = 0.0;
        for (long i = 0; i < d; ++i)
            nrm += (x[t * d + i] * s) * (x[t * d + i] * s);
        for (long j = 0; j < r; ++j) {
            double p = 0.0;
            for (long i = 0; i < d; ++i)
                p += w[j * d + i] * (x[t * d + i] * s);
#ifdef ORC_PLANT_FAVOR_NO_NORM
            y[t * r + j] = exp(p) * inv_sqrt_r;
#else
            y[t * r + j] = exp(p - 0.5 * nrm) * inv_sqrt_r;
#endif
        }
    }
}
