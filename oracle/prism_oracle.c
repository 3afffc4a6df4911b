/*
 * PRISM memory-recurrence forward -- sequential fp64 CPU oracle.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the CPU
 * baseline leg of the benchmark may build, load or call this file.  It shares
 * no code, header, table or helper with the CUDA library.
 *
 * What it computes, per (batch, head), one token at a time, exactly as the
 * method is defined ("PRISM: Parallel Residual Iterative Sequence Model",
 * arXiv 2602.10796; reading notes at liuzhao09.github.io/papers/prism.html,
 * section 2.2 "Write-Forget Decoupling" and section 2.3 "Input-Anchored
 * Simulation"; the Tencent article at youzy.cn, part 03 "PRISM" items
 * two to four):
 *
 *   anchor    h_t = sum_{j=0..3} w_j (.) v_{t-j}        (v_{t-j} for t - j < 0 from
 *             the optional history v_hist, else zero)
 *             The short causal convolution over v is the input-local proxy
 *             that stands in for S_{t-1} k_t (notes, section 2.3).
 *   gain      g_t = GELU'(h_t) = Phi(h_t) + h_t phi(h_t)  (exact erf GELU)
 *   residual  e_t = v_t - GELU(h_t) = v_t - h_t Phi(h_t)
 *   chain     r_{t,1} = e_t,  r_{t,l+1} = r_{t,l} (.) (1 - eta_{t,l} g_t)
 *             The GELU is absorbed into a per-channel preconditioner, so the
 *             chain is an element-wise linear recursion (article part 03,
 *             item three; digest ai-engineering-6yk.pages.dev, "eliminating
 *             step-to-step serialism").
 *   transition  S <- alpha_t (S - beta_t (S k_t) k_t^T)   (GDN forget path,
 *             notes section 2.2: A_t = alpha_t (I - beta_t k_t k_t^T))
 *   injection   S += beta_t v_t k_t^T + sum_{l=1..L-1} gamma_{t,l} (g_t (.) r_{t,l}) u_{t,l}^T
 *             (rank accumulation, notes section 2.2; the first term is the
 *             standard GDN write, article part 03 item four)
 *   readout   o_t = S_t q_t  (post-update state)
 *
 * Non-linear residual variant (optional input p_gain, notes section 2.3: a gain vector
 * p_{t,l} predicted from the anchor replaces GELU'(h), and each level takes a non-linear
 * step off the residual, "greedy residual subtraction"):
 *   delta_{t,l} = GELU(p_{t,l} (.) r_{t,l}),  r_{t,l+1} = r_{t,l} - delta_{t,l},
 *   injection factor of level l: gamma_{t,l} delta_{t,l}      (eta is not read)
 * Everything else (anchor, r_{t,1} = e_t, transition, GDN write, readout) is unchanged.
 *
 * Storage (row-major, contiguous), R = L - 1:
 *   q, k   [B,H,T,dk]      v, out [B,H,T,dv]      u [B,H,T,R,dk]
 *   beta, alpha [B,H,T]    gamma, eta [B,H,T,R]   conv_w [H,4,dv] (tap j
 *   multiplies v_{t-j}).  Slot l-1 of gamma/u/eta holds level l.  The last
 *   eta slot (level L-1) would only shape a residual that nothing uses, so
 *   it is never read.
 * Optional outputs (NULL to skip):
 *   S_final [B,H,dv,dk]   the state after the last token
 *   X_out   [B,H,T,R,dv]  injection factors x_{t,l} = gamma_{t,l} g_t (.) r_{t,l}
 *   h_out, g_out, e_out [B,H,T,dv]  anchor, gain and residual
 *   S_init  [B,H,dv,dk]   optional initial state (NULL means S_0 = 0)
 *   p_gain  [B,H,T,R,dv]  optional gains of the non-linear variant (slot l-1: level l)
 *   v_hist  [B,H,3,dv]    optional left context of the convolution: slot j holds
 *                         v_{j-3} (oldest first), the last three tokens before this
 *                         call's first one (NULL means zeros).  With S_init it lets
 *                         a sequence be evaluated in consecutive calls: the result
 *                         equals one call over the whole sequence.
 *
 * Build: gcc -O2 -fno-fast-math -shared -fPIC prism_oracle.c -lm -lpthread
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
    int B, H, T, dk, dv, L;
    const double *q, *k, *v, *beta, *alpha, *u, *gamma, *eta, *p_gain, *conv_w, *v_hist, *S_init;
    double *out, *S_final, *X_out, *h_out, *g_out, *e_out;
    int nthreads;
    int thread_id;
} oracle_args;

/* One (batch, head) sequence, token by token. */
static void run_head(const oracle_args *a, int b, int h)
{
    const int T = a->T, dk = a->dk, dv = a->dv, L = a->L, R = L - 1;
    const size_t bh = (size_t)b * a->H + h;
    const double *q = a->q + bh * T * dk;
    const double *k = a->k + bh * T * dk;
    const double *v = a->v + bh * T * dv;
    const double *beta = a->beta + bh * T;
    const double *alpha = a->alpha + bh * T;
    const double *u = R > 0 ? a->u + bh * T * R * dk : NULL;
    const double *gamma = R > 0 ? a->gamma + bh * T * R : NULL;
    const double *eta = (R > 0 && a->eta) ? a->eta + bh * T * R : NULL;
    const double *pg = (R > 0 && a->p_gain) ? a->p_gain + bh * T * R * dv : NULL;
    const double *w = a->conv_w + (size_t)h * 4 * dv;
    const double *vh = a->v_hist ? a->v_hist + bh * 3 * dv : NULL;
    double *out = a->out + bh * T * dv;

    double *S = calloc((size_t)dv * dk, sizeof(double));
    double *anchor = malloc(sizeof(double) * dv);
    double *g = malloc(sizeof(double) * dv);
    double *e = malloc(sizeof(double) * dv);
    double *r = malloc(sizeof(double) * dv);
    double *Sk = malloc(sizeof(double) * dv);
    if (a->S_init)
        memcpy(S, a->S_init + bh * dv * dk, sizeof(double) * dv * dk);

    const double inv_sqrt2 = 0.70710678118654752440;
    const double inv_sqrt2pi = 0.39894228040143267794;

    for (int t = 0; t < T; ++t) {
        const double *vt = v + (size_t)t * dv;
        const double *kt = k + (size_t)t * dk;
        const double *qt = q + (size_t)t * dk;

        /* anchor, gain and residual, channel by channel */
        for (int c = 0; c < dv; ++c) {
            double acc = 0.0;
            for (int j = 0; j < 4; ++j)
                if (t - j >= 0) acc += w[j * dv + c] * v[(size_t)(t - j) * dv + c];
                else if (vh) acc += w[j * dv + c] * vh[(size_t)(3 + t - j) * dv + c];
            anchor[c] = acc;
            double Phi = 0.5 * (1.0 + erf(acc * inv_sqrt2));
            double phi = exp(-0.5 * acc * acc) * inv_sqrt2pi;
            g[c] = Phi + acc * phi;
            e[c] = vt[c] - acc * Phi;
            r[c] = e[c];
        }
        if (a->h_out) memcpy(a->h_out + (bh * T + t) * dv, anchor, sizeof(double) * dv);
        if (a->g_out) memcpy(a->g_out + (bh * T + t) * dv, g, sizeof(double) * dv);
        if (a->e_out) memcpy(a->e_out + (bh * T + t) * dv, e, sizeof(double) * dv);

        /* forget path: S <- alpha (S - beta (S k) k^T), then the GDN write */
        const double al = alpha[t], be = beta[t];
        for (int i = 0; i < dv; ++i) {
            double s = 0.0;
            for (int j = 0; j < dk; ++j) s += S[(size_t)i * dk + j] * kt[j];
            Sk[i] = s;
        }
        for (int i = 0; i < dv; ++i)
            for (int j = 0; j < dk; ++j)
                S[(size_t)i * dk + j] = al * (S[(size_t)i * dk + j] - be * Sk[i] * kt[j])
                                      + be * vt[i] * kt[j];

        /* rank accumulation over the refinement levels l = 1..L-1 */
        for (int l = 1; l <= R; ++l) {
            const double gm = gamma[(size_t)t * R + (l - 1)];
            const double *ul = u + ((size_t)t * R + (l - 1)) * dk;
            const double *pl = pg ? pg + ((size_t)t * R + (l - 1)) * dv : NULL;
            for (int i = 0; i < dv; ++i) {
                double x = gm * g[i] * r[i];
                if (pl) { /* non-linear variant: delta = GELU(p r), r <- r - delta */
                    const double z = pl[i] * r[i];
                    const double delta = z * 0.5 * (1.0 + erf(z * inv_sqrt2));
                    x = gm * delta;
                    r[i] -= delta;
                }
                if (a->X_out) a->X_out[((bh * T + t) * R + (l - 1)) * dv + i] = x;
                for (int j = 0; j < dk; ++j) S[(size_t)i * dk + j] += x * ul[j];
            }
            if (!pl && l < R) {
                const double et = eta[(size_t)t * R + (l - 1)];
                for (int i = 0; i < dv; ++i) r[i] *= (1.0 - et * g[i]);
            }
        }

        /* readout from the post-update state */
        for (int i = 0; i < dv; ++i) {
            double s = 0.0;
            for (int j = 0; j < dk; ++j) s += S[(size_t)i * dk + j] * qt[j];
            out[(size_t)t * dv + i] = s;
        }
    }
    if (a->S_final) memcpy(a->S_final + bh * dv * dk, S, sizeof(double) * dv * dk);
    free(S); free(anchor); free(g); free(e); free(r); free(Sk);
}

static void *worker(void *p)
{
    const oracle_args *a = (const oracle_args *)p;
    const int units = a->B * a->H;
    for (int idx = a->thread_id; idx < units; idx += a->nthreads)
        run_head(a, idx / a->H, idx % a->H);
    return NULL;
}

/* Returns 0 on success, a negative number for bad arguments. */
int prism_oracle_forward_f64(int B, int H, int T, int dk, int dv, int L,
                             const double *q, const double *k, const double *v,
                             const double *beta, const double *alpha,
                             const double *u, const double *gamma, const double *eta,
                             const double *p_gain, const double *conv_w, const double *v_hist,
                             const double *S_init,
                             double *out, double *S_final, double *X_out,
                             double *h_out, double *g_out, double *e_out, int nthreads)
{
    if (B < 0 || H < 0 || T < 0 || dk <= 0 || dv <= 0 || L < 1) return -1;
    if (!q || !k || !v || !beta || !alpha || !conv_w || !out) return -2;
    if (L > 1 && (!u || !gamma || (!eta && !p_gain))) return -3;
    const int units = B * H;
    if (units == 0) return 0;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > units) nthreads = units;

    oracle_args base = {B, H, T, dk, dv, L, q, k, v, beta, alpha, u, gamma, eta, p_gain, conv_w, v_hist, S_init,
                        out, S_final, X_out, h_out, g_out, e_out, nthreads, 0};
    if (nthreads == 1) {
        worker(&base);
        return 0;
    }
    pthread_t *th = malloc(sizeof(pthread_t) * nthreads);
    oracle_args *args = malloc(sizeof(oracle_args) * nthreads);
    for (int i = 0; i < nthreads; ++i) {
        args[i] = base;
        args[i].thread_id = i;
        pthread_create(&th[i], NULL, worker, &args[i]);
    }
    for (int i = 0; i < nthreads; ++i) pthread_join(th[i], NULL);
    free(th);
    free(args);
    return 0;
}
