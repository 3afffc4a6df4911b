/*
 * PRISM memory-recurrence backward -- sequential fp64 CPU oracle.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the CPU
 * baseline leg of the benchmark may build, load or call this file.  It shares
 * no code, header, table or helper with the CUDA library.
 *
 * The forward it differentiates is the linear-chain PRISM recurrence
 * ("PRISM: Parallel Residual Iterative Sequence Model", arXiv 2602.10796;
 * reading notes at liuzhao09.github.io/papers/prism.html, sections 2.2 and
 * 2.3; the Tencent article at youzy.cn, part 03 "PRISM", items two to four),
 * per (batch, head), token by token:
 *
 *   h_t = sum_j w_j (.) v_{t-j}          g_t = Phi(h_t) + h_t phi(h_t)
 *   e_t = v_t - h_t Phi(h_t)             r_{t,1} = e_t,  r_{t,l+1} = r_{t,l} (.) (1 - eta_{t,l} g_t)
 *   x_{t,l} = gamma_{t,l} g_t (.) r_{t,l}
 *   S_t = alpha_t (S_{t-1} - beta_t (S_{t-1} k_t) k_t^T) + beta_t v_t k_t^T + sum_l x_{t,l} u_{t,l}^T
 *   o_t = S_t q_t
 *
 * Given the cotangents dO = dLoss/do (and optionally dS_final = dLoss/dS_T),
 * this file returns dLoss/d of every input by reverse-mode differentiation of
 * those steps, in the reverse order of the forward: the state cotangent dS
 * (the derivative with respect to S_t) is carried backwards through
 *   dS_{t-1} = alpha_t (dS_t - beta_t (dS_t k_t) k_t^T)
 * after the readout term dO_t q_t^T has been added to it.  With
 * P = S_{t-1}, y = P k_t and z = dS_t k_t (dS_t including the readout term):
 *   dq_t    = S_t^T dO_t
 *   dbeta_t = v_t . z - alpha_t y . z
 *   dalpha_t = <dS_t, P> - beta_t y . z
 *   dk_t    = dS_t^T (beta_t v_t - alpha_t beta_t y) - alpha_t beta_t P^T z
 *   dv_t   += beta_t z                                   (the GDN write)
 *   dx_{t,l} = dS_t u_{t,l},   du_{t,l} = dS_t^T x_{t,l}
 * then, channel by channel, the residual chain backwards (l = R .. 1, with the
 * cotangent of r_{t,R+1} equal to zero because nothing reads it):
 *   dr_{t,l}  = gamma_{t,l} g dx_{t,l} + (1 - eta_{t,l} g) dr_{t,l+1}
 *   dg       += gamma_{t,l} r_{t,l} dx_{t,l} - eta_{t,l} r_{t,l} dr_{t,l+1}
 *   dgamma_{t,l} = sum_c g r_{t,l} dx_{t,l}
 *   deta_{t,l}   = -sum_c g r_{t,l} dr_{t,l+1}
 *   dv_t += dr_{t,1},   dh_t = -g dr_{t,1} + phi(h_t) (2 - h_t^2) dg
 * (d e / d h = -(Phi + h phi) = -g and d g / d h = phi (2 - h^2)), and the
 * convolution backwards: dv_{t-j} += w_j (.) dh_t, dw_j += dh_t (.) v_{t-j},
 * where v_{t-j} with t - j < 0 is the history v_hist (zero when absent); the
 * cotangent of those history slots is returned in dv_hist.
 * dS_init is the state cotangent after token 0 has been processed.
 *
 * Non-linear residual variant (optional input p_gain [B,H,T,R,dv], notes section
 * 2.3; eta is then not read): r_{t,1} = e_t, delta_{t,l} = GELU(p_{t,l} (.) r_{t,l}),
 * x_{t,l} = gamma_{t,l} delta_{t,l}, r_{t,l+1} = r_{t,l} - delta_{t,l}.  Its chain
 * backwards, l = R .. 1 (the cotangent of r_{t,R+1} is zero), with z = p (.) r_{t,l}:
 *   ddelta = gamma_{t,l} dx_{t,l} - dr_{t,l+1},   dgamma_{t,l} = sum_c delta dx_{t,l}
 *   dz = ddelta GELU'(z),   dp_{t,l} = dz (.) r_{t,l},   dr_{t,l} = dr_{t,l+1} + dz (.) p
 * then dv_t += dr_{t,1} and dh_t = -g dr_{t,1} (the gain GELU'(h) is not used by this
 * chain); the cotangent of p_gain is returned in dp_gain instead of deta.
 *
 * The pre-update states S_{t-1} of one (batch, head) are all kept from a first
 * forward pass (T dv dk doubles).
 *
 * Storage: as the forward oracle (q, k [B,H,T,dk]; v, dout [B,H,T,dv];
 * u, du [B,H,T,R,dk]; beta, alpha [B,H,T]; gamma, eta [B,H,T,R]; conv_w
 * [H,4,dv]; S_init, dS_final, dS_init [B,H,dv,dk]; v_hist, dv_hist [B,H,3,dv]).
 * Every gradient has the layout of its input.  deta[..., R-1] is 0: that gain
 * is never read (as in the forward), so it may hold anything, NaN included.
 * Optional pointers may be NULL: S_init, v_hist (zeros), dS_final (zero),
 * dv_hist, dS_init (not returned).
 *
 * Build: gcc -O2 -fno-fast-math -shared -fPIC prism_oracle_bwd.c -lm -lpthread
 */
#include <math.h>
#include <pthread.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
    int B, H, T, dk, dv, L;
    const double *q, *k, *v, *beta, *alpha, *u, *gamma, *eta, *p_gain, *conv_w, *v_hist, *S_init, *dout, *dS_final;
    double *dq, *dk_, *dv_, *dbeta, *dalpha, *du, *dgamma, *deta, *dp_gain, *dconv_part, *dv_hist, *dS_init;
    int nthreads, thread_id, status;
} bwd_args;

static double Phi_of(double h) { return 0.5 * (1.0 + erf(h * 0.70710678118654752440)); }
static double phi_of(double h) { return exp(-0.5 * h * h) * 0.39894228040143267794; }

static void run_head(bwd_args *a, int b, int h)
{
    const int T = a->T, dk = a->dk, dv = a->dv, R = a->L - 1;
    const size_t bh = (size_t)b * a->H + h, DD = (size_t)dv * dk;
    const double *q = a->q + bh * T * dk, *k = a->k + bh * T * dk, *v = a->v + bh * T * dv;
    const double *beta = a->beta + bh * T, *alpha = a->alpha + bh * T;
    const double *u = R > 0 ? a->u + bh * T * R * dk : NULL;
    const double *gamma = R > 0 ? a->gamma + bh * T * R : NULL;
    const double *eta = (R > 0 && a->eta) ? a->eta + bh * T * R : NULL;
    const double *pg = (R > 0 && a->p_gain) ? a->p_gain + bh * T * R * dv : NULL;
    const double *w = a->conv_w + (size_t)h * 4 * dv;
    const double *vh = a->v_hist ? a->v_hist + bh * 3 * dv : NULL;
    const double *dO = a->dout + bh * T * dv;
    double *dq = a->dq + bh * T * dk, *dkk = a->dk_ + bh * T * dk, *dvv = a->dv_ + bh * T * dv;
    double *dbeta = a->dbeta + bh * T, *dalpha = a->dalpha + bh * T;
    double *du = R > 0 ? a->du + bh * T * R * dk : NULL;
    double *dgamma = R > 0 ? a->dgamma + bh * T * R : NULL;
    double *deta = (R > 0 && !pg) ? a->deta + bh * T * R : NULL;
    double *dpg = (R > 0 && pg) ? a->dp_gain + bh * T * R * dv : NULL;
    double *dw = a->dconv_part + bh * 4 * dv;

    double *Sprev = malloc(sizeof(double) * DD * (size_t)T);  /* S_{t-1} for every t */
    double *S = calloc(DD, sizeof(double));
    double *dS = calloc(DD, sizeof(double));
    double *hh = malloc(sizeof(double) * (size_t)T * dv);
    double *xs = malloc(sizeof(double) * (size_t)T * (R > 0 ? R : 1) * dv);
    double *rs = malloc(sizeof(double) * (size_t)(R > 0 ? R : 1) * dv);
    double *dx = malloc(sizeof(double) * (size_t)(R > 0 ? R : 1) * dv);
    double *dh = calloc((size_t)T * dv, sizeof(double));
    double *y = malloc(sizeof(double) * dv), *z = malloc(sizeof(double) * dv);
    if (!Sprev || !S || !dS || !hh || !xs || !rs || !dx || !dh || !y || !z) {
        a->status = -9;
        goto done;
    }
    if (a->S_init) memcpy(S, a->S_init + bh * DD, sizeof(double) * DD);

    /* forward: anchors, injection factors and the pre-update states */
    for (int t = 0; t < T; ++t) {
        const double *vt = v + (size_t)t * dv, *kt = k + (size_t)t * dk;
        double *ht = hh + (size_t)t * dv, *xt = xs + (size_t)t * (R > 0 ? R : 1) * dv;
        for (int c = 0; c < dv; ++c) {
            double s = 0.0;
            for (int j = 0; j < 4; ++j) {
                const int src = t - j;
                const double vv = src >= 0 ? v[(size_t)src * dv + c] : (vh ? vh[(size_t)(3 + src) * dv + c] : 0.0);
                s += w[j * dv + c] * vv;
            }
            ht[c] = s;
            const double g = Phi_of(s) + s * phi_of(s);
            double r = vt[c] - s * Phi_of(s);
            for (int l = 0; l < R; ++l) {
                if (pg) {  /* non-linear variant: delta = GELU(p r), r <- r - delta */
                    const double zz = pg[((size_t)t * R + l) * dv + c] * r;
                    const double delta = zz * Phi_of(zz);
                    xt[(size_t)l * dv + c] = gamma[(size_t)t * R + l] * delta;
                    r -= delta;
                    continue;
                }
                xt[(size_t)l * dv + c] = gamma[(size_t)t * R + l] * g * r;
                if (l + 1 < R) r *= 1.0 - eta[(size_t)t * R + l] * g;
            }
        }
        memcpy(Sprev + (size_t)t * DD, S, sizeof(double) * DD);
        const double al = alpha[t], be = beta[t];
        for (int i = 0; i < dv; ++i) {
            double s = 0.0;
            for (int j = 0; j < dk; ++j) s += S[(size_t)i * dk + j] * kt[j];
            y[i] = s;
        }
        for (int i = 0; i < dv; ++i)
            for (int j = 0; j < dk; ++j) {
                double val = al * (S[(size_t)i * dk + j] - be * y[i] * kt[j]) + be * vt[i] * kt[j];
                for (int l = 0; l < R; ++l) val += xt[(size_t)l * dv + i] * u[((size_t)t * R + l) * dk + j];
                S[(size_t)i * dk + j] = val;
            }
    }
    /* S now holds S_T */

    if (a->dS_final) memcpy(dS, a->dS_final + bh * DD, sizeof(double) * DD);
    for (int t = T - 1; t >= 0; --t) {
        const double *vt = v + (size_t)t * dv, *kt = k + (size_t)t * dk, *qt = q + (size_t)t * dk;
        const double *dOt = dO + (size_t)t * dv, *P = Sprev + (size_t)t * DD;
        const double *St = t + 1 < T ? Sprev + (size_t)(t + 1) * DD : S;
        const double *xt = xs + (size_t)t * (R > 0 ? R : 1) * dv;
        const double al = alpha[t], be = beta[t];

        /* readout o_t = S_t q_t */
        for (int j = 0; j < dk; ++j) {
            double s = 0.0;
            for (int i = 0; i < dv; ++i) s += St[(size_t)i * dk + j] * dOt[i];
            dq[(size_t)t * dk + j] = s;
        }
        for (int i = 0; i < dv; ++i)
            for (int j = 0; j < dk; ++j) dS[(size_t)i * dk + j] += dOt[i] * qt[j];

        /* the update S_t = alpha (P - beta (P k) k^T) + beta v k^T + sum_l x_l u_l^T */
        double yz = 0.0, vz = 0.0, dSP = 0.0;
        for (int i = 0; i < dv; ++i) {
            double sy = 0.0, sz = 0.0;
            for (int j = 0; j < dk; ++j) {
                sy += P[(size_t)i * dk + j] * kt[j];
                sz += dS[(size_t)i * dk + j] * kt[j];
                dSP += dS[(size_t)i * dk + j] * P[(size_t)i * dk + j];
            }
            y[i] = sy;
            z[i] = sz;
            yz += sy * sz;
            vz += vt[i] * sz;
        }
        dbeta[t] = vz - al * yz;
        dalpha[t] = dSP - be * yz;
        for (int j = 0; j < dk; ++j) {
            double s = 0.0;
            for (int i = 0; i < dv; ++i)
                s += dS[(size_t)i * dk + j] * (be * vt[i] - al * be * y[i]) - al * be * P[(size_t)i * dk + j] * z[i];
            dkk[(size_t)t * dk + j] = s;
        }
        for (int i = 0; i < dv; ++i) dvv[(size_t)t * dv + i] += be * z[i];
        for (int l = 0; l < R; ++l) {
            const double *ul = u + ((size_t)t * R + l) * dk;
            for (int i = 0; i < dv; ++i) {
                double s = 0.0;
                for (int j = 0; j < dk; ++j) s += dS[(size_t)i * dk + j] * ul[j];
                dx[(size_t)l * dv + i] = s;
            }
            for (int j = 0; j < dk; ++j) {
                double s = 0.0;
                for (int i = 0; i < dv; ++i) s += dS[(size_t)i * dk + j] * xt[(size_t)l * dv + i];
                du[((size_t)t * R + l) * dk + j] = s;
            }
        }

        /* residual chain and anchor, channel by channel */
        for (int l = 0; l < R; ++l) {
            dgamma[(size_t)t * R + l] = 0.0;
            if (deta) deta[(size_t)t * R + l] = 0.0;
        }
        for (int c = 0; pg && c < dv; ++c) {  /* the non-linear chain */
            const double hc = hh[(size_t)t * dv + c];
            const double g = Phi_of(hc) + hc * phi_of(hc);
            double r = vt[c] - hc * Phi_of(hc);
            for (int l = 0; l < R; ++l) {
                rs[(size_t)l * dv + c] = r;
                const double zz = pg[((size_t)t * R + l) * dv + c] * r;
                r -= zz * Phi_of(zz);
            }
            double dr_next = 0.0;  /* nothing reads r_{t,R+1} */
            for (int l = R - 1; l >= 0; --l) {
                const double gm = gamma[(size_t)t * R + l], p = pg[((size_t)t * R + l) * dv + c];
                const double rl = rs[(size_t)l * dv + c], dxl = dx[(size_t)l * dv + c];
                const double zz = p * rl, delta = zz * Phi_of(zz);
                /* x_l = gamma delta_l and r_{l+1} = r_l - delta_l */
                const double ddelta = gm * dxl - dr_next;
                dgamma[(size_t)t * R + l] += delta * dxl;
                const double dz = ddelta * (Phi_of(zz) + zz * phi_of(zz));
                dpg[((size_t)t * R + l) * dv + c] = dz * rl;
                dr_next = dr_next + dz * p;
            }
            dvv[(size_t)t * dv + c] += dr_next;
            dh[(size_t)t * dv + c] = -g * dr_next;  /* e = v - GELU(h); the gain g is not used */
        }
        for (int c = 0; !pg && c < dv; ++c) {
            const double hc = hh[(size_t)t * dv + c];
            const double Ph = Phi_of(hc), ph = phi_of(hc);
            const double g = Ph + hc * ph;
            double r = vt[c] - hc * Ph;
            for (int l = 0; l < R; ++l) {  /* the chain's values r_{t,l} */
                rs[(size_t)l * dv + c] = r;
                if (l + 1 < R) r *= 1.0 - eta[(size_t)t * R + l] * g;
            }
            double dr_next = 0.0, dg = 0.0;
            for (int l = R - 1; l >= 0; --l) {
                /* the last level's gain shapes nothing (the cotangent of r_{t,R+1} is zero) */
                const double gm = gamma[(size_t)t * R + l], et = l + 1 < R ? eta[(size_t)t * R + l] : 0.0;
                const double rl = rs[(size_t)l * dv + c], dxl = dx[(size_t)l * dv + c];
                dgamma[(size_t)t * R + l] += g * rl * dxl;
                deta[(size_t)t * R + l] += -g * rl * dr_next;
                dg += gm * rl * dxl - et * rl * dr_next;
                dr_next = gm * g * dxl + (1.0 - et * g) * dr_next;
            }
            /* dr_next is now the cotangent of r_{t,1} = e_t */
            dvv[(size_t)t * dv + c] += dr_next;
            dh[(size_t)t * dv + c] = -g * dr_next + ph * (2.0 - hc * hc) * dg;
        }

        /* carry the state cotangent to S_{t-1} */
        for (int i = 0; i < dv; ++i)
            for (int j = 0; j < dk; ++j)
                dS[(size_t)i * dk + j] = al * (dS[(size_t)i * dk + j] - be * z[i] * kt[j]);
    }
    if (a->dS_init) memcpy(a->dS_init + bh * DD, dS, sizeof(double) * DD);

    /* the convolution: h_t = sum_j w_j (.) v_{t-j} */
    for (int t = 0; t < T; ++t)
        for (int j = 0; j < 4; ++j) {
            const int src = t - j;
            for (int c = 0; c < dv; ++c) {
                const double d = dh[(size_t)t * dv + c];
                if (src >= 0) {
                    dvv[(size_t)src * dv + c] += w[j * dv + c] * d;
                    dw[j * dv + c] += v[(size_t)src * dv + c] * d;
                } else {
                    if (a->dv_hist) a->dv_hist[(bh * 3 + (size_t)(3 + src)) * dv + c] += w[j * dv + c] * d;
                    if (vh) dw[j * dv + c] += vh[(size_t)(3 + src) * dv + c] * d;
                }
            }
        }
done:
    free(Sprev); free(S); free(dS); free(hh); free(xs); free(rs); free(dx); free(dh); free(y); free(z);
}

static void *worker(void *p)
{
    bwd_args *a = (bwd_args *)p;
    const int units = a->B * a->H;
    for (int idx = a->thread_id; idx < units; idx += a->nthreads) run_head(a, idx / a->H, idx % a->H);
    return NULL;
}

/* Returns 0 on success, a negative number for bad arguments or an allocation failure. */
int prism_oracle_backward_f64(int B, int H, int T, int dk, int dv, int L,
                              const double *q, const double *k, const double *v,
                              const double *beta, const double *alpha,
                              const double *u, const double *gamma, const double *eta,
                              const double *p_gain, const double *conv_w, const double *v_hist,
                              const double *S_init, const double *dout, const double *dS_final,
                              double *dq, double *dk_, double *dv_, double *dbeta, double *dalpha,
                              double *du, double *dgamma, double *deta, double *dp_gain, double *dconv_w,
                              double *dv_hist, double *dS_init, int nthreads)
{
    if (B < 0 || H < 0 || T < 1 || dk <= 0 || dv <= 0 || L < 1) return -1;
    if (!q || !k || !v || !beta || !alpha || !conv_w || !dout) return -2;
    if (!dq || !dk_ || !dv_ || !dbeta || !dalpha || !dconv_w) return -2;
    if (L > 1 && (!u || !gamma || !du || !dgamma)) return -3;
    if (L > 1 && (p_gain ? !dp_gain : (!eta || !deta))) return -3;
    const int units = B * H;
    if (units == 0) return 0;
    const size_t th = (size_t)units * T;
    memset(dv_, 0, sizeof(double) * th * dv);
    if (dv_hist) memset(dv_hist, 0, sizeof(double) * units * 3 * dv);
    /* per-(batch, head) sums of the convolution weight's cotangent, added over the batch below */
    double *part = calloc((size_t)units * 4 * dv, sizeof(double));
    if (!part) return -9;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > units) nthreads = units;
    bwd_args base = {B, H, T, dk, dv, L, q, k, v, beta, alpha, u, gamma, eta, p_gain, conv_w, v_hist, S_init,
                     dout, dS_final, dq, dk_, dv_, dbeta, dalpha, du, dgamma, deta, dp_gain, part, dv_hist,
                     dS_init, nthreads, 0, 0};
    pthread_t *th_ids = malloc(sizeof(pthread_t) * nthreads);
    bwd_args *args = malloc(sizeof(bwd_args) * nthreads);
    int status = 0;
    if (!th_ids || !args) {
        status = -9;
    } else {
        for (int i = 0; i < nthreads; ++i) {
            args[i] = base;
            args[i].thread_id = i;
            pthread_create(&th_ids[i], NULL, worker, &args[i]);
        }
        for (int i = 0; i < nthreads; ++i) {
            pthread_join(th_ids[i], NULL);
            if (args[i].status) status = args[i].status;
        }
    }
    memset(dconv_w, 0, sizeof(double) * H * 4 * dv);
    for (int b = 0; b < B; ++b)
        for (int h = 0; h < H; ++h)
            for (int n = 0; n < 4 * dv; ++n) dconv_w[(size_t)h * 4 * dv + n] += part[((size_t)b * H + h) * 4 * dv + n];
    free(part);
    free(th_ids);
    free(args);
    return status;
}
