// Portable fp32 path of the PRISM memory-recurrence forward (SIMT, no tensor cores).
//
// One kernel per step of the chunked evaluation, intermediates in the plan's
// workspace.  This path computes in fp32 throughout, so it is the one used for
// float32 io (where bf16 tensor-core operands could not meet a 1e-4 relative
// error), and it is a second, independently structured GPU evaluation that the
// tensor-core path is tested against.
//
// Chunked form (chunk of C = 64 tokens, local index i, j; lambda_i = sum_{m<=i}
// ln alpha_m inside the chunk, Gamma_i = exp(lambda_i), D_ij = exp(lambda_i - lambda_j)).
// Writing S_t = alpha_t S_{t-1} + vt_t k_t^T + sum_l x_{t,l} u_{t,l}^T with
// vt_t = beta_t v_t - alpha_t beta_t S_{t-1} k_t (the GDN transition of the
// notes on PRISM, section 2.2, expanded) and unrolling over the chunk gives
//   (I + A) V~ = diag(beta) V - M X - diag(beta Gamma) K S0^T,
//   A_ij = beta_i D_ij k_i.k_j (j < i),  M_{i,(j,l)} = beta_i D_ij k_i.u_{j,l} (j < i),
// so V~ = U' - W S0^T with T = (I + A)^{-1}, W = T diag(beta Gamma) K and
// U' = T (diag(beta) V - M X).  Then
//   S_C = Gamma_C S0 + V~^T diag(Gamma_C / Gamma) K + sum_l X_l^T diag(Gamma_C / Gamma) U_l,
//   O   = diag(Gamma) Q S0^T + (Q K^T o D) V~ + sum_l (Q U_l^T o D) X_l   (D incl. diagonal).
#include "prism_internal.h"

namespace prism {
namespace simt {

constexpr int C = kChunk;
constexpr int NT = 256;   // threads per block
constexpr int VB = 16;    // value rows of the state per state-passing block

__device__ __forceinline__ float ldf(const float *p) { return *p; }
__device__ __forceinline__ float ldf(const __nv_bfloat16 *p) { return __bfloat162float(*p); }
__device__ __forceinline__ void stf(float *p, float x) { *p = x; }
__device__ __forceinline__ void stf(__nv_bfloat16 *p, float x) { *p = __float2bfloat16_rn(x); }

// ---------------------------------------------------------------------------------------------
// Step a1: anchor, gain, residual and the closed-form residual chain -> X [BH][T][R][dv].
// v_hist [BH][3][dv] (v_{-3}, v_{-2}, v_{-1}) supplies the window before the first token; null
// means zeros.  With p_gain [BH][T][R][dv] the chain is the non-linear residual variant of the
// notes on PRISM (section 2.3): delta_l = GELU(p_l r_l), x_l = gamma_l delta_l,
// r_{l+1} = r_l - delta_l (eta is not read).
template <typename io_t>
__global__ void __launch_bounds__(NT) prep_kernel(const io_t *__restrict__ v, const io_t *__restrict__ v_hist,
                                                  const io_t *__restrict__ conv_w,
                                                  const io_t *__restrict__ p_gain,
                                                  const float *__restrict__ gamma,
                                                  const float *__restrict__ eta, float *__restrict__ X,
                                                  int H, int T, int dv, int R)
{
    const int bh = blockIdx.y;
    const int h = bh % H;
    const long long idx = (long long)blockIdx.x * NT + threadIdx.x;
    if (idx >= (long long)T * dv) return;
    const int t = (int)(idx / dv), c = (int)(idx % dv);
    const io_t *vb = v + (size_t)bh * T * dv;
    float a = 0.f;
#pragma unroll
    for (int j = 0; j < 4; ++j)
        if (t - j >= 0)
            a = fmaf(ldf(conv_w + ((size_t)h * 4 + j) * dv + c), ldf(vb + (size_t)(t - j) * dv + c), a);
        else if (v_hist)
            a = fmaf(ldf(conv_w + ((size_t)h * 4 + j) * dv + c), ldf(v_hist + ((size_t)bh * 3 + 3 + t - j) * dv + c), a);
    const float Phi = 0.5f * erfcf(-a * 0.70710678118654752f);
    const float phi = 0.39894228040143268f * expf(-0.5f * a * a);
    const float g = fmaf(a, phi, Phi);
    float r = ldf(vb + (size_t)t * dv + c) - a * Phi;
    const float *gm = gamma + ((size_t)bh * T + t) * R;
    const float *et = eta + ((size_t)bh * T + t) * R;
    float *xo = X + ((size_t)bh * T + t) * R * dv + c;
    if (p_gain) {
        const io_t *pg = p_gain + ((size_t)bh * T + t) * R * dv + c;
        for (int l = 0; l < R; ++l) {
            const float z = ldf(pg + (size_t)l * dv) * r;
            const float d = z * (0.5f * erfcf(-z * 0.70710678118654752f));
            xo[(size_t)l * dv] = gm[l] * d;
            r -= d;
        }
        return;
    }
    for (int l = 0; l < R; ++l) {
        xo[(size_t)l * dv] = gm[l] * g * r;
        if (l + 1 < R) r *= (1.f - et[l] * g);
    }
}

// ---------------------------------------------------------------------------------------------
// Steps a2-a4: chunk-local log-decay cumsum, Gram A and T = (I + A)^{-1}.
template <typename io_t>
__global__ void __launch_bounds__(NT) chunk_solve_kernel(const io_t *__restrict__ k, const float *__restrict__ beta,
                                                         const float *__restrict__ alpha,
                                                         float *__restrict__ lam_ws, float *__restrict__ T_ws,
                                                         int T, int dk, int NC)
{
    extern __shared__ float smem[];
    const int c = blockIdx.x, bh = blockIdx.y, tid = threadIdx.x;
    const int t0 = c * C;
    const int n = min(C, T - t0);
    const int ldk = dk + 1, ldc = C + 1;
    float *Ks = smem;            // C x ldk
    float *As = Ks + C * ldk;    // C x ldc
    float *Ts = As + C * ldc;    // C x ldc
    float *lam = Ts + C * ldc;   // C
    float *bet = lam + C;        // C

    const io_t *kb = k + ((size_t)bh * T + t0) * dk;
    for (int e = tid; e < C * dk; e += NT) {
        const int i = e / dk, m = e % dk;
        Ks[i * ldk + m] = (i < n) ? ldf(kb + (size_t)i * dk + m) : 0.f;
    }
    if (tid < C) {
        bet[tid] = (tid < n) ? beta[(size_t)bh * T + t0 + tid] : 0.f;
        lam[tid] = (tid < n) ? logf(alpha[(size_t)bh * T + t0 + tid]) : 0.f;
    }
    __syncthreads();
    if (tid < 32) {  // inclusive scan of the 64 log-decays by one warp (two values per lane)
        float a0 = lam[2 * tid], a1 = lam[2 * tid + 1];
        float s = a0 + a1;
        for (int off = 1; off < 32; off <<= 1) {
            const float y = __shfl_up_sync(0xffffffffu, s, off);
            if (tid >= off) s += y;
        }
        lam[2 * tid + 1] = s;
        lam[2 * tid] = s - a1;
    }
    __syncthreads();
    if (tid < n) lam_ws[(size_t)bh * T + t0 + tid] = lam[tid];
    for (int e = tid; e < C * C; e += NT) {
        const int i = e / C, j = e % C;
        float a = 0.f;
        if (j < i) {
            float d = 0.f;
            for (int m = 0; m < dk; ++m) d = fmaf(Ks[i * ldk + m], Ks[j * ldk + m], d);
            a = bet[i] * expf(lam[i] - lam[j]) * d;
        }
        As[i * ldc + j] = a;
    }
    __syncthreads();
    if (tid < C) {  // column-parallel forward substitution: (I + A) T = I
        const int col = tid;
        for (int i = 0; i < C; ++i) {
            float x = (i == col) ? 1.f : 0.f;
            if (i > col) {
                float s = 0.f;
                for (int j = col; j < i; ++j) s = fmaf(As[i * ldc + j], Ts[j * ldc + col], s);
                x = -s;
            }
            Ts[i * ldc + col] = x;
        }
    }
    __syncthreads();
    float *Tout = T_ws + ((size_t)bh * NC + c) * C * C;
    for (int e = tid; e < C * C; e += NT) Tout[e] = Ts[(e / C) * ldc + (e % C)];
}

// ---------------------------------------------------------------------------------------------
// Step a5: W = T diag(beta Gamma) K and U' = T (diag(beta) V - M X).
template <typename io_t>
__global__ void __launch_bounds__(NT) wy_kernel(const io_t *__restrict__ k, const io_t *__restrict__ v,
                                                const float *__restrict__ beta, const io_t *__restrict__ u,
                                                const float *__restrict__ X, const float *__restrict__ lam_ws,
                                                const float *__restrict__ T_ws, float *__restrict__ W_ws,
                                                float *__restrict__ Up_ws, int T, int dk, int dv, int R, int NC)
{
    extern __shared__ float smem[];
    const int c = blockIdx.x, bh = blockIdx.y, tid = threadIdx.x;
    const int t0 = c * C;
    const int n = min(C, T - t0);
    const int ldk = dk + 1, ldv = dv + 1, ldc = C + 1;
    float *Ts = smem;           // C x ldc
    float *Ks = Ts + C * ldc;   // C x ldk
    float *Us = Ks + C * ldk;   // C x ldk
    float *Xs = Us + C * ldk;   // C x ldv
    float *G = Xs + C * ldv;    // C x ldc
    float *lam = G + C * ldc;   // C
    float *bet = lam + C;       // C

    const float *Tin = T_ws + ((size_t)bh * NC + c) * C * C;
    for (int e = tid; e < C * C; e += NT) Ts[(e / C) * ldc + (e % C)] = Tin[e];
    const io_t *kb = k + ((size_t)bh * T + t0) * dk;
    for (int e = tid; e < C * dk; e += NT) {
        const int i = e / dk, m = e % dk;
        Ks[i * ldk + m] = (i < n) ? ldf(kb + (size_t)i * dk + m) : 0.f;
    }
    if (tid < C) {
        bet[tid] = (tid < n) ? beta[(size_t)bh * T + t0 + tid] : 0.f;
        lam[tid] = (tid < n) ? lam_ws[(size_t)bh * T + t0 + tid] : 0.f;
    }
    __syncthreads();

    const int i = tid >> 2, cq = tid & 3;
    const int nv = dv >> 2;  // <= 32 value columns per thread
    float acc[32];
    const io_t *vb = v + ((size_t)bh * T + t0) * dv;
#pragma unroll
    for (int m = 0; m < 32; ++m)
        if (m < nv) acc[m] = (i < n) ? bet[i] * ldf(vb + (size_t)i * dv + cq + 4 * m) : 0.f;

    for (int l = 0; l < R; ++l) {
        __syncthreads();
        for (int e = tid; e < C * dk; e += NT) {
            const int ii = e / dk, m = e % dk;
            Us[ii * ldk + m] = (ii < n) ? ldf(u + (((size_t)bh * T + t0 + ii) * R + l) * dk + m) : 0.f;
        }
        for (int e = tid; e < C * dv; e += NT) {
            const int ii = e / dv, m = e % dv;
            Xs[ii * ldv + m] = (ii < n) ? X[(((size_t)bh * T + t0 + ii) * R + l) * dv + m] : 0.f;
        }
        __syncthreads();
        for (int e = tid; e < C * C; e += NT) {
            const int ii = e / C, j = e % C;
            float gval = 0.f;
            if (j < ii) {
                float d = 0.f;
                for (int m = 0; m < dk; ++m) d = fmaf(Ks[ii * ldk + m], Us[j * ldk + m], d);
                gval = bet[ii] * expf(lam[ii] - lam[j]) * d;
            }
            G[ii * ldc + j] = gval;
        }
        __syncthreads();
        for (int j = 0; j < i; ++j) {
            const float gij = G[i * ldc + j];
#pragma unroll
            for (int m = 0; m < 32; ++m)
                if (m < nv) acc[m] = fmaf(-gij, Xs[j * ldv + cq + 4 * m], acc[m]);
        }
    }
    __syncthreads();
    // U' = T * RHS (RHS parked in Xs)
#pragma unroll
    for (int m = 0; m < 32; ++m)
        if (m < nv) Xs[i * ldv + cq + 4 * m] = acc[m];
    __syncthreads();
#pragma unroll
    for (int m = 0; m < 32; ++m)
        if (m < nv) acc[m] = 0.f;
    for (int j = 0; j <= i; ++j) {
        const float tij = Ts[i * ldc + j];
#pragma unroll
        for (int m = 0; m < 32; ++m)
            if (m < nv) acc[m] = fmaf(tij, Xs[j * ldv + cq + 4 * m], acc[m]);
    }
    float *up = Up_ws + ((size_t)bh * NC * C + t0 + i) * dv;
#pragma unroll
    for (int m = 0; m < 32; ++m)
        if (m < nv) up[cq + 4 * m] = acc[m];
    // W = T * diag(beta Gamma) K
    for (int e = tid; e < C * dk; e += NT) {
        const int ii = e / dk, m = e % dk;
        Ks[ii * ldk + m] *= bet[ii] * expf(lam[ii]);
    }
    __syncthreads();
    const int nk = dk >> 2;
#pragma unroll
    for (int m = 0; m < 32; ++m)
        if (m < nk) acc[m] = 0.f;
    for (int j = 0; j <= i; ++j) {
        const float tij = Ts[i * ldc + j];
#pragma unroll
        for (int m = 0; m < 32; ++m)
            if (m < nk) acc[m] = fmaf(tij, Ks[j * ldk + cq + 4 * m], acc[m]);
    }
    float *wo = W_ws + ((size_t)bh * NC * C + t0 + i) * dk;
#pragma unroll
    for (int m = 0; m < 32; ++m)
        if (m < nk) wo[cq + 4 * m] = acc[m];
}

// ---------------------------------------------------------------------------------------------
// Step a6: inter-chunk state passing, sequential over chunks, VB value rows per block, from
// S_init (or 0); S_final, if given, receives the state after the last token.  Each block reads
// and writes only its own rows, so S_final may be S_init.
template <typename io_t>
__global__ void __launch_bounds__(NT) state_kernel(const io_t *__restrict__ k, const io_t *__restrict__ u,
                                                   const float *__restrict__ X, const float *__restrict__ lam_ws,
                                                   const float *__restrict__ W_ws, const float *__restrict__ Up_ws,
                                                   float *__restrict__ S0_ws, float *__restrict__ Vt_ws,
                                                   const float *S_init, float *S_final,
                                                   int T, int dk, int dv, int R, int NC)
{
    extern __shared__ float smem[];
    const int bh = blockIdx.x, r0 = blockIdx.y * VB, tid = threadIdx.x;
    const int ldk = dk + 1, ldb = VB + 1;
    float *S = smem;            // VB x ldk
    float *Ws = S + VB * ldk;   // C x ldk
    float *Ks = Ws + C * ldk;   // C x ldk
    float *Vs = Ks + C * ldk;   // C x ldb
    float *lam = Vs + C * ldb;  // C

    for (int e = tid; e < VB * dk; e += NT) {
        const int r = e / dk, m = e % dk;
        S[r * ldk + m] = S_init ? S_init[((size_t)bh * dv + r0 + r) * dk + m] : 0.f;
    }
    for (int c = 0; c < NC; ++c) {
        const int t0 = c * C;
        const int n = min(C, T - t0);
        __syncthreads();
        const float *wb = W_ws + ((size_t)bh * NC * C + t0) * dk;
        const io_t *kb = k + ((size_t)bh * T + t0) * dk;
        for (int e = tid; e < C * dk; e += NT) {
            const int i = e / dk, m = e % dk;
            Ws[i * ldk + m] = wb[(size_t)i * dk + m];
            Ks[i * ldk + m] = (i < n) ? ldf(kb + (size_t)i * dk + m) : 0.f;
        }
        if (tid < C) lam[tid] = lam_ws[(size_t)bh * T + t0 + min(tid, n - 1)];
        float *s0 = S0_ws + ((size_t)bh * NC + c) * dv * dk;
        for (int e = tid; e < VB * dk; e += NT) {
            const int r = e / dk, m = e % dk;
            s0[(size_t)(r0 + r) * dk + m] = S[r * ldk + m];
        }
        __syncthreads();
        const float lam_last = lam[C - 1];
        // V~ = U' - W S0^T, and its decayed copy for the state update
        for (int e = tid; e < C * VB; e += NT) {
            const int i = e / VB, r = e % VB;
            float d = 0.f;
            for (int m = 0; m < dk; ++m) d = fmaf(Ws[i * ldk + m], S[r * ldk + m], d);
            const float vt = Up_ws[((size_t)bh * NC * C + t0 + i) * dv + r0 + r] - d;
            Vt_ws[((size_t)bh * NC * C + t0 + i) * dv + r0 + r] = vt;
            Vs[i * ldb + r] = (i < n) ? vt * expf(lam_last - lam[i]) : 0.f;
        }
        __syncthreads();
        const float gC = expf(lam_last);
        for (int e = tid; e < VB * dk; e += NT) {
            const int r = e / dk, m = e % dk;
            float s = gC * S[r * ldk + m];
            for (int i = 0; i < C; ++i) s = fmaf(Vs[i * ldb + r], Ks[i * ldk + m], s);
            S[r * ldk + m] = s;
        }
        for (int l = 0; l < R; ++l) {
            __syncthreads();
            for (int e = tid; e < C * dk; e += NT) {
                const int i = e / dk, m = e % dk;
                Ks[i * ldk + m] = (i < n) ? ldf(u + (((size_t)bh * T + t0 + i) * R + l) * dk + m) : 0.f;
            }
            for (int e = tid; e < C * VB; e += NT) {
                const int i = e / VB, r = e % VB;
                Vs[i * ldb + r] = (i < n) ? X[(((size_t)bh * T + t0 + i) * R + l) * dv + r0 + r] * expf(lam_last - lam[i])
                                          : 0.f;
            }
            __syncthreads();
            for (int e = tid; e < VB * dk; e += NT) {
                const int r = e / dk, m = e % dk;
                float s = S[r * ldk + m];
                for (int i = 0; i < C; ++i) s = fmaf(Vs[i * ldb + r], Ks[i * ldk + m], s);
                S[r * ldk + m] = s;
            }
        }
    }
    if (S_final) {
        __syncthreads();
        for (int e = tid; e < VB * dk; e += NT) {
            const int r = e / dk, m = e % dk;
            S_final[((size_t)bh * dv + r0 + r) * dk + m] = S[r * ldk + m];
        }
    }
}

// ---------------------------------------------------------------------------------------------
// Step a7: O = diag(Gamma) Q S0^T + (Q K^T o D) V~ + sum_l (Q U_l^T o D) X_l.
template <typename io_t, typename out_t>
__global__ void __launch_bounds__(NT) out_kernel(const io_t *__restrict__ q, const io_t *__restrict__ k,
                                                 const io_t *__restrict__ u, const float *__restrict__ X,
                                                 const float *__restrict__ lam_ws, const float *__restrict__ S0_ws,
                                                 const float *__restrict__ Vt_ws, out_t *__restrict__ out,
                                                 int T, int dk, int dv, int R, int NC)
{
    extern __shared__ float smem[];
    const int c = blockIdx.x, bh = blockIdx.y, tid = threadIdx.x;
    const int t0 = c * C;
    const int n = min(C, T - t0);
    const int ldk = dk + 1, ldv = dv + 1, ldc = C + 1;
    float *Qs = smem;           // C x ldk
    float *Bs = Qs + C * ldk;   // C x ldk
    float *G = Bs + C * ldk;    // C x ldc
    float *Ms = G + C * ldc;    // max(dv x ldk, C x ldv)
    float *lam = Ms + (size_t)max(dv * ldk, C * ldv);

    const io_t *qb = q + ((size_t)bh * T + t0) * dk;
    for (int e = tid; e < C * dk; e += NT) {
        const int i = e / dk, m = e % dk;
        Qs[i * ldk + m] = (i < n) ? ldf(qb + (size_t)i * dk + m) : 0.f;
    }
    const float *s0 = S0_ws + ((size_t)bh * NC + c) * dv * dk;
    for (int e = tid; e < dv * dk; e += NT) Ms[(e / dk) * ldk + (e % dk)] = s0[e];
    if (tid < C) lam[tid] = lam_ws[(size_t)bh * T + t0 + min(tid, n - 1)];
    __syncthreads();

    const int i = tid >> 2, cq = tid & 3;
    const int nv = dv >> 2;
    float acc[32];
    const float gi = expf(lam[i]);
#pragma unroll
    for (int m = 0; m < 32; ++m) {
        if (m < nv) {
            const int cc = cq + 4 * m;
            float d = 0.f;
            for (int p = 0; p < dk; ++p) d = fmaf(Qs[i * ldk + p], Ms[cc * ldk + p], d);
            acc[m] = gi * d;
        }
    }
    for (int l = -1; l < R; ++l) {  // l = -1: keys with V~, then each level with its X
        __syncthreads();
        for (int e = tid; e < C * dk; e += NT) {
            const int ii = e / dk, m = e % dk;
            float x = 0.f;
            if (ii < n)
                x = (l < 0) ? ldf(k + ((size_t)bh * T + t0 + ii) * dk + m)
                            : ldf(u + (((size_t)bh * T + t0 + ii) * R + l) * dk + m);
            Bs[ii * ldk + m] = x;
        }
        for (int e = tid; e < C * dv; e += NT) {
            const int ii = e / dv, m = e % dv;
            float x = 0.f;
            if (ii < n)
                x = (l < 0) ? Vt_ws[((size_t)bh * NC * C + t0 + ii) * dv + m]
                            : X[(((size_t)bh * T + t0 + ii) * R + l) * dv + m];
            Ms[ii * ldv + m] = x;
        }
        __syncthreads();
        for (int e = tid; e < C * C; e += NT) {
            const int ii = e / C, j = e % C;
            float gval = 0.f;
            if (j <= ii) {
                float d = 0.f;
                for (int m = 0; m < dk; ++m) d = fmaf(Qs[ii * ldk + m], Bs[j * ldk + m], d);
                gval = expf(lam[ii] - lam[j]) * d;
            }
            G[ii * ldc + j] = gval;
        }
        __syncthreads();
        for (int j = 0; j <= i; ++j) {
            const float gij = G[i * ldc + j];
#pragma unroll
            for (int m = 0; m < 32; ++m)
                if (m < nv) acc[m] = fmaf(gij, Ms[j * ldv + cq + 4 * m], acc[m]);
        }
    }
    if (i < n) {
        out_t *o = out + ((size_t)bh * T + t0 + i) * dv;
#pragma unroll
        for (int m = 0; m < 32; ++m)
            if (m < nv) stf(o + cq + 4 * m, acc[m]);
    }
}

// ---------------------------------------------------------------------------------------------
struct Smem {
    size_t solve, wy, state, out;
};

static Smem smem_bytes(int dk, int dv)
{
    const size_t ldk = dk + 1, ldv = dv + 1, ldc = C + 1;
    Smem s;
    s.solve = sizeof(float) * (C * ldk + 2 * C * ldc + 2 * C);
    s.wy = sizeof(float) * (C * ldc + 2 * C * ldk + C * ldv + C * ldc + 2 * C);
    s.state = sizeof(float) * (VB * ldk + 2 * C * ldk + C * (VB + 1) + C);
    s.out = sizeof(float) * (2 * C * ldk + C * ldc + (dv * ldk > C * ldv ? dv * ldk : C * ldv) + C);
    return s;
}

template <typename io_t>
static cudaError_t prepare_t(int dk, int dv)
{
    const Smem s = smem_bytes(dk, dv);
    cudaError_t e;
    if ((e = cudaFuncSetAttribute(chunk_solve_kernel<io_t>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)s.solve))) return e;
    if ((e = cudaFuncSetAttribute(wy_kernel<io_t>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)s.wy))) return e;
    if ((e = cudaFuncSetAttribute(state_kernel<io_t>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)s.state))) return e;
    if ((e = cudaFuncSetAttribute(out_kernel<io_t, float>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)s.out))) return e;
    if ((e = cudaFuncSetAttribute(out_kernel<io_t, __nv_bfloat16>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)s.out)))
        return e;
    return cudaSuccess;
}

template <typename io_t, typename out_t>
static cudaError_t forward_t(const Shape &s, const ForwardArgs &a, const SimtWorkspace &w, KernelTimer &tm)
{
    cudaStream_t st = tm.stream;
    const Smem sm = smem_bytes(s.dk, s.dv);
    const io_t *q = (const io_t *)a.q, *k = (const io_t *)a.k, *v = (const io_t *)a.v;
    const io_t *u = (const io_t *)a.u, *cw = (const io_t *)a.conv_w;
    out_t *out = (out_t *)a.out;
    if (s.R > 0) {
        const long long elems = (long long)s.T * s.dv;
        dim3 grid((unsigned)((elems + NT - 1) / NT), s.BH);
        tm.begin("simt_prep");
        prep_kernel<io_t><<<grid, NT, 0, st>>>(v, (const io_t *)a.v_hist, cw, (const io_t *)a.p_gain, a.gamma, a.eta,
                                               w.X, s.H, s.T, s.dv, s.R);
        tm.end();
    }
    tm.begin("simt_chunk_solve");
    chunk_solve_kernel<io_t><<<dim3(s.NC, s.BH), NT, sm.solve, st>>>(k, a.beta, a.alpha, w.lam, w.Tm, s.T, s.dk, s.NC);
    tm.end();
    tm.begin("simt_wy");
    wy_kernel<io_t><<<dim3(s.NC, s.BH), NT, sm.wy, st>>>(k, v, a.beta, u, w.X, w.lam, w.Tm, w.W, w.Up, s.T, s.dk,
                                                         s.dv, s.R, s.NC);
    tm.end();
    tm.begin("simt_state");
    state_kernel<io_t><<<dim3(s.BH, s.dv / VB), NT, sm.state, st>>>(k, u, w.X, w.lam, w.W, w.Up, w.S0, w.Vt,
                                                                    a.S_init, a.S_final, s.T, s.dk, s.dv, s.R,
                                                                    s.NC);
    tm.end();
    tm.begin("simt_out");
    out_kernel<io_t, out_t><<<dim3(s.NC, s.BH), NT, sm.out, st>>>(q, k, u, w.X, w.lam, w.S0, w.Vt, out, s.T, s.dk, s.dv,
                                                           s.R, s.NC);
    tm.end();
    return cudaGetLastError();
}

}  // namespace simt

size_t simt_workspace_bytes(const Shape &s)
{
    const size_t BH = s.BH, T = s.T, NCC = (size_t)s.NC * kChunk;
    size_t f = 0;
    f += BH * T * (size_t)s.R * s.dv;               // X
    f += BH * T;                                    // lam
    f += BH * (size_t)s.NC * kChunk * kChunk;       // Tm
    f += BH * NCC * s.dk;                           // W
    f += BH * NCC * s.dv;                           // Up
    f += BH * (size_t)s.NC * s.dv * s.dk;           // S0
    f += BH * NCC * s.dv;                           // Vt
    return f * sizeof(float) + 6 * 256;             // alignment slack
}

void simt_carve(const Shape &s, void *base, SimtWorkspace *w)
{
    const size_t BH = s.BH, T = s.T, NCC = (size_t)s.NC * kChunk;
    uintptr_t p = (uintptr_t)base;
    auto take = [&](size_t nfloat) {
        p = (p + 255) & ~(uintptr_t)255;
        float *r = (float *)p;
        p += nfloat * sizeof(float);
        return r;
    };
    w->X = take(BH * T * (size_t)s.R * s.dv);
    w->lam = take(BH * T);
    w->Tm = take(BH * (size_t)s.NC * kChunk * kChunk);
    w->W = take(BH * NCC * s.dk);
    w->Up = take(BH * NCC * s.dv);
    w->S0 = take(BH * (size_t)s.NC * s.dv * s.dk);
    w->Vt = take(BH * NCC * s.dv);
}

cudaError_t simt_prepare(const Shape &s, prism_dtype io)
{
    return io == PRISM_BF16 ? simt::prepare_t<__nv_bfloat16>(s.dk, s.dv) : simt::prepare_t<float>(s.dk, s.dv);
}

cudaError_t simt_forward(const Shape &s, prism_dtype io, prism_dtype out, const ForwardArgs &a, const SimtWorkspace &w,
                         int *d_status, KernelTimer &timer)
{
    (void)d_status;
    cudaError_t e;
    if (io == PRISM_BF16)
        e = out == PRISM_F32 ? simt::forward_t<__nv_bfloat16, float>(s, a, w, timer)
                             : simt::forward_t<__nv_bfloat16, __nv_bfloat16>(s, a, w, timer);
    else
        e = out == PRISM_F32 ? simt::forward_t<float, float>(s, a, w, timer)
                             : simt::forward_t<float, __nv_bfloat16>(s, a, w, timer);
    if (e == cudaSuccess && a.v_hist_out) e = launch_history(s, io, a.v_hist, a.v, a.v_hist_out, timer);
    return e;
}

}  // namespace prism
