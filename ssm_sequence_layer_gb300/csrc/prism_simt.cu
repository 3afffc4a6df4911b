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
//
// Register-tiled like the output kernel (helpers below): thread (ti, tc) owns rows 4 ti .. 4 ti + 3
// and the float4 column groups 4 tc + 64 g of each product.  The strictly lower scores
// M_l = beta_i D_ij (K U_l^T)_ij come in causal 4 x 4 tiles, parked transposed over U_l; T is
// kept transposed, so every sweep reads one float4 of a transposed factor per token.
__device__ __forceinline__ float4 ld4(const float *p) { return *reinterpret_cast<const float4 *>(p); }
__device__ __forceinline__ float4 ld4(const __nv_bfloat16 *p)
{
    const uint2 w = *reinterpret_cast<const uint2 *>(p);
    const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&w.x));
    const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&w.y));
    return make_float4(a.x, a.y, b.x, b.y);
}
__device__ __forceinline__ float dot4(const float4 a, const float4 b, float acc)
{
    return fmaf(a.x, b.x, fmaf(a.y, b.y, fmaf(a.z, b.z, fmaf(a.w, b.w, acc))));
}
// acc[a][g] += sgn * sum_{j < jend} At[j][4 ti + a] * Bm[j][4 tc + 64 g]   (At, Bm in shared memory)
template <int NG>
__device__ __forceinline__ void sweep_rows(float4 (&acc)[4][NG], const float *At, int lda, const float *Bm, int ldb,
                                           int ti, int tc, int jend, float sgn)
{
#pragma unroll 4
    for (int j = 0; j < jend; ++j) {
        const float4 av = ld4(At + j * lda + 4 * ti);
        const float aa[4] = {sgn * av.x, sgn * av.y, sgn * av.z, sgn * av.w};
#pragma unroll
        for (int g = 0; g < NG; ++g) {
            const float4 bv = ld4(Bm + j * ldb + 4 * tc + 64 * g);
#pragma unroll
            for (int a = 0; a < 4; ++a) {
                acc[a][g].x = fmaf(aa[a], bv.x, acc[a][g].x);
                acc[a][g].y = fmaf(aa[a], bv.y, acc[a][g].y);
                acc[a][g].z = fmaf(aa[a], bv.z, acc[a][g].z);
                acc[a][g].w = fmaf(aa[a], bv.w, acc[a][g].w);
            }
        }
    }
}
// the 4 x 4 tile (rows gi0.., columns gj0..) of P Q^T over DK (P, Q rows in shared memory)
template <int DK>
__device__ __forceinline__ void score_tile(float (&gt)[4][4], const float *P, const float *Qm, int ld, int gi0, int gj0)
{
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int b = 0; b < 4; ++b) gt[a][b] = 0.f;
#pragma unroll 2
    for (int m = 0; m < DK; m += 4) {
        float4 pv[4], qv[4];
#pragma unroll
        for (int a = 0; a < 4; ++a) pv[a] = ld4(P + (gi0 + a) * ld + m);
#pragma unroll
        for (int b = 0; b < 4; ++b) qv[b] = ld4(Qm + (gj0 + b) * ld + m);
#pragma unroll
        for (int a = 0; a < 4; ++a)
#pragma unroll
            for (int b = 0; b < 4; ++b) gt[a][b] = dot4(pv[a], qv[b], gt[a][b]);
    }
}

template <int DK, int DV>
struct WyTile {
    static constexpr int LDK = DK + 4, LDV = DV + 4, LDG = C + 4;
    static constexpr int UG = (C * LDK > C * LDG ? C * LDK : C * LDG);  // U_l, then M_l^T over it
    static constexpr size_t SMEM = sizeof(float) * (C * LDG + C * LDK + UG + C * LDV + 2 * C);
};

template <typename io_t, int DK, int DV>
__global__ void __launch_bounds__(NT) wy_kernel(const io_t *__restrict__ k, const io_t *__restrict__ v,
                                                const float *__restrict__ beta, const io_t *__restrict__ u,
                                                const float *__restrict__ X, const float *__restrict__ lam_ws,
                                                const float *__restrict__ T_ws, float *__restrict__ W_ws,
                                                float *__restrict__ Up_ws, int T, int R, int NC)
{
    using TL = WyTile<DK, DV>;
    constexpr int LDK = TL::LDK, LDV = TL::LDV, LDG = TL::LDG, NGV = DV / 64, NGK = DK / 64;
    extern __shared__ __align__(16) float smem[];
    float *Tt = smem;               // C x LDG   T transposed: Tt[j][i] = T[i][j]
    float *Ks = Tt + C * LDG;       // C x LDK   K, later diag(beta Gamma) K
    float *Us = Ks + C * LDK;       // C x LDK   U_l, then M_l^T (C x LDG)
    float *Xs = Us + TL::UG;        // C x LDV   X_l, then the right-hand side
    float *lam = Xs + C * LDV;      // C
    float *bet = lam + C;           // C
    const int c = blockIdx.x, bh = blockIdx.y, tid = threadIdx.x;
    const int t0 = c * C;
    const int n = min(C, T - t0);
    const int ti = tid >> 4, tc = tid & 15;
    const int gi0 = 4 * ti, gj0 = 4 * tc;

    const float *Tin = T_ws + ((size_t)bh * NC + c) * C * C;
    for (int e = tid; e < C * C; e += NT) Tt[(e % C) * LDG + e / C] = Tin[e];
    const io_t *kb = k + ((size_t)bh * T + t0) * DK;
    for (int e = tid; e < C * (DK / 4); e += NT) {
        const int i = e / (DK / 4), m4 = e % (DK / 4);
        const float4 x = (i < n) ? ld4(kb + (size_t)i * DK + 4 * m4) : make_float4(0.f, 0.f, 0.f, 0.f);
        *reinterpret_cast<float4 *>(Ks + i * LDK + 4 * m4) = x;
    }
    if (tid < C) {
        bet[tid] = (tid < n) ? beta[(size_t)bh * T + t0 + tid] : 0.f;
        lam[tid] = (tid < n) ? lam_ws[(size_t)bh * T + t0 + tid] : 0.f;
    }
    __syncthreads();

    // right-hand side diag(beta) V - sum_l M_l X_l, rows 4 ti + a, columns 4 tc + 64 g
    float4 acc[4][NGV];
    const io_t *vb = v + ((size_t)bh * T + t0) * DV;
#pragma unroll
    for (int a = 0; a < 4; ++a) {
        const int i = 4 * ti + a;
#pragma unroll
        for (int g = 0; g < NGV; ++g) {
            float4 x = (i < n) ? ld4(vb + (size_t)i * DV + 4 * tc + 64 * g) : make_float4(0.f, 0.f, 0.f, 0.f);
            x.x *= bet[i];
            x.y *= bet[i];
            x.z *= bet[i];
            x.w *= bet[i];
            acc[a][g] = x;
        }
    }
    for (int l = 0; l < R; ++l) {
        __syncthreads();  // the previous level's M^T and X are no longer read
        for (int e = tid; e < C * (DK / 4); e += NT) {
            const int i = e / (DK / 4), m4 = e % (DK / 4);
            const float4 x = (i < n) ? ld4(u + (((size_t)bh * T + t0 + i) * R + l) * DK + 4 * m4)
                                     : make_float4(0.f, 0.f, 0.f, 0.f);
            *reinterpret_cast<float4 *>(Us + i * LDK + 4 * m4) = x;
        }
        for (int e = tid; e < C * (DV / 4); e += NT) {
            const int i = e / (DV / 4), m4 = e % (DV / 4);
            const float4 x = (i < n) ? ld4(X + (((size_t)bh * T + t0 + i) * R + l) * DV + 4 * m4)
                                     : make_float4(0.f, 0.f, 0.f, 0.f);
            *reinterpret_cast<float4 *>(Xs + i * LDV + 4 * m4) = x;
        }
        __syncthreads();
        float gt[4][4];
        const bool live = gj0 < gi0 + 3;  // the tile holds some j < i
        if (live) {
            score_tile<DK>(gt, Ks, Us, LDK, gi0, gj0);
#pragma unroll
            for (int a = 0; a < 4; ++a)
#pragma unroll
                for (int b = 0; b < 4; ++b) {
                    const int i = gi0 + a, j = gj0 + b;
                    gt[a][b] = (j < i) ? bet[i] * expf(lam[i] - lam[j]) * gt[a][b] : 0.f;
                }
        }
        __syncthreads();  // U_l is no longer read: M_l^T goes over it
#pragma unroll
        for (int b = 0; b < 4; ++b)
            *reinterpret_cast<float4 *>(Us + (gj0 + b) * LDG + gi0) =
                live ? make_float4(gt[0][b], gt[1][b], gt[2][b], gt[3][b]) : make_float4(0.f, 0.f, 0.f, 0.f);
        __syncthreads();
        sweep_rows<NGV>(acc, Us, LDG, Xs, LDV, ti, tc, 4 * ti + 4, -1.f);
    }
    __syncthreads();
    // U' = T * RHS (RHS parked in Xs)
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int g = 0; g < NGV; ++g) *reinterpret_cast<float4 *>(Xs + (4 * ti + a) * LDV + 4 * tc + 64 * g) = acc[a][g];
    // diag(beta Gamma) K for W
    for (int e = tid; e < C * (DK / 4); e += NT) {
        const int i = e / (DK / 4), m4 = e % (DK / 4);
        const float f = bet[i] * expf(lam[i]);
        float4 *p = reinterpret_cast<float4 *>(Ks + i * LDK + 4 * m4);
        float4 x = *p;
        x.x *= f;
        x.y *= f;
        x.z *= f;
        x.w *= f;
        *p = x;
    }
    __syncthreads();
    {
        float4 o[4][NGV];
#pragma unroll
        for (int a = 0; a < 4; ++a)
#pragma unroll
            for (int g = 0; g < NGV; ++g) o[a][g] = make_float4(0.f, 0.f, 0.f, 0.f);
        sweep_rows<NGV>(o, Tt, LDG, Xs, LDV, ti, tc, 4 * ti + 4, 1.f);
#pragma unroll
        for (int a = 0; a < 4; ++a) {
            float *up = Up_ws + ((size_t)bh * NC * C + t0 + 4 * ti + a) * DV;
#pragma unroll
            for (int g = 0; g < NGV; ++g) *reinterpret_cast<float4 *>(up + 4 * tc + 64 * g) = o[a][g];
        }
    }
    {
        float4 o[4][NGK];
#pragma unroll
        for (int a = 0; a < 4; ++a)
#pragma unroll
            for (int g = 0; g < NGK; ++g) o[a][g] = make_float4(0.f, 0.f, 0.f, 0.f);
        sweep_rows<NGK>(o, Tt, LDG, Ks, LDK, ti, tc, 4 * ti + 4, 1.f);
#pragma unroll
        for (int a = 0; a < 4; ++a) {
            float *wo = W_ws + ((size_t)bh * NC * C + t0 + 4 * ti + a) * DK;
#pragma unroll
            for (int g = 0; g < NGK; ++g) *reinterpret_cast<float4 *>(wo + 4 * tc + 64 * g) = o[a][g];
        }
    }
}

// ---------------------------------------------------------------------------------------------
// Step a6: inter-chunk state passing, sequential over chunks, VB value rows per block, from
// S_init (or 0); S_final, if given, receives the state after the last token.  Each block reads
// and writes only its own rows, so S_final may be S_init.
//
// The block's VB x DK slice of S stays in registers: thread (rg, cg) holds rows RPT rg ..
// RPT rg + RPT - 1 and columns 4 cg .. 4 cg + 3.  A chunk is a sequence of phases: the key phase
// (V~ = U' - W S0^T in 2 x 2 tiles from shared copies of W and S0, then S <- Gamma_C S0 +
// (decayed V~)^T K) and one phase per level (S += (decayed X_l)^T U_l), each an outer-product
// sweep over the chunk's tokens.  The operands of the next phase (K or U_l, and U' or X_l) are
// loaded into registers before the current sweep and parked in shared memory after it, so their
// latency overlaps the sweep; only W is loaded at the phase that uses it.
template <int DK>
struct StateTile {
    static constexpr int LD = DK + 4;     // row stride (floats) of the shared tiles: 16-byte rows
    static constexpr int CG = DK / 4;     // column groups of 4
    static constexpr int RG = NT / CG;    // row groups
    static constexpr int RPT = VB / RG;   // rows per thread
    static constexpr int PB = C * CG / NT;  // float4 groups of a [C x DK] tile per thread
    static_assert(RPT * RG == VB && RPT >= 1 && PB * NT == C * CG && C * VB == 4 * NT, "splits");
    static constexpr size_t SMEM = sizeof(float) * (2 * C * LD + VB * LD + 2 * C * VB + C);
};

template <typename io_t>
struct Raw4;  // 4 io values as loaded from global memory
template <>
struct Raw4<float> {
    using type = float4;
};
template <>
struct Raw4<__nv_bfloat16> {
    using type = uint2;
};
__device__ __forceinline__ float4 raw_to_f4(float4 r) { return r; }
__device__ __forceinline__ float4 raw_to_f4(uint2 w)
{
    const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&w.x));
    const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&w.y));
    return make_float4(a.x, a.y, b.x, b.y);
}

template <typename io_t, int DK>
__global__ void __launch_bounds__(NT) state_kernel(const io_t *__restrict__ k, const io_t *__restrict__ u,
                                                   const float *__restrict__ X, const float *__restrict__ lam_ws,
                                                   const float *__restrict__ W_ws, const float *__restrict__ Up_ws,
                                                   float *__restrict__ S0_ws, float *__restrict__ Vt_ws,
                                                   const float *S_init, float *S_final, int T, int dv, int R, int NC)
{
    using TL = StateTile<DK>;
    using raw_t = typename Raw4<io_t>::type;
    constexpr int LD = TL::LD, CG = TL::CG, RPT = TL::RPT, PB = TL::PB;
    extern __shared__ __align__(16) float smem[];
    float *Ws = smem;             // C x LD   W of the chunk
    float *Ks = Ws + C * LD;      // C x LD   K, then U_l
    float *Ss = Ks + C * LD;      // VB x LD  S at the chunk start
    float *Vs = Ss + VB * LD;     // C x VB   decayed V~, then decayed X_l
    float *Ups = Vs + C * VB;     // C x VB   U' of the block's rows
    float *lam = Ups + C * VB;    // C
    const int bh = blockIdx.x, r0 = blockIdx.y * VB, tid = threadIdx.x;
    const int cg = tid % CG, rg = tid / CG;
    const int ip = tid >> 3, rp = tid & 7;  // V~ tile: tokens 2 ip, 2 ip + 1; rows 2 rp, 2 rp + 1
    const int xi = tid >> 2, xq = tid & 3;  // this thread's float4 of a [C x VB] tile: row xi, columns 4 xq

    float4 s[RPT];
#pragma unroll
    for (int r = 0; r < RPT; ++r)
        s[r] = S_init ? ld4(S_init + ((size_t)bh * dv + r0 + rg * RPT + r) * DK + 4 * cg) : make_float4(0.f, 0.f, 0.f, 0.f);

    // operands of one phase in registers: ph = c (1 + R) + 1 + l, l = -1 for the key phase
    raw_t pb[PB];
    float4 px;
    float pl = 0.f;
    auto prefetch = [&](int ph) {
        const int c = ph / (1 + R), l = ph % (1 + R) - 1;
        if (c >= NC) return;
        const int t0 = c * C, n = min(C, T - t0);
        const io_t *src = (l < 0) ? k + ((size_t)bh * T + t0) * DK : u + (((size_t)bh * T + t0) * R + l) * DK;
        const size_t stride = (l < 0) ? DK : (size_t)R * DK;
#pragma unroll
        for (int q = 0; q < PB; ++q) {
            const int e = tid + q * NT, i = e / CG, m4 = e % CG;
            if (i < n)
                pb[q] = *reinterpret_cast<const raw_t *>(src + (size_t)i * stride + 4 * m4);
            else
                pb[q] = raw_t{};
        }
        if (l < 0) {
            px = ld4(Up_ws + ((size_t)bh * NC * C + t0 + xi) * dv + r0 + 4 * xq);
            if (tid < C) pl = lam_ws[(size_t)bh * T + t0 + min(tid, n - 1)];
        } else {
            px = (xi < n) ? ld4(X + (((size_t)bh * T + t0 + xi) * R + l) * dv + r0 + 4 * xq)
                          : make_float4(0.f, 0.f, 0.f, 0.f);
        }
    };
    auto park_b = [&]() {
#pragma unroll
        for (int q = 0; q < PB; ++q) {
            const int e = tid + q * NT, i = e / CG, m4 = e % CG;
            *reinterpret_cast<float4 *>(Ks + i * LD + 4 * m4) = raw_to_f4(pb[q]);
        }
    };
    // S += V^T B over the chunk's tokens (V in Vs, B in Ks)
    auto sweep = [&]() {
#pragma unroll 4
        for (int i = 0; i < C; ++i) {
            const float4 b4 = ld4(Ks + i * LD + 4 * cg);
#pragma unroll
            for (int r = 0; r < RPT; ++r) {
                const float v = Vs[i * VB + rg * RPT + r];
                s[r].x = fmaf(v, b4.x, s[r].x);
                s[r].y = fmaf(v, b4.y, s[r].y);
                s[r].z = fmaf(v, b4.z, s[r].z);
                s[r].w = fmaf(v, b4.w, s[r].w);
            }
        }
    };

    prefetch(0);
    int ph = 0;
    for (int c = 0; c < NC; ++c) {
        const int t0 = c * C;
        const int n = min(C, T - t0);
        __syncthreads();  // the previous sweep is done: the shared tiles are free
        park_b();
        *reinterpret_cast<float4 *>(Ups + xi * VB + 4 * xq) = px;
        if (tid < C) lam[tid] = pl;
        float *s0 = S0_ws + ((size_t)bh * NC + c) * dv * DK;
#pragma unroll
        for (int r = 0; r < RPT; ++r) {
            const int row = rg * RPT + r;
            *reinterpret_cast<float4 *>(s0 + (size_t)(r0 + row) * DK + 4 * cg) = s[r];
            *reinterpret_cast<float4 *>(Ss + row * LD + 4 * cg) = s[r];
        }
        const float *wb = W_ws + ((size_t)bh * NC * C + t0) * DK;
#pragma unroll
        for (int q = 0; q < PB; ++q) {
            const int e = tid + q * NT, i = e / CG, m4 = e % CG;
            *reinterpret_cast<float4 *>(Ws + i * LD + 4 * m4) = ld4(wb + (size_t)i * DK + 4 * m4);
        }
        __syncthreads();
        prefetch(++ph);  // the first level (or the next chunk's key phase)
        const float lam_last = lam[C - 1];
        {  // V~ = U' - W S0^T, and its decayed copy for the state update
            float a00 = 0.f, a01 = 0.f, a10 = 0.f, a11 = 0.f;
            const float *w0 = Ws + (2 * ip) * LD, *w1 = w0 + LD;
            const float *sa = Ss + (2 * rp) * LD, *sb = sa + LD;
#pragma unroll 8
            for (int m = 0; m < DK; m += 4) {
                const float4 x0 = ld4(w0 + m), x1 = ld4(w1 + m), y0 = ld4(sa + m), y1 = ld4(sb + m);
                a00 = dot4(x0, y0, a00);
                a01 = dot4(x0, y1, a01);
                a10 = dot4(x1, y0, a10);
                a11 = dot4(x1, y1, a11);
            }
            const float acc[2][2] = {{a00, a01}, {a10, a11}};
#pragma unroll
            for (int di = 0; di < 2; ++di) {
                const int i = 2 * ip + di;
                const float2 up = *reinterpret_cast<const float2 *>(Ups + i * VB + 2 * rp);
                const float2 vt = make_float2(up.x - acc[di][0], up.y - acc[di][1]);
                *reinterpret_cast<float2 *>(Vt_ws + ((size_t)bh * NC * C + t0 + i) * dv + r0 + 2 * rp) = vt;
                const float f = (i < n) ? expf(lam_last - lam[i]) : 0.f;
                Vs[i * VB + 2 * rp] = vt.x * f;
                Vs[i * VB + 2 * rp + 1] = vt.y * f;
            }
        }
        __syncthreads();
        const float gC = expf(lam_last);
#pragma unroll
        for (int r = 0; r < RPT; ++r) {
            s[r].x *= gC;
            s[r].y *= gC;
            s[r].z *= gC;
            s[r].w *= gC;
        }
        sweep();
        for (int l = 0; l < R; ++l) {
            __syncthreads();
            park_b();
            {
                const float f = (xi < n) ? expf(lam_last - lam[xi]) : 0.f;
                *reinterpret_cast<float4 *>(Vs + xi * VB + 4 * xq) = make_float4(px.x * f, px.y * f, px.z * f, px.w * f);
            }
            __syncthreads();
            prefetch(++ph);
            sweep();
        }
    }
    if (S_final)
#pragma unroll
        for (int r = 0; r < RPT; ++r)
            *reinterpret_cast<float4 *>(S_final + ((size_t)bh * dv + r0 + rg * RPT + r) * DK + 4 * cg) = s[r];
}

// ---------------------------------------------------------------------------------------------
// Step a7: O = diag(Gamma) Q S0^T + (Q K^T o D) V~ + sum_l (Q U_l^T o D) X_l.
//
// Register-tiled: thread (ti, tc) accumulates rows 4 ti .. 4 ti + 3 of O and the NCW float4
// column groups 4 tc + 64 g.  Q stays in shared memory; per source (K with V~, then U_l with
// X_l) the scores G = (Q B^T o D) are formed in 4 x 4 tiles (causal tiles only), parked
// transposed over B's tile, and swept into O one token j at a time (one float4 of G^T and NCW
// float4s of V~ or X_l per step).
template <int DK, int DV>
struct OutTile {
    static constexpr int LDK = DK + 4, LDV = DV + 4, LDG = C + 4;
    static constexpr int NCW = DV / 64;  // float4 column groups per thread
    // Q | (S0 ; or B-then-G^T | M) | lam
    static constexpr int B_FLOATS = (C * LDK > C * LDG ? C * LDK : C * LDG);
    static constexpr int REGION = (DV * LDK > B_FLOATS + C * LDV ? DV * LDK : B_FLOATS + C * LDV);
    static constexpr size_t SMEM = sizeof(float) * (C * LDK + REGION + C);
};

template <typename T4>
__device__ __forceinline__ void st_out4(T4 *p, float4 v);
template <>
__device__ __forceinline__ void st_out4<float>(float *p, float4 v) { *reinterpret_cast<float4 *>(p) = v; }
template <>
__device__ __forceinline__ void st_out4<__nv_bfloat16>(__nv_bfloat16 *p, float4 v)
{
    __nv_bfloat162 lo = __floats2bfloat162_rn(v.x, v.y), hi = __floats2bfloat162_rn(v.z, v.w);
    uint2 w;
    w.x = *reinterpret_cast<uint32_t *>(&lo);
    w.y = *reinterpret_cast<uint32_t *>(&hi);
    *reinterpret_cast<uint2 *>(p) = w;
}

template <typename io_t, typename out_t, int DK, int DV>
__global__ void __launch_bounds__(NT) out_kernel(const io_t *__restrict__ q, const io_t *__restrict__ k,
                                                 const io_t *__restrict__ u, const float *__restrict__ X,
                                                 const float *__restrict__ lam_ws, const float *__restrict__ S0_ws,
                                                 const float *__restrict__ Vt_ws, out_t *__restrict__ out,
                                                 int T, int R, int NC)
{
    using TL = OutTile<DK, DV>;
    constexpr int LDK = TL::LDK, LDV = TL::LDV, LDG = TL::LDG, NCW = TL::NCW;
    extern __shared__ __align__(16) float smem[];
    float *Qs = smem;                      // C x LDK
    float *S0s = Qs + C * LDK;             // DV x LDK (first phase)
    float *Bs = S0s;                       // C x LDK  K or U_l, then G^T (C x LDG)
    float *Ms = Bs + TL::B_FLOATS;         // C x LDV  V~ or X_l
    float *lam = Qs + C * LDK + TL::REGION;
    const int c = blockIdx.x, bh = blockIdx.y, tid = threadIdx.x;
    const int t0 = c * C;
    const int n = min(C, T - t0);
    const int ti = tid >> 4, tc = tid & 15;  // O tile: rows 4 ti + a, column groups 4 tc + 64 g

    const io_t *qb = q + ((size_t)bh * T + t0) * DK;
    for (int e = tid; e < C * (DK / 4); e += NT) {
        const int i = e / (DK / 4), m4 = e % (DK / 4);
        const float4 v = (i < n) ? ld4(qb + (size_t)i * DK + 4 * m4) : make_float4(0.f, 0.f, 0.f, 0.f);
        *reinterpret_cast<float4 *>(Qs + i * LDK + 4 * m4) = v;
    }
    const float *s0 = S0_ws + ((size_t)bh * NC + c) * DV * DK;
    for (int e = tid; e < DV * (DK / 4); e += NT) {
        const int r = e / (DK / 4), m4 = e % (DK / 4);
        *reinterpret_cast<float4 *>(S0s + r * LDK + 4 * m4) = ld4(s0 + (size_t)r * DK + 4 * m4);
    }
    if (tid < C) lam[tid] = lam_ws[(size_t)bh * T + t0 + min(tid, n - 1)];
    __syncthreads();

    float4 acc[4][NCW];
    {  // diag(Gamma) Q S0^T
#pragma unroll
        for (int a = 0; a < 4; ++a)
#pragma unroll
            for (int g = 0; g < NCW; ++g) acc[a][g] = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 2
        for (int m = 0; m < DK; m += 4) {
            float4 qv[4];
#pragma unroll
            for (int a = 0; a < 4; ++a) qv[a] = ld4(Qs + (4 * ti + a) * LDK + m);
#pragma unroll
            for (int g = 0; g < NCW; ++g) {
                float4 sv[4];
#pragma unroll
                for (int b = 0; b < 4; ++b) sv[b] = ld4(S0s + (4 * tc + 64 * g + b) * LDK + m);
#pragma unroll
                for (int a = 0; a < 4; ++a) {
                    acc[a][g].x = dot4(qv[a], sv[0], acc[a][g].x);
                    acc[a][g].y = dot4(qv[a], sv[1], acc[a][g].y);
                    acc[a][g].z = dot4(qv[a], sv[2], acc[a][g].z);
                    acc[a][g].w = dot4(qv[a], sv[3], acc[a][g].w);
                }
            }
        }
#pragma unroll
        for (int a = 0; a < 4; ++a) {
            const float gi = expf(lam[4 * ti + a]);
#pragma unroll
            for (int g = 0; g < NCW; ++g) {
                acc[a][g].x *= gi;
                acc[a][g].y *= gi;
                acc[a][g].z *= gi;
                acc[a][g].w *= gi;
            }
        }
    }
    const int gi0 = 4 * (tid >> 4), gj0 = 4 * (tid & 15);  // score tile: rows gi0.., columns gj0..
    for (int l = -1; l < R; ++l) {  // l = -1: keys with V~, then each level with its X_l
        __syncthreads();  // S0s / the previous G^T and M are no longer read
        const io_t *bsrc = (l < 0) ? k + ((size_t)bh * T + t0) * DK : u + (((size_t)bh * T + t0) * R + l) * DK;
        const size_t bstride = (l < 0) ? DK : (size_t)R * DK;
        for (int e = tid; e < C * (DK / 4); e += NT) {
            const int i = e / (DK / 4), m4 = e % (DK / 4);
            const float4 v = (i < n) ? ld4(bsrc + (size_t)i * bstride + 4 * m4) : make_float4(0.f, 0.f, 0.f, 0.f);
            *reinterpret_cast<float4 *>(Bs + i * LDK + 4 * m4) = v;
        }
        for (int e = tid; e < C * (DV / 4); e += NT) {
            const int i = e / (DV / 4), m4 = e % (DV / 4);
            float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
            if (i < n)
                v = (l < 0) ? ld4(Vt_ws + ((size_t)bh * NC * C + t0 + i) * DV + 4 * m4)
                            : ld4(X + (((size_t)bh * T + t0 + i) * R + l) * DV + 4 * m4);
            *reinterpret_cast<float4 *>(Ms + i * LDV + 4 * m4) = v;
        }
        __syncthreads();
        // scores of the causal 4 x 4 tiles (j <= i), decayed
        float gt[4][4];
        const bool live = gj0 <= gi0 + 3;
        if (live) {
#pragma unroll
            for (int a = 0; a < 4; ++a)
#pragma unroll
                for (int b = 0; b < 4; ++b) gt[a][b] = 0.f;
#pragma unroll 2
            for (int m = 0; m < DK; m += 4) {
                float4 qv[4], bv[4];
#pragma unroll
                for (int a = 0; a < 4; ++a) qv[a] = ld4(Qs + (gi0 + a) * LDK + m);
#pragma unroll
                for (int b = 0; b < 4; ++b) bv[b] = ld4(Bs + (gj0 + b) * LDK + m);
#pragma unroll
                for (int a = 0; a < 4; ++a)
#pragma unroll
                    for (int b = 0; b < 4; ++b) gt[a][b] = dot4(qv[a], bv[b], gt[a][b]);
            }
#pragma unroll
            for (int a = 0; a < 4; ++a)
#pragma unroll
                for (int b = 0; b < 4; ++b) {
                    const int i = gi0 + a, j = gj0 + b;
                    gt[a][b] = (j <= i) ? gt[a][b] * expf(lam[i] - lam[j]) : 0.f;
                }
        }
        __syncthreads();  // B is no longer read: G^T goes over it
        float *Gt = Bs;   // C x LDG, Gt[j][i]
#pragma unroll
        for (int b = 0; b < 4; ++b)
            *reinterpret_cast<float4 *>(Gt + (gj0 + b) * LDG + gi0) =
                live ? make_float4(gt[0][b], gt[1][b], gt[2][b], gt[3][b]) : make_float4(0.f, 0.f, 0.f, 0.f);
        __syncthreads();
        const int jend = 4 * ti + 4;  // tokens j <= the tile's last row
#pragma unroll 4
        for (int j = 0; j < jend; ++j) {
            const float4 gv = ld4(Gt + j * LDG + 4 * ti);
#pragma unroll
            for (int g = 0; g < NCW; ++g) {
                const float4 mv = ld4(Ms + j * LDV + 4 * tc + 64 * g);
                const float ga[4] = {gv.x, gv.y, gv.z, gv.w};
#pragma unroll
                for (int a = 0; a < 4; ++a) {
                    acc[a][g].x = fmaf(ga[a], mv.x, acc[a][g].x);
                    acc[a][g].y = fmaf(ga[a], mv.y, acc[a][g].y);
                    acc[a][g].z = fmaf(ga[a], mv.z, acc[a][g].z);
                    acc[a][g].w = fmaf(ga[a], mv.w, acc[a][g].w);
                }
            }
        }
    }
#pragma unroll
    for (int a = 0; a < 4; ++a) {
        const int i = 4 * ti + a;
        if (i < n) {
            out_t *o = out + ((size_t)bh * T + t0 + i) * DV;
#pragma unroll
            for (int g = 0; g < NCW; ++g) st_out4<out_t>(o + 4 * tc + 64 * g, acc[a][g]);
        }
    }
}

// ---------------------------------------------------------------------------------------------
// dynamic shared memory of the chunk-solve kernel (the product kernels size theirs with their
// tile structs)
static size_t solve_smem_bytes(int dk) { return sizeof(float) * (C * (dk + 1) + 2 * C * (C + 1) + 2 * C); }

template <typename io_t>
static cudaError_t prepare_t(int dk, int dv)
{
    (void)dv;
    cudaError_t e;
    if ((e = cudaFuncSetAttribute(chunk_solve_kernel<io_t>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  (int)solve_smem_bytes(dk))))
        return e;
#define PRISM_WY_ATTR(DK_, DV_)                                                                                   \
    if ((e = cudaFuncSetAttribute(wy_kernel<io_t, DK_, DV_>, cudaFuncAttributeMaxDynamicSharedMemorySize,              \
                                  (int)WyTile<DK_, DV_>::SMEM)))                                                       \
        return e;
    PRISM_WY_ATTR(64, 64)
    PRISM_WY_ATTR(64, 128)
    PRISM_WY_ATTR(128, 64)
    PRISM_WY_ATTR(128, 128)
#undef PRISM_WY_ATTR
    if ((e = cudaFuncSetAttribute(state_kernel<io_t, 64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  (int)StateTile<64>::SMEM)))
        return e;
    if ((e = cudaFuncSetAttribute(state_kernel<io_t, 128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  (int)StateTile<128>::SMEM)))
        return e;
#define PRISM_OUT_ATTR(DK_, DV_)                                                                                  \
    if ((e = cudaFuncSetAttribute(out_kernel<io_t, float, DK_, DV_>, cudaFuncAttributeMaxDynamicSharedMemorySize,       \
                                  (int)OutTile<DK_, DV_>::SMEM)))                                                      \
        return e;                                                                                                      \
    if ((e = cudaFuncSetAttribute(out_kernel<io_t, __nv_bfloat16, DK_, DV_>,                                          \
                                  cudaFuncAttributeMaxDynamicSharedMemorySize, (int)OutTile<DK_, DV_>::SMEM)))         \
        return e;
    PRISM_OUT_ATTR(64, 64)
    PRISM_OUT_ATTR(64, 128)
    PRISM_OUT_ATTR(128, 64)
    PRISM_OUT_ATTR(128, 128)
#undef PRISM_OUT_ATTR
    return cudaSuccess;
}

template <typename io_t, typename out_t>
static cudaError_t forward_t(const Shape &s, const ForwardArgs &a, const SimtWorkspace &w, KernelTimer &tm)
{
    cudaStream_t st = tm.stream;
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
    chunk_solve_kernel<io_t><<<dim3(s.NC, s.BH), NT, solve_smem_bytes(s.dk), st>>>(k, a.beta, a.alpha, w.lam, w.Tm, s.T, s.dk, s.NC);
    tm.end();
    tm.begin("simt_wy");
    {
        const dim3 grid(s.NC, s.BH);
        if (s.dk == 64 && s.dv == 64)
            wy_kernel<io_t, 64, 64><<<grid, NT, WyTile<64, 64>::SMEM, st>>>(k, v, a.beta, u, w.X, w.lam, w.Tm, w.W, w.Up, s.T, s.R, s.NC);
        else if (s.dk == 64)
            wy_kernel<io_t, 64, 128><<<grid, NT, WyTile<64, 128>::SMEM, st>>>(k, v, a.beta, u, w.X, w.lam, w.Tm, w.W, w.Up, s.T, s.R, s.NC);
        else if (s.dv == 64)
            wy_kernel<io_t, 128, 64><<<grid, NT, WyTile<128, 64>::SMEM, st>>>(k, v, a.beta, u, w.X, w.lam, w.Tm, w.W, w.Up, s.T, s.R, s.NC);
        else
            wy_kernel<io_t, 128, 128><<<grid, NT, WyTile<128, 128>::SMEM, st>>>(k, v, a.beta, u, w.X, w.lam, w.Tm, w.W, w.Up, s.T, s.R, s.NC);
    }
    tm.end();
    tm.begin("simt_state");
    if (s.dk == 64)
        state_kernel<io_t, 64><<<dim3(s.BH, s.dv / VB), NT, StateTile<64>::SMEM, st>>>(
            k, u, w.X, w.lam, w.W, w.Up, w.S0, w.Vt, a.S_init, a.S_final, s.T, s.dv, s.R, s.NC);
    else
        state_kernel<io_t, 128><<<dim3(s.BH, s.dv / VB), NT, StateTile<128>::SMEM, st>>>(
            k, u, w.X, w.lam, w.W, w.Up, w.S0, w.Vt, a.S_init, a.S_final, s.T, s.dv, s.R, s.NC);
    tm.end();
    tm.begin("simt_out");
    {
        const dim3 grid(s.NC, s.BH);
        if (s.dk == 64 && s.dv == 64)
            out_kernel<io_t, out_t, 64, 64><<<grid, NT, OutTile<64, 64>::SMEM, st>>>(q, k, u, w.X, w.lam, w.S0, w.Vt, out, s.T, s.R, s.NC);
        else if (s.dk == 64)
            out_kernel<io_t, out_t, 64, 128><<<grid, NT, OutTile<64, 128>::SMEM, st>>>(q, k, u, w.X, w.lam, w.S0, w.Vt, out, s.T, s.R, s.NC);
        else if (s.dv == 64)
            out_kernel<io_t, out_t, 128, 64><<<grid, NT, OutTile<128, 64>::SMEM, st>>>(q, k, u, w.X, w.lam, w.S0, w.Vt, out, s.T, s.R, s.NC);
        else
            out_kernel<io_t, out_t, 128, 128><<<grid, NT, OutTile<128, 128>::SMEM, st>>>(q, k, u, w.X, w.lam, w.S0, w.Vt, out, s.T, s.R, s.NC);
    }
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
