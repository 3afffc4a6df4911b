// Backward pass of the PRISM memory recurrence (portable fp32 kernels, no tensor cores).
//
// The recurrence S_t = S_{t-1} A_t + B_t with A_t = alpha_t (I - beta_t k_t k_t^T) acts on each
// row of S on its own (row i of S_t depends only on row i of S_{t-1}; notes on PRISM, section
// 2.2), and so does its transpose, the carry of the state cotangent
//   dS_{t-1} = alpha_t (dS_t - beta_t (dS_t k_t) k_t^T),   dS_t += dout_t q_t^T first.
// So the two sequential scans run eight lanes per state row, token by token, with the row in
// registers and one dot product on the dependency chain per token.  They do not
// depend on each other and run side by side in one launch (scan_kernel):
//   forward half   S_{t-1} for every t -> workspace (forward order)
//   reverse half   dS_t for every t -> workspace, z_t = dS_t k_t, dx_{t,l} = dS_t u_{t,l}
//                  (reverse order)
// Everything that needs sums over the rows is then token-parallel:
//   token_grad   dq, dk, du, dalpha, dbeta and the write's share of dv, from S_{t-1}, dS_t
//   chain_grad   the residual chain and gain backwards: dgamma, deta, dh and e's share of dv
//   conv_grad    the short convolution backwards: v's share, dv_hist, per-tile dconv_w sums
//   conv_reduce  dconv_w = the sum of the tiles over the batch
// The formulas (reverse-mode differentiation of the sequential definition), with P = S_{t-1},
// y = P k_t, z = dS_t k_t:
//   dq_t = S_t^T dout_t = alpha P^T dout - alpha beta k (y . dout) + beta k (v . dout)
//          + sum_l u_l (x_l . dout)
//   dk_t = dS_t^T (beta v - alpha beta y) - alpha beta P^T z
//   dalpha_t = <dS_t, P> - beta y . z,   dbeta_t = v . z - alpha y . z
//   dv_t += beta z,   du_{t,l} = dS_t^T x_{t,l}
// and per channel, levels l = R .. 1 (the cotangent of r_{t,R+1} is zero):
//   dr_l = gamma_l g dx_l + (1 - eta_l g) dr_{l+1},   dg += gamma_l r_l dx_l - eta_l r_l dr_{l+1}
//   dgamma_l = sum_c g r_l dx_l,   deta_l = -sum_c g r_l dr_{l+1}
//   dv_t += dr_1,   dh_t = -g dr_1 + phi(h) (2 - h^2) dg
// then dv_{t-j} += w_j dh_t and dw_j += dh_t v_{t-j} over the window.
#include <type_traits>

#include "prism_internal.h"
#include "tc_util.h"

namespace prism {
namespace bwd {

constexpr int NT = 256;    // threads of the token-parallel kernels
constexpr int CT = 64;     // tokens per block of the convolution kernel
constexpr int RMAX = 15;   // largest R = L - 1

__device__ __forceinline__ float ldf(const float *p) { return *p; }
__device__ __forceinline__ float ldf(const __nv_bfloat16 *p) { return __bfloat162float(*p); }

__device__ __forceinline__ float warp_sum(float x)
{
#pragma unroll
    for (int o = 16; o; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

// Anchor h, its normal cdf Phi and density phi for channel c of token t of sequence bh.
template <typename io_t>
__device__ __forceinline__ void anchor_at(const io_t *v, const io_t *v_hist, const io_t *conv_w, int bh, int h, int t,
                                          int T, int dv, int c, float &a, float &Phi, float &phi)
{
    const io_t *vb = v + (size_t)bh * T * dv;
    a = 0.f;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const float w = ldf(conv_w + ((size_t)h * 4 + j) * dv + c);
        if (t - j >= 0)
            a = fmaf(w, ldf(vb + (size_t)(t - j) * dv + c), a);
        else if (v_hist)
            a = fmaf(w, ldf(v_hist + ((size_t)bh * 3 + 3 + t - j) * dv + c), a);
    }
    Phi = 0.5f * erfcf(-a * 0.70710678118654752f);
    phi = 0.39894228040143268f * expf(-0.5f * a * a);
}

// Injection factors x_{t,l} = gamma_l g r_l -> X [BH][T][R][dv]; with gains p_gain (the non-linear
// chain) x_{t,l} = gamma_l GELU(p_l r_l) and r_{l+1} = r_l - GELU(p_l r_l) instead.
template <typename io_t>
__global__ void __launch_bounds__(NT) factors_kernel(const io_t *__restrict__ v, const io_t *__restrict__ v_hist,
                                                     const io_t *__restrict__ conv_w, const float *__restrict__ gamma,
                                                     const float *__restrict__ eta, const io_t *__restrict__ p_gain,
                                                     float *__restrict__ X, int H, int T, int dv, int R)
{
    const int bh = blockIdx.y;
    const long long idx = (long long)blockIdx.x * NT + threadIdx.x;
    if (idx >= (long long)T * dv) return;
    const int t = (int)(idx / dv), c = (int)(idx % dv);
    float a, Phi, phi;
    anchor_at(v, v_hist, conv_w, bh, bh % H, t, T, dv, c, a, Phi, phi);
    const float g = fmaf(a, phi, Phi);
    float r = ldf(v + ((size_t)bh * T + t) * dv + c) - a * Phi;
    const size_t tok = (size_t)bh * T + t;
    if (p_gain) {
        for (int l = 0; l < R; ++l) {
            const float z = ldf(p_gain + (tok * R + l) * dv + c) * r;
            const float delta = z * (0.5f * erfcf(-z * 0.70710678118654752f));
            X[(tok * R + l) * dv + c] = gamma[tok * R + l] * delta;
            r -= delta;
        }
        return;
    }
    for (int l = 0; l < R; ++l) {
        X[(tok * R + l) * dv + c] = gamma[tok * R + l] * g * r;
        if (l + 1 < R) r *= 1.f - eta[tok * R + l] * g;  // the last gain is never read
    }
}

// The two sequential scans.  A block of SCAN_WARPS warps owns ROWS = 4 SCAN_WARPS state rows of
// one sequence: each row is spread over 8 lanes (LPR), each lane holding DK / 8 consecutive
// columns, so a row's dot product ends in a 3-step shuffle tree.  The per-token inputs of a
// chunk of `ct` tokens are staged in shared memory by cp.async, in two buffers: the copies of
// the next chunk are in flight while the warps walk the current one, so only the dot product
// and the row update remain on the per-token dependency chain.
constexpr int LPR = 8;                      // lanes per state row
constexpr int SCAN_WARPS = 4;
constexpr int ROWS = SCAN_WARPS * 32 / LPR;  // state rows per scan block (16)

__device__ __forceinline__ uint32_t smem_addr(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void cp16(void *dst, const void *src)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp4(void *dst, const void *src)
{
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_addr(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// Sum over the 8 lanes of a row (lanes 8r .. 8r + 7).
__device__ __forceinline__ float row_sum(float x)
{
    x += __shfl_xor_sync(0xffffffffu, x, 4);
    x += __shfl_xor_sync(0xffffffffu, x, 2);
    x += __shfl_xor_sync(0xffffffffu, x, 1);
    return x;
}

// N consecutive values from a 16-byte aligned address (shared or global) as floats.
template <int N>
__device__ __forceinline__ void load_vec(const float *p, float (&o)[N])
{
#pragma unroll
    for (int e = 0; e < N; e += 4) {
        const float4 t = *reinterpret_cast<const float4 *>(p + e);
        o[e] = t.x;
        o[e + 1] = t.y;
        o[e + 2] = t.z;
        o[e + 3] = t.w;
    }
}
template <int N>
__device__ __forceinline__ void load_vec(const __nv_bfloat16 *p, float (&o)[N])
{
#pragma unroll
    for (int e = 0; e < N; e += 8) {
        const uint4 t = *reinterpret_cast<const uint4 *>(p + e);
        const uint32_t wds[4] = {t.x, t.y, t.z, t.w};
#pragma unroll
        for (int h = 0; h < 4; ++h) {
            const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&wds[h]));
            o[e + 2 * h] = f.x;
            o[e + 2 * h + 1] = f.y;
        }
    }
}
template <int N>
__device__ __forceinline__ void store_vec(float *p, const float (&o)[N])
{
#pragma unroll
    for (int e = 0; e < N; e += 4) *reinterpret_cast<float4 *>(p + e) = make_float4(o[e], o[e + 1], o[e + 2], o[e + 3]);
}

// Byte offsets of one stage buffer of `ct` tokens (each part a multiple of 16 bytes).
struct StageLayout {
    int q, k, u, row, x, gate, bytes;
};
__host__ __device__ inline int align16(int n) { return (n + 15) & ~15; }
__host__ __device__ inline StageLayout stage_layout(int ct, int dk, int R, int io_bytes)
{
    StageLayout s;
    s.q = 0;                                        // q [ct][dk] io (reverse half)
    s.k = s.q + align16(ct * dk * io_bytes);        // k [ct][dk] io
    s.u = s.k + align16(ct * dk * io_bytes);        // u [ct][R][dk] io
    s.row = s.u + align16(ct * R * dk * io_bytes);  // v (io) or dout (fp32) of the ROWS rows, 64 B a token
    s.x = s.row + ct * ROWS * 4;                    // x [ct][R][ROWS] fp32 (forward half)
    s.gate = s.x + ct * R * ROWS * 4;               // alpha [ct], beta [ct] fp32
    s.bytes = s.gate + align16(2 * ct * 4);
    return s;
}

// Queue the copies of tokens [t0, t0 + n) of sequence bh for rows i0 .. i0 + ROWS - 1.
template <typename io_t, int DK>
__device__ __forceinline__ void stage_issue(char *buf, const StageLayout &L, bool reverse, const io_t *q,
                                            const io_t *k, const io_t *u, const io_t *v, const float *dout,
                                            const float *X, const float *alpha, const float *beta, int bh, int T,
                                            int t0, int n, int dv, int R, int i0)
{
    const int tid = threadIdx.x, nth = SCAN_WARPS * 32;
    const size_t tok0 = (size_t)bh * T + t0;
    constexpr int PER16 = 16 / sizeof(io_t);
    const int nk = n * DK / PER16;  // 16-byte pieces of k (and q)
    for (int p = tid; p < nk; p += nth) {
        cp16(buf + L.k + p * 16, k + tok0 * DK + (size_t)p * PER16);
        if (reverse) cp16(buf + L.q + p * 16, q + tok0 * DK + (size_t)p * PER16);
    }
    const int nu = n * R * DK / PER16;
    for (int p = tid; p < nu; p += nth) cp16(buf + L.u + p * 16, u + tok0 * R * DK + (size_t)p * PER16);
    // the rows' entries of v (ROWS io values) or of dout (ROWS floats): 16-byte pieces
    const int row_pieces = reverse ? ROWS * 4 / 16 : ROWS * (int)sizeof(io_t) / 16;
    for (int p = tid; p < n * row_pieces; p += nth) {
        const int tt = p / row_pieces, pc = p % row_pieces;
        if (reverse) cp16(buf + L.row + tt * ROWS * 4 + pc * 16, dout + (tok0 + tt) * dv + i0 + pc * 4);
        else cp16(buf + L.row + tt * ROWS * 4 + pc * 16, v + (tok0 + tt) * dv + i0 + pc * PER16);
    }
    for (int p = tid; p < n; p += nth) {
        cp4(buf + L.gate + p * 4, alpha + tok0 + p);
        cp4(buf + L.gate + (n + p) * 4, beta + tok0 + p);
    }
    if (!reverse)
        for (int p = tid; p < n * R * (ROWS / 4); p += nth) {
            const int tl = p / (ROWS / 4), pc = p % (ROWS / 4);  // (token, level) pair and its piece
            cp16(buf + L.x + tl * ROWS * 4 + pc * 16, X + ((tok0 + tl / R) * R + tl % R) * dv + i0 + pc * 4);
        }
}

// NPL io values as raw 16-byte words (read from shared memory ahead of their use).
template <typename io_t, int N>
struct Raw {
    static constexpr int W = N * (int)sizeof(io_t) / 16;
    uint4 w[W];
};
template <typename io_t, int N>
__device__ __forceinline__ void load_raw(const io_t *p, Raw<io_t, N> &r)
{
#pragma unroll
    for (int j = 0; j < Raw<io_t, N>::W; ++j) r.w[j] = reinterpret_cast<const uint4 *>(p)[j];
}
template <int N>
__device__ __forceinline__ void unpack(const Raw<float, N> &r, float (&o)[N])
{
#pragma unroll
    for (int j = 0; j < N / 4; ++j) {
        o[4 * j] = __uint_as_float(r.w[j].x);
        o[4 * j + 1] = __uint_as_float(r.w[j].y);
        o[4 * j + 2] = __uint_as_float(r.w[j].z);
        o[4 * j + 3] = __uint_as_float(r.w[j].w);
    }
}
template <int N>
__device__ __forceinline__ void unpack(const Raw<__nv_bfloat16, N> &r, float (&o)[N])
{
    // a 32-bit word holds two consecutive bf16 values, the first in its low half
#pragma unroll
    for (int j = 0; j < N / 8; ++j) {
        const uint32_t wd[4] = {r.w[j].x, r.w[j].y, r.w[j].z, r.w[j].w};
#pragma unroll
        for (int h = 0; h < 4; ++h) {
            o[8 * j + 2 * h] = __uint_as_float(wd[h] << 16);
            o[8 * j + 2 * h + 1] = __uint_as_float(wd[h] & 0xffff0000u);
        }
    }
}

// One token's inputs for a lane of the forward half and of the reverse half.
template <typename io_t, int N, int RT>
struct FwdTok {
    Raw<io_t, N> k, u[RT > 0 ? RT : 1];
    float x[RT > 0 ? RT : 1], a, b, v;
};
template <typename io_t, int N, int RT>
struct RevTok {
    Raw<io_t, N> k, q, u[RT > 0 ? RT : 1];
    float d, a, b;
};
template <typename io_t, int N, int RT>
__device__ __forceinline__ void fetch_fwd(FwdTok<io_t, N, RT> &f, const io_t *kS, const io_t *uS, const float *xS,
                                          const io_t *vS, const float *aS, const float *bS, int tt, int dk, int col,
                                          int rw)
{
    load_raw(kS + tt * dk + col, f.k);
#pragma unroll
    for (int l = 0; l < RT; ++l) {
        load_raw(uS + (tt * RT + l) * dk + col, f.u[l]);
        f.x[l] = xS[(tt * RT + l) * ROWS + rw];
    }
    f.a = aS[tt];
    f.b = bS[tt];
    f.v = ldf(vS + tt * (ROWS * 4 / (int)sizeof(io_t)) + rw);
}
template <typename io_t, int N, int RT>
__device__ __forceinline__ void fetch_rev(RevTok<io_t, N, RT> &f, const io_t *kS, const io_t *qS, const io_t *uS,
                                          const float *dS, const float *aS, const float *bS, int tt, int dk, int col,
                                          int rw)
{
    load_raw(kS + tt * dk + col, f.k);
    load_raw(qS + tt * dk + col, f.q);
#pragma unroll
    for (int l = 0; l < RT; ++l) load_raw(uS + (tt * RT + l) * dk + col, f.u[l]);
    f.d = dS[tt * ROWS + rw];
    f.a = aS[tt];
    f.b = bS[tt];
}

// blockIdx.z = 0: S_{t-1} of every token (forward order) -> Sp.
// blockIdx.z = 1: dS_t of every token (reverse order) -> Gs, with z_t = dS_t k_t -> Z and
//                 dx_{t,l} = dS_t u_{t,l} -> dX; the last cotangent -> dS_init.
// RT >= 0: R = RT levels, known at compile time; RT = -1: any R.
template <typename io_t, int DK, int RT>
__global__ void __launch_bounds__(SCAN_WARPS * 32) scan_kernel(
    const io_t *__restrict__ q, const io_t *__restrict__ k, const io_t *__restrict__ v, const io_t *__restrict__ u,
    const float *__restrict__ beta, const float *__restrict__ alpha, const float *__restrict__ X,
    const float *__restrict__ S_init, const float *__restrict__ dout, const float *__restrict__ dS_final,
    float *__restrict__ Sp, float *__restrict__ Gs, float *__restrict__ Z, float *__restrict__ dX,
    float *__restrict__ dS_init, int T, int dv, int R, int ct)
{
    constexpr int NPL = DK / LPR;  // columns per lane
    extern __shared__ __align__(16) char stage[];
    const bool rev = blockIdx.z == 1;
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int rw = w * (32 / LPR) + lane / LPR;  // row within the block
    const int col = (lane % LPR) * NPL;          // first column of this lane
    const bool lead = (lane % LPR) == 0;
    const int bh = blockIdx.y, i0 = blockIdx.x * ROWS, i = i0 + rw;  // grid.x = dv / ROWS
    const size_t DD = (size_t)dv * DK;
    const StageLayout L = stage_layout(ct, DK, R, sizeof(io_t));
    const int nch = (T + ct - 1) / ct;
    float S[NPL];
    const float *S0 = rev ? dS_final : S_init;
    if (S0) load_vec(S0 + bh * DD + (size_t)i * DK + col, S);
    else
#pragma unroll
        for (int e = 0; e < NPL; ++e) S[e] = 0.f;

    auto issue = [&](int c) {
        const int t0 = (rev ? nch - 1 - c : c) * ct;
        stage_issue<io_t, DK>(stage + (c & 1) * L.bytes, L, rev, q, k, u, v, dout, X, alpha, beta, bh, T, t0,
                              min(ct, T - t0), dv, R, i0);
        cp_commit();
    };
    issue(0);
    for (int c = 0; c < nch; ++c) {
        if (c + 1 < nch) {
            issue(c + 1);
            cp_wait<1>();
        } else {
            cp_wait<0>();
        }
        __syncthreads();
        const char *b = stage + (c & 1) * L.bytes;
        const int t0 = (rev ? nch - 1 - c : c) * ct, n = min(ct, T - t0);
        const io_t *kS = reinterpret_cast<const io_t *>(b + L.k);
        const io_t *uS = reinterpret_cast<const io_t *>(b + L.u);
        const float *aS = reinterpret_cast<const float *>(b + L.gate), *bS = aS + n;
        if constexpr (RT >= 0) {
            // the level count is known: each token's shared-memory inputs are read one token
            // ahead into registers, and the rank-R injection is formed off the chain
            if (!rev) {
                const io_t *vS = reinterpret_cast<const io_t *>(b + L.row);
                const float *xS = reinterpret_cast<const float *>(b + L.x);
                FwdTok<io_t, NPL, RT> cur, nxt;
                fetch_fwd(cur, kS, uS, xS, vS, aS, bS, 0, DK, col, rw);
                for (int tt = 0; tt < n; ++tt) {
                    fetch_fwd(nxt, kS, uS, xS, vS, aS, bS, min(tt + 1, n - 1), DK, col, rw);
                    const size_t tok = (size_t)bh * T + t0 + tt;
                    float kk[NPL];
                    unpack(cur.k, kk);
                    store_vec(Sp + tok * DD + (size_t)i * DK + col, S);
                    float y0 = 0.f, y1 = 0.f;
#pragma unroll
                    for (int e = 0; e < NPL; e += 2) {
                        y0 = fmaf(S[e], kk[e], y0);
                        y1 = fmaf(S[e + 1], kk[e + 1], y1);
                    }
                    const float y = row_sum(y0 + y1);
                    float wv[NPL];  // beta v k + sum_l x_l u_l: does not depend on S
                    const float bv = cur.b * cur.v;
#pragma unroll
                    for (int e = 0; e < NPL; ++e) wv[e] = bv * kk[e];
#pragma unroll
                    for (int l = 0; l < RT; ++l) {
                        float ul[NPL];
                        unpack(cur.u[l], ul);
#pragma unroll
                        for (int e = 0; e < NPL; ++e) wv[e] = fmaf(cur.x[l], ul[e], wv[e]);
                    }
                    const float c = -cur.b * y;
#pragma unroll
                    for (int e = 0; e < NPL; ++e) S[e] = fmaf(cur.a, fmaf(c, kk[e], S[e]), wv[e]);
                    cur = nxt;
                }
            } else {
                const io_t *qS = reinterpret_cast<const io_t *>(b + L.q);
                const float *dS = reinterpret_cast<const float *>(b + L.row);
                RevTok<io_t, NPL, RT> cur, nxt;
                fetch_rev(cur, kS, qS, uS, dS, aS, bS, n - 1, DK, col, rw);
                for (int tt = n - 1; tt >= 0; --tt) {
                    fetch_rev(nxt, kS, qS, uS, dS, aS, bS, max(tt - 1, 0), DK, col, rw);
                    const size_t tok = (size_t)bh * T + t0 + tt;
                    float kk[NPL], qq[NPL];
                    unpack(cur.k, kk);
                    unpack(cur.q, qq);
#pragma unroll
                    for (int e = 0; e < NPL; ++e) S[e] = fmaf(cur.d, qq[e], S[e]);
                    store_vec(Gs + tok * DD + (size_t)i * DK + col, S);
                    float z0 = 0.f, z1 = 0.f;
#pragma unroll
                    for (int e = 0; e < NPL; e += 2) {
                        z0 = fmaf(S[e], kk[e], z0);
                        z1 = fmaf(S[e + 1], kk[e + 1], z1);
                    }
                    const float z = row_sum(z0 + z1);
#pragma unroll
                    for (int l = 0; l < RT; ++l) {
                        float ul[NPL];
                        unpack(cur.u[l], ul);
                        float s0 = 0.f, s1 = 0.f;
#pragma unroll
                        for (int e = 0; e < NPL; e += 2) {
                            s0 = fmaf(S[e], ul[e], s0);
                            s1 = fmaf(S[e + 1], ul[e + 1], s1);
                        }
                        const float s = row_sum(s0 + s1);
                        if (lead) dX[(tok * RT + l) * dv + i] = s;
                    }
                    if (lead) Z[tok * dv + i] = z;
                    const float c = -cur.b * z;
#pragma unroll
                    for (int e = 0; e < NPL; ++e) S[e] = cur.a * fmaf(c, kk[e], S[e]);
                    cur = nxt;
                }
            }
        } else if (!rev) {
            const io_t *vS = reinterpret_cast<const io_t *>(b + L.row);
            const float *xS = reinterpret_cast<const float *>(b + L.x);
            for (int tt = 0; tt < n; ++tt) {
                const size_t tok = (size_t)bh * T + t0 + tt;
                float kk[NPL];
                load_vec(kS + tt * DK + col, kk);
                store_vec(Sp + tok * DD + (size_t)i * DK + col, S);
                float y0 = 0.f, y1 = 0.f;
#pragma unroll
                for (int e = 0; e < NPL; e += 2) {
                    y0 = fmaf(S[e], kk[e], y0);
                    y1 = fmaf(S[e + 1], kk[e + 1], y1);
                }
                const float y = row_sum(y0 + y1);
                const float al = aS[tt], be = bS[tt];
                const float vi = ldf(vS + tt * (ROWS * 4 / sizeof(io_t)) + rw);
#pragma unroll
                for (int e = 0; e < NPL; ++e) S[e] = fmaf(al, fmaf(-be * y, kk[e], S[e]), be * vi * kk[e]);
                for (int l = 0; l < R; ++l) {
                    const float xl = xS[(tt * R + l) * ROWS + rw];
                    float ul[NPL];
                    load_vec(uS + (tt * R + l) * DK + col, ul);
#pragma unroll
                    for (int e = 0; e < NPL; ++e) S[e] = fmaf(xl, ul[e], S[e]);
                }
            }
        } else {
            const io_t *qS = reinterpret_cast<const io_t *>(b + L.q);
            const float *dS = reinterpret_cast<const float *>(b + L.row);
            for (int tt = n - 1; tt >= 0; --tt) {
                const size_t tok = (size_t)bh * T + t0 + tt;
                const float di = dS[tt * ROWS + rw];
                float kk[NPL], qq[NPL];
                load_vec(kS + tt * DK + col, kk);
                load_vec(qS + tt * DK + col, qq);
                float z0 = 0.f, z1 = 0.f;
#pragma unroll
                for (int e = 0; e < NPL; ++e) S[e] = fmaf(di, qq[e], S[e]);
                store_vec(Gs + tok * DD + (size_t)i * DK + col, S);
#pragma unroll
                for (int e = 0; e < NPL; e += 2) {
                    z0 = fmaf(S[e], kk[e], z0);
                    z1 = fmaf(S[e + 1], kk[e + 1], z1);
                }
                const float z = row_sum(z0 + z1);
                for (int l = 0; l < R; ++l) {
                    float ul[NPL];
                    load_vec(uS + (tt * R + l) * DK + col, ul);
                    float s0 = 0.f, s1 = 0.f;
#pragma unroll
                    for (int e = 0; e < NPL; e += 2) {
                        s0 = fmaf(S[e], ul[e], s0);
                        s1 = fmaf(S[e + 1], ul[e + 1], s1);
                    }
                    const float s = row_sum(s0 + s1);
                    if (lead) dX[(tok * R + l) * dv + i] = s;
                }
                if (lead) Z[tok * dv + i] = z;
                const float al = aS[tt], be = bS[tt];
#pragma unroll
                for (int e = 0; e < NPL; ++e) S[e] = al * fmaf(-be * z, kk[e], S[e]);
            }
        }
        __syncthreads();  // the buffer is refilled by the copies issued in the next iteration
    }
    if (rev && dS_init) store_vec(dS_init + bh * DD + (size_t)i * DK + col, S);
}

// Tokens per stage buffer: the largest power of two up to 32 whose two buffers fit in kScanSmem.
constexpr int kScanSmem = 96 * 1024;
inline int scan_chunk(int dk, int R, int io_bytes)
{
    int ct = 32;
    while (ct > 1 && 2 * stage_layout(ct, dk, R, io_bytes).bytes > kScanSmem) ct >>= 1;
    return ct;
}

// Shared-memory floats of token_grad_kernel.
__host__ __device__ constexpr size_t token_grad_smem_floats(int dk, int dv, int R)
{
    return (size_t)dv * dk + dk + 4 * (size_t)dv + (size_t)R * dv + (size_t)(NT / dk) * (3 + R) * dk +
           (NT / 32) * (4 + R) + NT / 32 + 4 + R;
}

// Per token: dq, dk, du, dalpha, dbeta and dv <- beta z (the later kernels add to dv).
template <typename io_t, int DK>
__global__ void __launch_bounds__(NT) token_grad_kernel(const io_t *__restrict__ q, const io_t *__restrict__ k,
                                                        const io_t *__restrict__ v, const io_t *__restrict__ u,
                                                        const float *__restrict__ beta,
                                                        const float *__restrict__ alpha,
                                                        const float *__restrict__ X, const float *__restrict__ Sp,
                                                        const float *__restrict__ Gs, const float *__restrict__ Z,
                                                        const float *__restrict__ dout, float *__restrict__ dq,
                                                        float *__restrict__ dk, float *__restrict__ dv_out,
                                                        float *__restrict__ dbeta, float *__restrict__ dalpha,
                                                        float *__restrict__ du, long long ntok, int dv, int R)
{
    constexpr int NG = NT / DK;  // row groups of the column sums
    const int NS = 4 + R;        // per-token scalars: y.dout, v.dout, y.z, v.z, x_l.dout
    extern __shared__ float sm[];
    float *Ps = sm;                         // [dv][DK]  S_{t-1}
    float *ks = Ps + (size_t)dv * DK;       // [DK]
    float *ys = ks + DK;                    // [dv]  y = S_{t-1} k
    float *ws = ys + dv;                    // [dv]  beta v - alpha beta y
    float *ds = ws + dv;                    // [dv]  dout_t
    float *zs = ds + dv;                    // [dv]  z
    float *xs = zs + dv;                    // [R][dv]
    float *cs = xs + (size_t)R * dv;        // [NG][3 + R][DK]
    float *red = cs + (size_t)NG * (3 + R) * DK;  // [NT/32][NS]
    float *redp = red + (NT / 32) * NS;     // [NT/32]  <dS_t, S_{t-1}> per warp
    float *scal = redp + NT / 32;           // [NS]
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    for (long long tok = blockIdx.x; tok < ntok; tok += gridDim.x) {
        const float al = alpha[tok], be = beta[tok];
        const float4 *P4 = reinterpret_cast<const float4 *>(Sp + (size_t)tok * dv * DK);
        for (int n = tid; n < dv * DK / 4; n += NT) reinterpret_cast<float4 *>(Ps)[n] = P4[n];
        for (int j = tid; j < DK; j += NT) ks[j] = ldf(k + (size_t)tok * DK + j);
        if (tid < dv) {
            ds[tid] = dout[(size_t)tok * dv + tid];
            zs[tid] = Z[(size_t)tok * dv + tid];
            for (int l = 0; l < R; ++l) xs[l * dv + tid] = X[((size_t)tok * R + l) * dv + tid];
        }
        __syncthreads();
        for (int i = wid; i < dv; i += NT / 32) {
            float s = 0.f;
            for (int j = lane; j < DK; j += 32) s = fmaf(Ps[i * DK + j], ks[j], s);
            s = warp_sum(s);
            if (lane == 0) ys[i] = s;
        }
        __syncthreads();
        if (tid < dv) {  // dv is a multiple of 32: whole warps
            const float yi = ys[tid], vi = ldf(v + (size_t)tok * dv + tid), di = ds[tid], zi = zs[tid];
            ws[tid] = be * vi - al * be * yi;
            dv_out[(size_t)tok * dv + tid] = be * zi;
            float part[4] = {yi * di, vi * di, yi * zi, vi * zi};
#pragma unroll
            for (int s = 0; s < 4; ++s) {
                const float r = warp_sum(part[s]);
                if (lane == 0) red[wid * NS + s] = r;
            }
            for (int l = 0; l < R; ++l) {
                const float r = warp_sum(xs[l * dv + tid] * di);
                if (lane == 0) red[wid * NS + 4 + l] = r;
            }
        }
        __syncthreads();
        if (tid < NS) {
            float s = 0.f;
            for (int w = 0; w < dv / 32; ++w) s += red[w * NS + tid];
            scal[tid] = s;
        }
        // column sums over the rows of group g
        {
            const int g = tid / DK, j = tid % DK;
            float a = 0.f, c = 0.f, b = 0.f, dsp = 0.f, dul[RMAX];
#pragma unroll
            for (int l = 0; l < RMAX; ++l) dul[l] = 0.f;
            const float *G = Gs + (size_t)tok * dv * DK;
            for (int i = g; i < dv; i += NG) {
                const float p = Ps[i * DK + j], gg = G[(size_t)i * DK + j];
                a = fmaf(p, ds[i], a);
                c = fmaf(p, zs[i], c);
                b = fmaf(gg, ws[i], b);
                dsp = fmaf(gg, p, dsp);
#pragma unroll
                for (int l = 0; l < RMAX; ++l)
                    if (l < R) dul[l] = fmaf(gg, xs[l * dv + i], dul[l]);
            }
            float *cg = cs + (size_t)g * (3 + R) * DK;
            cg[j] = a;
            cg[DK + j] = c;
            cg[2 * DK + j] = b;
#pragma unroll
            for (int l = 0; l < RMAX; ++l)
                if (l < R) cg[(3 + l) * DK + j] = dul[l];
            dsp = warp_sum(dsp);
            if (lane == 0) redp[wid] = dsp;
        }
        __syncthreads();
        if (tid < DK) {
            const int j = tid;
            float A = 0.f, Cc = 0.f, Bb = 0.f;
            for (int g = 0; g < NG; ++g) {
                const float *cg = cs + (size_t)g * (3 + R) * DK;
                A += cg[j];
                Cc += cg[DK + j];
                Bb += cg[2 * DK + j];
            }
            const float kj = ks[j];
            float dqj = al * A - al * be * kj * scal[0] + be * kj * scal[1];
            for (int l = 0; l < R; ++l) {
                float Ul = 0.f;
                for (int g = 0; g < NG; ++g) Ul += cs[((size_t)g * (3 + R) + 3 + l) * DK + j];
                du[((size_t)tok * R + l) * DK + j] = Ul;
                dqj = fmaf(ldf(u + ((size_t)tok * R + l) * DK + j), scal[4 + l], dqj);
            }
            dq[(size_t)tok * DK + j] = dqj;
            dk[(size_t)tok * DK + j] = Bb - al * be * Cc;
        }
        if (tid == 0) {
            float s = 0.f;
            for (int w = 0; w < NT / 32; ++w) s += redp[w];
            dalpha[tok] = s - be * scal[2];
            dbeta[tok] = scal[3] - al * scal[2];
        }
        __syncthreads();  // the shared buffers are reused by the next token
    }
}

// The residual chain and the gain backwards, one warp per token, lane c handling the channel
// pairs 2 (c + 32 k), k < CPL (CPL = dv / 64); every load of the token is issued before the
// arithmetic; the per-level sums over channels (dgamma, deta) are warp reductions.
template <typename io_t>
__device__ __forceinline__ float2 ld2(const io_t *p);
template <>
__device__ __forceinline__ float2 ld2<float>(const float *p)
{
    return *reinterpret_cast<const float2 *>(p);
}
template <>
__device__ __forceinline__ float2 ld2<__nv_bfloat16>(const __nv_bfloat16 *p)
{
    return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(p));
}

// One channel of one token, linear chain: from the anchor a = h_t, v_t and the level cotangents
// dx_l, the chain's share of dv (drn, the cotangent of r_1) and dh; dgam and det gather the
// channel's terms of dgamma and deta.
template <int RM>
__device__ __forceinline__ void chain_lin_channel(float a, float v0, const float (&gm)[RM], const float (&et)[RM],
                                                  const float (&dx)[RM], int R, float (&dgam)[RM], float (&det)[RM],
                                                  float &drn_out, float &dh_out)
{
    float Phi, phi;
    tcu::gauss_parts(a, Phi, phi);
    const float g = fmaf(a, phi, Phi);
    float rl[RM];
    float r = v0 - a * Phi;
#pragma unroll
    for (int l = 0; l < RM; ++l)
        if (l < R) {
            rl[l] = r;
            r *= 1.f - et[l] * g;
        }
    float drn = 0.f, dg = 0.f;
#pragma unroll
    for (int l = RM - 1; l >= 0; --l)
        if (l < R) {
            dgam[l] = fmaf(g * rl[l], dx[l], dgam[l]);
            det[l] = fmaf(-g * rl[l], drn, det[l]);
            dg += gm[l] * rl[l] * dx[l] - et[l] * rl[l] * drn;
            drn = gm[l] * g * dx[l] + (1.f - et[l] * g) * drn;
        }
    drn_out = drn;
    dh_out = -g * drn + phi * (2.f - a * a) * dg;
}

// The same for the non-linear chain (gains pl in place of eta): dp receives the gains' cotangents.
template <int RM>
__device__ __forceinline__ void chain_nl_channel(float a, float v0, const float (&gm)[RM], const float (&pl)[RM],
                                                 const float (&dx)[RM], int R, float (&dgam)[RM], float (&dp)[RM],
                                                 float &drn_out, float &dh_out)
{
    float Phi, phi;
    tcu::gauss_parts(a, Phi, phi);
    const float g = fmaf(a, phi, Phi);
    float rl[RM];  // r_l, kept from the forward steps
    float r = v0 - a * Phi;
#pragma unroll
    for (int l = 0; l < RM; ++l)
        if (l < R) {
            rl[l] = r;
            r -= tcu::gelu_value(pl[l] * r);
        }
    float drn = 0.f;
#pragma unroll
    for (int l = RM - 1; l >= 0; --l)
        if (l < R) {
            const float z = pl[l] * rl[l];
            float Pz, pz;
            tcu::gauss_parts(z, Pz, pz);
            const float ddelta = gm[l] * dx[l] - drn;
            dgam[l] = fmaf(z * Pz, dx[l], dgam[l]);
            const float dz = ddelta * fmaf(z, pz, Pz);
            dp[l] = dz * rl[l];
            drn = fmaf(dz, pl[l], drn);
        }
    drn_out = drn;
    dh_out = -g * drn;
}

template <typename io_t, int CPL, int RM>
__global__ void __launch_bounds__(NT) chain_grad_kernel(const io_t *__restrict__ v, const io_t *__restrict__ v_hist,
                                                        const io_t *__restrict__ conv_w,
                                                        const float *__restrict__ gamma,
                                                        const float *__restrict__ eta, const float *__restrict__ dX,
                                                        float *__restrict__ dH, float *__restrict__ dv_out,
                                                        float *__restrict__ dgamma, float *__restrict__ deta,
                                                        long long ntok, int H, int T, int R)
{
    constexpr int dv = 64 * CPL;
    const int lane = threadIdx.x & 31;
    const long long tok = (long long)blockIdx.x * (NT / 32) + (threadIdx.x >> 5);
    if (tok >= ntok) return;
    const int bh = (int)(tok / T), t = (int)(tok % T), h = bh % H;
    float gm[RM], et[RM];
#pragma unroll
    for (int l = 0; l < RM; ++l) {
        // the last level's gain shapes nothing (the cotangent of r_{t,R+1} is zero)
        gm[l] = l < R ? gamma[(size_t)tok * R + l] : 0.f;
        et[l] = l + 1 < R ? eta[(size_t)tok * R + l] : 0.f;
    }
    float2 vv[CPL][4], w[CPL][4], dxv[CPL][RM], dvo[CPL];  // dvo: dv (beta z) as the kernel found it
#pragma unroll
    for (int k = 0; k < CPL; ++k) {
        const int c = 2 * (lane + 32 * k);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            w[k][j] = ld2(conv_w + ((size_t)h * 4 + j) * dv + c);
            vv[k][j] = make_float2(0.f, 0.f);
            if (t - j >= 0) vv[k][j] = ld2(v + ((size_t)bh * T + t - j) * dv + c);
            else if (v_hist) vv[k][j] = ld2(v_hist + ((size_t)bh * 3 + 3 + t - j) * dv + c);
        }
#pragma unroll
        for (int l = 0; l < RM; ++l)
            if (l < R) dxv[k][l] = *reinterpret_cast<const float2 *>(dX + ((size_t)tok * R + l) * dv + c);
        dvo[k] = *reinterpret_cast<const float2 *>(dv_out + (size_t)tok * dv + c);
    }
    float dgam[RM], det[RM];
#pragma unroll
    for (int l = 0; l < RM; ++l) dgam[l] = det[l] = 0.f;
#pragma unroll
    for (int k = 0; k < CPL; ++k) {
        const int c = 2 * (lane + 32 * k);
        float drn2[2], dh2[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            float a = 0.f;
#pragma unroll
            for (int j = 0; j < 4; ++j) a = fmaf(e ? w[k][j].y : w[k][j].x, e ? vv[k][j].y : vv[k][j].x, a);
            float dx[RM];
#pragma unroll
            for (int l = 0; l < RM; ++l) dx[l] = e ? dxv[k][l].y : dxv[k][l].x;
            chain_lin_channel<RM>(a, e ? vv[k][0].y : vv[k][0].x, gm, et, dx, R, dgam, det, drn2[e], dh2[e]);
        }
        *reinterpret_cast<float2 *>(dv_out + (size_t)tok * dv + c) = make_float2(dvo[k].x + drn2[0], dvo[k].y + drn2[1]);
        *reinterpret_cast<float2 *>(dH + (size_t)tok * dv + c) = make_float2(dh2[0], dh2[1]);
    }
#pragma unroll
    for (int l = 0; l < RM; ++l)
        if (l < R) {
            const float s1 = warp_sum(dgam[l]), s2 = warp_sum(det[l]);
            if (lane == 0) {
                dgamma[(size_t)tok * R + l] = s1;
                deta[(size_t)tok * R + l] = s2;
            }
        }
}

// The non-linear chain backwards (gains p in place of eta), laid out as chain_grad_kernel: per
// channel, the residuals r_l are stepped forwards again (r_{l+1} = r_l - GELU(p_l r_l)), then with
// z = p_l r_l, for l = R .. 1 and the cotangent of r_{R+1} zero:
//   ddelta = gamma_l dx_l - dr_{l+1},  dgamma_l += GELU(z) dx_l,  dz = ddelta GELU'(z),
//   dp_l = dz r_l,  dr_l = dr_{l+1} + dz p_l;  then dv += dr_1 and dh = -GELU'(h) dr_1.
template <typename io_t, int CPL, int RM>
__global__ void __launch_bounds__(NT) chain_grad_nl_kernel(const io_t *__restrict__ v, const io_t *__restrict__ v_hist,
                                                           const io_t *__restrict__ conv_w,
                                                           const float *__restrict__ gamma,
                                                           const io_t *__restrict__ p_gain,
                                                           const float *__restrict__ dX, float *__restrict__ dH,
                                                           float *__restrict__ dv_out, float *__restrict__ dgamma,
                                                           float *__restrict__ dp_gain, long long ntok, int H, int T,
                                                           int R)
{
    constexpr int dv = 64 * CPL;
    const int lane = threadIdx.x & 31;
    const long long tok = (long long)blockIdx.x * (NT / 32) + (threadIdx.x >> 5);
    if (tok >= ntok) return;
    const int bh = (int)(tok / T), t = (int)(tok % T), h = bh % H;
    float gm[RM];
#pragma unroll
    for (int l = 0; l < RM; ++l) gm[l] = l < R ? gamma[(size_t)tok * R + l] : 0.f;
    float2 vv[CPL][4], w[CPL][4], dxv[CPL][RM], pv[CPL][RM], dvo[CPL];
#pragma unroll
    for (int k = 0; k < CPL; ++k) {
        const int c = 2 * (lane + 32 * k);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            w[k][j] = ld2(conv_w + ((size_t)h * 4 + j) * dv + c);
            vv[k][j] = make_float2(0.f, 0.f);
            if (t - j >= 0) vv[k][j] = ld2(v + ((size_t)bh * T + t - j) * dv + c);
            else if (v_hist) vv[k][j] = ld2(v_hist + ((size_t)bh * 3 + 3 + t - j) * dv + c);
        }
#pragma unroll
        for (int l = 0; l < RM; ++l)
            if (l < R) {
                dxv[k][l] = *reinterpret_cast<const float2 *>(dX + ((size_t)tok * R + l) * dv + c);
                pv[k][l] = ld2(p_gain + ((size_t)tok * R + l) * dv + c);
            }
        dvo[k] = *reinterpret_cast<const float2 *>(dv_out + (size_t)tok * dv + c);
    }
    float dgam[RM];
#pragma unroll
    for (int l = 0; l < RM; ++l) dgam[l] = 0.f;
#pragma unroll
    for (int k = 0; k < CPL; ++k) {
        const int c = 2 * (lane + 32 * k);
        float drn2[2], dh2[2], dp2[RM][2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            float a = 0.f;
#pragma unroll
            for (int j = 0; j < 4; ++j) a = fmaf(e ? w[k][j].y : w[k][j].x, e ? vv[k][j].y : vv[k][j].x, a);
            float dx[RM], pl[RM], dp[RM];
#pragma unroll
            for (int l = 0; l < RM; ++l) {
                dx[l] = e ? dxv[k][l].y : dxv[k][l].x;
                pl[l] = e ? pv[k][l].y : pv[k][l].x;
            }
            chain_nl_channel<RM>(a, e ? vv[k][0].y : vv[k][0].x, gm, pl, dx, R, dgam, dp, drn2[e], dh2[e]);
#pragma unroll
            for (int l = 0; l < RM; ++l) dp2[l][e] = dp[l];
        }
        *reinterpret_cast<float2 *>(dv_out + (size_t)tok * dv + c) = make_float2(dvo[k].x + drn2[0], dvo[k].y + drn2[1]);
        *reinterpret_cast<float2 *>(dH + (size_t)tok * dv + c) = make_float2(dh2[0], dh2[1]);
#pragma unroll
        for (int l = 0; l < RM; ++l)
            if (l < R)
                *reinterpret_cast<float2 *>(dp_gain + ((size_t)tok * R + l) * dv + c) = make_float2(dp2[l][0], dp2[l][1]);
    }
#pragma unroll
    for (int l = 0; l < RM; ++l)
        if (l < R) {
            const float s1 = warp_sum(dgam[l]);
            if (lane == 0) dgamma[(size_t)tok * R + l] = s1;
        }
}

// The convolution backwards over tiles of CT tokens: v's share of dv, dv_hist (first tile)
// and the tile's sums for dconv_w -> dWp [BH][ntile][4][dv].  Thread (c, sub) walks the CSUB
// tokens of sub-tile sub for channel c (blockDim = dv x CT / CSUB); the sub-tiles' sums meet in
// shared memory in a fixed order.
constexpr int CSUB = 16;
template <typename io_t>
__global__ void __launch_bounds__(512) conv_grad_kernel(const io_t *__restrict__ v, const io_t *__restrict__ v_hist,
                                                        const io_t *__restrict__ conv_w, const float *__restrict__ dH,
                                                        float *__restrict__ dv_out, float *__restrict__ dv_hist,
                                                        float *__restrict__ dWp, int H, int T, int dv, int ntile)
{
    __shared__ float part[CT / CSUB][4][128];
    const int c = threadIdx.x % dv, sub = threadIdx.x / dv, bh = blockIdx.y, tile = blockIdx.x, h = bh % H;
    const int t0 = tile * CT + sub * CSUB, t1 = min(T, t0 + CSUB);
    float w[4], acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int j = 0; j < 4; ++j) w[j] = ldf(conv_w + ((size_t)h * 4 + j) * dv + c);
    const size_t base = (size_t)bh * T;
    auto vat = [&](int src) -> float {
        if (src >= 0) return ldf(v + (base + src) * dv + c);
        return v_hist ? ldf(v_hist + ((size_t)bh * 3 + 3 + src) * dv + c) : 0.f;
    };
    // the sub-tile's dH[t0 .. t0 + CSUB + 2], v[t0 - 3 .. t0 + CSUB - 1] and dv, all loaded before
    // the arithmetic (0 past the end; history or 0 before the start)
    float hs[CSUB + 3], vs[CSUB + 3], dvs[CSUB];
#pragma unroll
    for (int i = 0; i < CSUB + 3; ++i) {
        const int t = t0 + i;
        hs[i] = t < T ? dH[(base + t) * dv + c] : 0.f;
        vs[i] = (t0 < T && t - 3 < T) ? vat(t - 3) : 0.f;
    }
#pragma unroll
    for (int i = 0; i < CSUB; ++i) dvs[i] = t0 + i < T ? dv_out[(base + t0 + i) * dv + c] : 0.f;
#pragma unroll
    for (int i = 0; i < CSUB; ++i) {
        if (t0 + i >= t1) break;
        // token t = t0 + i: dv_t += sum_j w_j dH_{t+j};  dw_j += dH_t v_{t-j}
        const float s = fmaf(w[0], hs[i], fmaf(w[1], hs[i + 1], fmaf(w[2], hs[i + 2], w[3] * hs[i + 3])));
        dv_out[(base + t0 + i) * dv + c] = dvs[i] + s;
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[j] = fmaf(hs[i], vs[i + 3 - j], acc[j]);
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) part[sub][j][c] = acc[j];
    __syncthreads();
    if (sub == 0) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            float sum = part[0][j][c];
#pragma unroll
            for (int q = 1; q < CT / CSUB; ++q) sum += part[q][j][c];
            dWp[(((size_t)bh * ntile + tile) * 4 + j) * dv + c] = sum;
        }
        if (tile == 0 && dv_hist) {
            // slot s holds v_{s-3}, which enters h_t through tap j = t - s + 3 for t in [0, s]
            for (int s = 0; s < 3; ++s) {
                float g = 0.f;
                for (int t = 0; t <= s && t < T; ++t) g = fmaf(w[t - s + 3], dH[(base + t) * dv + c], g);
                dv_hist[((size_t)bh * 3 + s) * dv + c] = g;
            }
        }
    }
}

// The token-local tail in one pass for bf16 io and dv = 64: a block takes a tile of CT tokens.
// Its eight warps run the chain and gain backwards (as chain_grad_kernel / chain_grad_nl_kernel,
// lane c the channel pair 2c, 2c + 1) for the tile's tokens and the three after it, whose dH the
// transposed convolution needs; dH, the chain's share of dv and the tile's v stay in shared memory.
// Then thread (c, sub) takes channel c of sub-tile sub (CSUB tokens) through the convolution
// backwards as conv_grad_kernel does, in the same order of operations, and writes dv once.
constexpr int TAIL_NT = 256;
template <int RM, bool NL>
__global__ void __launch_bounds__(TAIL_NT) tail_kernel(const __nv_bfloat16 *__restrict__ v,
                                                       const __nv_bfloat16 *__restrict__ v_hist,
                                                       const __nv_bfloat16 *__restrict__ conv_w,
                                                       const float *__restrict__ gamma, const float *__restrict__ eta,
                                                       const __nv_bfloat16 *__restrict__ p_gain,
                                                       const float *__restrict__ dX, float *__restrict__ dv_out,
                                                       float *__restrict__ dgamma, float *__restrict__ deta,
                                                       float *__restrict__ dp_gain, float *__restrict__ dv_hist,
                                                       float *__restrict__ dWp, int H, int T, int R, int ntile)
{
    constexpr int D = 64, NTOK = CT + 3;
    static_assert(TAIL_NT == D * (CT / CSUB), "one thread per channel and sub-tile");
    __shared__ float dHs[NTOK][D];             // dH of tokens t0 .. t0 + CT + 2 (0 past the end)
    __shared__ float dvs[CT][D];               // dv with the chain's share
    __shared__ __nv_bfloat16 vs[CT + 3][D];    // v of tokens t0 - 3 .. t0 + CT - 1 (history or 0 before)
    __shared__ float part[CT / CSUB][4][D];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, tile = blockIdx.x, bh = blockIdx.y, h = bh % H;
    const int t0 = tile * CT;
    const size_t base = (size_t)bh * T;
    // dX and dv of the gradient kernel (launched behind it).  The weight reduction behind this kernel
    // is not let in early: its 1024-thread blocks would hold half of an SM's threads while they wait.
    prism::tc::grid_dependency_wait();
    auto vpair = [&](int t, int c) -> __nv_bfloat162 {  // v_t, channels c, c + 1 (history before 0)
        if (t >= 0) return *reinterpret_cast<const __nv_bfloat162 *>(v + (base + t) * D + c);
        if (v_hist) return *reinterpret_cast<const __nv_bfloat162 *>(v_hist + ((size_t)bh * 3 + 3 + t) * D + c);
        return __floats2bfloat162_rn(0.f, 0.f);
    };
    {
        const int c = 2 * lane;
        float2 w[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) w[j] = ld2(conv_w + ((size_t)h * 4 + j) * D + c);
        if (warp == 0) {
#pragma unroll
            for (int j = 0; j < 3; ++j) {  // the three tokens before the tile
                const int t = t0 - 3 + j;
                *reinterpret_cast<__nv_bfloat162 *>(&vs[j][c]) = t < T ? vpair(t, c) : __floats2bfloat162_rn(0.f, 0.f);
            }
        }
#pragma unroll 2
        for (int tau = warp; tau < NTOK; tau += TAIL_NT / 32) {
            const int t = t0 + tau;
            float2 dh = make_float2(0.f, 0.f);
            if (t < T) {
                const size_t tok = base + t;
                float gm[RM], et[RM];
                float2 vv[4], dxv[RM], pv[RM], dvo = make_float2(0.f, 0.f);
#pragma unroll
                for (int l = 0; l < RM; ++l) {
                    gm[l] = l < R ? gamma[tok * R + l] : 0.f;
                    et[l] = (!NL && l + 1 < R) ? eta[tok * R + l] : 0.f;
                    dxv[l] = l < R ? *reinterpret_cast<const float2 *>(dX + (tok * R + l) * D + c) : make_float2(0.f, 0.f);
                    pv[l] = (NL && l < R) ? ld2(p_gain + (tok * R + l) * D + c) : make_float2(0.f, 0.f);
                }
                __nv_bfloat162 v0 = vpair(t, c);
                vv[0] = __bfloat1622float2(v0);
#pragma unroll
                for (int j = 1; j < 4; ++j) vv[j] = __bfloat1622float2(vpair(t - j, c));
                if (tau < CT) dvo = *reinterpret_cast<const float2 *>(dv_out + tok * D + c);
                float dgam[RM], det[RM], drn2[2], dh2[2], dp2[RM][2];
#pragma unroll
                for (int l = 0; l < RM; ++l) dgam[l] = det[l] = 0.f;
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    float a = 0.f;
#pragma unroll
                    for (int j = 0; j < 4; ++j) a = fmaf(e ? w[j].y : w[j].x, e ? vv[j].y : vv[j].x, a);
                    float dx[RM];
#pragma unroll
                    for (int l = 0; l < RM; ++l) dx[l] = e ? dxv[l].y : dxv[l].x;
                    if constexpr (NL) {
                        float pl[RM], dp[RM];
#pragma unroll
                        for (int l = 0; l < RM; ++l) pl[l] = e ? pv[l].y : pv[l].x;
                        chain_nl_channel<RM>(a, e ? vv[0].y : vv[0].x, gm, pl, dx, R, dgam, dp, drn2[e], dh2[e]);
#pragma unroll
                        for (int l = 0; l < RM; ++l) dp2[l][e] = dp[l];
                    } else {
                        chain_lin_channel<RM>(a, e ? vv[0].y : vv[0].x, gm, et, dx, R, dgam, det, drn2[e], dh2[e]);
                    }
                }
                dh = make_float2(dh2[0], dh2[1]);
                if (tau < CT) {  // the tile's own tokens: dv's chain share, the gains' cotangents
                    *reinterpret_cast<float2 *>(&dvs[tau][c]) = make_float2(dvo.x + drn2[0], dvo.y + drn2[1]);
                    *reinterpret_cast<__nv_bfloat162 *>(&vs[tau + 3][c]) = v0;
                    if constexpr (NL) {
#pragma unroll
                        for (int l = 0; l < RM; ++l)
                            if (l < R)
                                *reinterpret_cast<float2 *>(dp_gain + (tok * R + l) * D + c) = make_float2(dp2[l][0], dp2[l][1]);
                    }
#pragma unroll
                    for (int l = 0; l < RM; ++l)
                        if (l < R) {
                            const float s1 = warp_sum(dgam[l]);
                            if (lane == 0) dgamma[tok * R + l] = s1;
                            if constexpr (!NL) {
                                const float s2 = warp_sum(det[l]);
                                if (lane == 0) deta[tok * R + l] = s2;
                            }
                        }
                }
            } else if (tau < CT) {
                *reinterpret_cast<__nv_bfloat162 *>(&vs[tau + 3][c]) = __floats2bfloat162_rn(0.f, 0.f);
            }
            *reinterpret_cast<float2 *>(&dHs[tau][c]) = dh;
        }
    }
    __syncthreads();
    // the convolution backwards: thread (c, sub), tokens t0 + CSUB sub ..
    const int c = tid % D, sub = tid / D, i0 = sub * CSUB;
    float w[4], acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int j = 0; j < 4; ++j) w[j] = __bfloat162float(conv_w[((size_t)h * 4 + j) * D + c]);
#pragma unroll
    for (int i = 0; i < CSUB; ++i) {
        const int tau = i0 + i;
        if (t0 + tau >= T) break;
        // token t: dv_t += sum_j w_j dH_{t+j};  dw_j += dH_t v_{t-j}
        const float s = fmaf(w[0], dHs[tau][c], fmaf(w[1], dHs[tau + 1][c], fmaf(w[2], dHs[tau + 2][c], w[3] * dHs[tau + 3][c])));
        dv_out[(base + t0 + tau) * D + c] = dvs[tau][c] + s;
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[j] = fmaf(dHs[tau][c], __bfloat162float(vs[tau + 3 - j][c]), acc[j]);
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) part[sub][j][c] = acc[j];
    __syncthreads();
    if (sub == 0) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            float sum = part[0][j][c];
#pragma unroll
            for (int q = 1; q < CT / CSUB; ++q) sum += part[q][j][c];
            dWp[(((size_t)bh * ntile + tile) * 4 + j) * D + c] = sum;
        }
        if (tile == 0 && dv_hist) {
            // slot s holds v_{s-3}, which enters h_t through tap j = t - s + 3 for t in [0, s]
            for (int s = 0; s < 3; ++s) {
                float g = 0.f;
                for (int t = 0; t <= s && t < T; ++t) g = fmaf(w[t - s + 3], dHs[t][c], g);
                dv_hist[((size_t)bh * 3 + s) * D + c] = g;
            }
        }
    }
}

// dconv_w[h][j][c] = sum over the batch and the tiles of dWp: a block takes 32 consecutive
// (h, j, c) outputs; its 32 warps take the (b, tile) terms e = warp, warp + 32, ... (lane =
// output), and the 32 partial sums meet in shared memory in a fixed order.
__global__ void __launch_bounds__(1024) conv_reduce_kernel(const float *__restrict__ dWp, float *__restrict__ dconv_w,
                                                           int B, int H, int dv, int ntile)
{
    __shared__ float part[32][33];
    const int lane = threadIdx.x & 31, wp = threadIdx.x >> 5;
    prism::tc::grid_dependency_wait();  // dWp (a no-op unless launched behind the kernel writing it)
    const int o = blockIdx.x * 32 + lane, nout = H * 4 * dv;
    float s = 0.f;
    if (o < nout) {
        const int h = o / (4 * dv), jc = o % (4 * dv);
        const int nterm = B * ntile;
        // the warp's terms e = wp, wp + 32, ... in batches of 16 whose loads are all in flight
        // before the first is added (the sum keeps the order of e)
        for (int e0 = wp; e0 < nterm; e0 += 32 * 16) {
            float x[16];
#pragma unroll
            for (int q = 0; q < 16; ++q) {
                const int e = e0 + 32 * q;
                const int b = e / ntile, tile = e % ntile;
                x[q] = e < nterm ? dWp[(((size_t)b * H + h) * ntile + tile) * 4 * dv + jc] : 0.f;
            }
#pragma unroll
            for (int q = 0; q < 16; ++q)
                if (e0 + 32 * q < nterm) s += x[q];
        }
    }
    part[wp][lane] = s;
    __syncthreads();
    if (wp == 0) {
        float sum = 0.f;
#pragma unroll
        for (int q = 0; q < 32; ++q) sum += part[q][lane];
        if (o < nout) dconv_w[o] = sum;
    }
}

struct Carve {
    float *X, *Sp, *Gs, *Z, *dX, *dH, *dWp;
};

size_t carve(const Shape &s, void *base, Carve *out)
{
    Carve scratch{};
    Carve *w = out ? out : &scratch;
    const size_t th = (size_t)s.BH * s.T;
    const int ntile = (s.T + CT - 1) / CT;
    const size_t n[7] = {th * s.R * s.dv, th * s.dv * s.dk, th * s.dv * s.dk, th * s.dv, th * s.R * s.dv,
                         th * s.dv, (size_t)s.BH * ntile * 4 * s.dv};
    float **dst[7] = {&w->X, &w->Sp, &w->Gs, &w->Z, &w->dX, &w->dH, &w->dWp};
    size_t off = 0;
    for (int i = 0; i < 7; ++i) {
        if (base) *dst[i] = reinterpret_cast<float *>(static_cast<char *>(base) + off);
        off += (n[i] * sizeof(float) + 255) & ~(size_t)255;
    }
    return off;
}

// The token-local tail of the backward, given dX (the cotangents of the injection factors) and dv
// holding beta z: the residual chain and gain backwards (dv, dgamma, deta, dH), then the
// convolution backwards (v's share of dv, dv_hist, dconv_w).
template <typename io_t>
cudaError_t token_local(const Shape &s, const BackwardArgs &a, float *dX, float *dH, float *dWp, KernelTimer &tm)
{
    cudaStream_t st = tm.stream;
    const io_t *v = static_cast<const io_t *>(a.v);
    const io_t *cw = static_cast<const io_t *>(a.conv_w), *vh = static_cast<const io_t *>(a.v_hist);
    const long long ntok = (long long)s.BH * s.T;
    const int ntile = (s.T + CT - 1) / CT;
    const long long cg_grid = (ntok + NT / 32 - 1) / (NT / 32);  // one warp per token
    if constexpr (std::is_same<io_t, __nv_bfloat16>::value) {
        if (s.dv == 64) {  // the fused tail: dH and the chain's share of dv stay on chip
            // launched behind the previous kernel (programmatic dependent launch): the blocks wait
            // for it in griddepcontrol.wait before they read what it wrote
            cudaLaunchAttribute pdl[1];
            pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
            pdl[0].val.programmaticStreamSerializationAllowed = 1;
            cudaLaunchConfig_t cfg = {};
            cfg.stream = st;
            cfg.attrs = pdl;
            cfg.numAttrs = 1;
            cfg.gridDim = dim3((unsigned)ntile, (unsigned)s.BH);
            cfg.blockDim = dim3(TAIL_NT);
            cudaError_t e;
            tm.begin("bwd_tail");
            if (a.p_gain) {
                auto kern = s.R <= 3 ? tail_kernel<3, true> : tail_kernel<RMAX, true>;
                e = cudaLaunchKernelEx(&cfg, kern, v, vh, cw, a.gamma, (const float *)nullptr,
                                       static_cast<const io_t *>(a.p_gain), (const float *)dX, a.dv, a.dgamma,
                                       (float *)nullptr, a.dp_gain, a.dv_hist, dWp, s.H, s.T, s.R, ntile);
            } else {
                auto kern = s.R <= 3 ? tail_kernel<3, false> : tail_kernel<RMAX, false>;
                e = cudaLaunchKernelEx(&cfg, kern, v, vh, cw, a.gamma, a.eta, (const io_t *)nullptr, (const float *)dX,
                                       a.dv, a.dgamma, a.deta, (float *)nullptr, a.dv_hist, dWp, s.H, s.T, s.R, ntile);
            }
            tm.end();
            if (e != cudaSuccess) return e;
            tm.begin("bwd_conv_reduce");
            cfg.gridDim = dim3((unsigned)((s.H * 4 * s.dv + 31) / 32));
            cfg.blockDim = dim3(1024);
            e = cudaLaunchKernelEx(&cfg, conv_reduce_kernel, (const float *)dWp, a.dconv_w, s.B, s.H, s.dv, ntile);
            tm.end();
            if (e != cudaSuccess) return e;
            return cudaGetLastError();
        }
    }
    tm.begin("bwd_chain_grad");
    // the level arrays sized for L <= 4 or for the largest L (registers)
    if (a.p_gain) {
        auto kern = s.dv == 64 ? (s.R <= 3 ? chain_grad_nl_kernel<io_t, 1, 3> : chain_grad_nl_kernel<io_t, 1, RMAX>)
                               : (s.R <= 3 ? chain_grad_nl_kernel<io_t, 2, 3> : chain_grad_nl_kernel<io_t, 2, RMAX>);
        kern<<<(unsigned)cg_grid, NT, 0, st>>>(v, vh, cw, a.gamma, static_cast<const io_t *>(a.p_gain), dX, dH, a.dv,
                                               a.dgamma, a.dp_gain, ntok, s.H, s.T, s.R);
    } else {
        auto kern = s.dv == 64 ? (s.R <= 3 ? chain_grad_kernel<io_t, 1, 3> : chain_grad_kernel<io_t, 1, RMAX>)
                               : (s.R <= 3 ? chain_grad_kernel<io_t, 2, 3> : chain_grad_kernel<io_t, 2, RMAX>);
        kern<<<(unsigned)cg_grid, NT, 0, st>>>(v, vh, cw, a.gamma, a.eta, dX, dH, a.dv, a.dgamma, a.deta, ntok, s.H,
                                               s.T, s.R);
    }
    tm.end();
    tm.begin("bwd_conv_grad");
    conv_grad_kernel<io_t><<<dim3(ntile, s.BH), s.dv * (CT / CSUB), 0, st>>>(v, vh, cw, dH, a.dv, a.dv_hist, dWp,
                                                                             s.H, s.T, s.dv, ntile);
    tm.end();
    tm.begin("bwd_conv_reduce");
    conv_reduce_kernel<<<(s.H * 4 * s.dv + 31) / 32, 1024, 0, st>>>(dWp, a.dconv_w, s.B, s.H, s.dv, ntile);
    tm.end();
    return cudaGetLastError();
}

template <typename io_t, int DK>
cudaError_t launch(const Shape &s, const BackwardArgs &a, void *ws, KernelTimer &tm)
{
    Carve w{};
    carve(s, ws, &w);
    cudaStream_t st = tm.stream;
    const io_t *q = static_cast<const io_t *>(a.q), *k = static_cast<const io_t *>(a.k);
    const io_t *v = static_cast<const io_t *>(a.v), *u = static_cast<const io_t *>(a.u);
    const io_t *cw = static_cast<const io_t *>(a.conv_w), *vh = static_cast<const io_t *>(a.v_hist);
    const long long ntok = (long long)s.BH * s.T;
    if (s.R > 0) {
        tm.begin("bwd_factors");
        factors_kernel<io_t><<<dim3((unsigned)(((long long)s.T * s.dv + NT - 1) / NT), s.BH), NT, 0, st>>>(
            v, vh, cw, a.gamma, a.eta, static_cast<const io_t *>(a.p_gain), w.X, s.H, s.T, s.dv, s.R);
        tm.end();
    }
    const int ct = scan_chunk(DK, s.R, sizeof(io_t));
    const size_t scan_smem = 2 * (size_t)stage_layout(ct, DK, s.R, sizeof(io_t)).bytes;
    tm.begin("bwd_scan");
    auto kern = scan_kernel<io_t, DK, -1>;
    switch (s.R) {
    case 0: kern = scan_kernel<io_t, DK, 0>; break;
    case 1: kern = scan_kernel<io_t, DK, 1>; break;
    case 2: kern = scan_kernel<io_t, DK, 2>; break;
    case 3: kern = scan_kernel<io_t, DK, 3>; break;
    case 4: kern = scan_kernel<io_t, DK, 4>; break;
    default: break;
    }
    kern<<<dim3(s.dv / ROWS, s.BH, 2), SCAN_WARPS * 32, scan_smem, st>>>(q, k, v, u, a.beta, a.alpha, w.X, a.S_init,
                                                                        a.dout, a.dS_final, w.Sp, w.Gs, w.Z, w.dX,
                                                                        a.dS_init, s.T, s.dv, s.R, ct);
    tm.end();
    const size_t smem = token_grad_smem_floats(DK, s.dv, s.R) * sizeof(float);
    const long long tg_grid = ntok < (1LL << 30) ? ntok : (1LL << 30);
    tm.begin("bwd_token_grad");
    token_grad_kernel<io_t, DK><<<(unsigned)tg_grid, NT, smem, st>>>(q, k, v, u, a.beta, a.alpha, w.X, w.Sp, w.Gs,
                                                                     w.Z, a.dout, a.dq, a.dk, a.dv, a.dbeta,
                                                                     a.dalpha, a.du, ntok, s.dv, s.R);
    tm.end();
    return token_local<io_t>(s, a, w.dX, w.dH, w.dWp, tm);
}

template <typename io_t, int DK>
cudaError_t set_smem()
{
    const size_t most = token_grad_smem_floats(DK, 128, RMAX) * sizeof(float);
    cudaError_t e =
        cudaFuncSetAttribute(token_grad_kernel<io_t, DK>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)most);
    if (e != cudaSuccess) return e;
    using scan_fn = decltype(&scan_kernel<io_t, DK, -1>);
    const scan_fn kerns[] = {scan_kernel<io_t, DK, -1>, scan_kernel<io_t, DK, 0>, scan_kernel<io_t, DK, 1>,
                             scan_kernel<io_t, DK, 2>, scan_kernel<io_t, DK, 3>, scan_kernel<io_t, DK, 4>};
    for (scan_fn kern : kerns)
        if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kScanSmem)) != cudaSuccess)
            return e;
    return cudaSuccess;
}

}  // namespace bwd

size_t backward_workspace_bytes(const Shape &s) { return bwd::carve(s, nullptr, nullptr); }

cudaError_t backward_prepare()
{
    cudaError_t e;
    if ((e = bwd::set_smem<float, 64>()) != cudaSuccess) return e;
    if ((e = bwd::set_smem<float, 128>()) != cudaSuccess) return e;
    if ((e = bwd::set_smem<__nv_bfloat16, 64>()) != cudaSuccess) return e;
    return bwd::set_smem<__nv_bfloat16, 128>();
}

cudaError_t backward(const Shape &s, prism_dtype io, const BackwardArgs &a, void *ws, KernelTimer &tm)
{
    if (io == PRISM_BF16)
        return s.dk == 64 ? bwd::launch<__nv_bfloat16, 64>(s, a, ws, tm) : bwd::launch<__nv_bfloat16, 128>(s, a, ws, tm);
    return s.dk == 64 ? bwd::launch<float, 64>(s, a, ws, tm) : bwd::launch<float, 128>(s, a, ws, tm);
}

int backward_conv_tiles(int T) { return (T + bwd::CT - 1) / bwd::CT; }

cudaError_t backward_token_local(const Shape &s, prism_dtype io, const BackwardArgs &a, float *dX, float *dH,
                                 float *dWp, KernelTimer &tm)
{
    return io == PRISM_BF16 ? bwd::token_local<__nv_bfloat16>(s, a, dX, dH, dWp, tm)
                            : bwd::token_local<float>(s, a, dX, dH, dWp, tm);
}

}  // namespace prism
