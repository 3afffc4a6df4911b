// State carried across calls: the convolution history of a sequence and the recurrent
// single-token step (decode).
//
// Recurrent form of the method, per (batch, head) and token (the notes on PRISM, section 2.2:
// the state update is an input-driven transition plus a rank-L write; section 2.3: the anchor is
// a causal four-tap convolution over v):
//   h = w_0 v + w_1 v_{-1} + w_2 v_{-2} + w_3 v_{-3},   g = GELU'(h),   e = v - GELU(h)
//   x_l = gamma_l g (.) r_l,   r_1 = e,   r_{l+1} = r_l (.) (1 - eta_l g)
//   S <- alpha (S - beta (S k) k^T) + beta v k^T + sum_l x_l u_l^T,      o = S q
// Row i of S (value channel i) depends only on channel i's scalars (v_i, g_i, r_{l,i}) and the
// head's vectors k, q, u_l, so a step is one pass over the state, row by row: read a row, two dot
// products, write it back.  The state dominates the traffic (2 dv dk 4 bytes per head and step),
// so the kernel is bound by HBM bandwidth; it reads and writes each row once with 16-byte
// accesses, a row spread over dk/4 lanes.
#include "prism_internal.h"

namespace prism {
namespace state {

__device__ __forceinline__ float ldf(const float *p) { return *p; }
__device__ __forceinline__ float ldf(const __nv_bfloat16 *p) { return __bfloat162float(*p); }
__device__ __forceinline__ void stf(float *p, float x) { *p = x; }
__device__ __forceinline__ void stf(__nv_bfloat16 *p, float x) { *p = __float2bfloat16_rn(x); }

// ---------------------------------------------------------------------------------------------
// history: out[bh][j] = token T - 3 + j of [v_hist; v] (v_hist = zeros when null).  One thread
// per (sequence, channel) reads its three values before writing them, so out may be v_hist.
template <typename io_t>
__global__ void history_kernel(const io_t *v_hist, const io_t *__restrict__ v, io_t *out, int T, int dv, long long n)
{
    const long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= n) return;
    const long long bh = idx / dv;
    const int c = (int)(idx % dv);
    io_t w[3];
#pragma unroll
    for (int j = 0; j < 3; ++j) {
        const int t = T - 3 + j;
        if (t >= 0)
            w[j] = v[((size_t)bh * T + t) * dv + c];
        else
            w[j] = v_hist ? v_hist[((size_t)bh * 3 + 3 + t) * dv + c] : io_t(0.f);
    }
#pragma unroll
    for (int j = 0; j < 3; ++j) out[((size_t)bh * 3 + j) * dv + c] = w[j];
}

// ---------------------------------------------------------------------------------------------
// decode: one token for every (batch, head).  Grid (BH, dv / DEC_ROWS): a CTA owns DEC_ROWS value
// channels of one head -- their rows of S and their entries of v_hist -- so the in-place updates
// of S and of the history never race.
constexpr int DEC_THREADS = 256;
constexpr int DEC_ROWS = 32;
constexpr int DEC_RMAX = 15;

struct DecodeParams {
    const void *q, *k, *v, *u, *conv_w;
    const float *beta, *alpha, *gamma, *eta;
    void *v_hist;  // [BH][3][dv] io, read and shifted by one token
    float *S;      // [BH][dv][dk] fp32, read and updated
    void *out;     // [BH][dv]
    int H, dv, R;
};

template <typename io_t, typename out_t, int DK>
__global__ void __launch_bounds__(DEC_THREADS) decode_kernel(const DecodeParams p)
{
    constexpr int LPR = DK / 4;                      // lanes per row, one float4 each
    constexpr int RPW = 32 / LPR;                    // rows per warp and pass
    constexpr int ROWS_W = DEC_ROWS / (DEC_THREADS / 32);
    constexpr int PASSES = ROWS_W / RPW;
    static_assert(PASSES * RPW * (DEC_THREADS / 32) == DEC_ROWS, "row split");
    __shared__ __align__(16) float vec[(2 + DEC_RMAX) * DK];  // k | q | u_1 .. u_R
    __shared__ float xs[DEC_RMAX][DEC_ROWS];                  // x_l of this CTA's channels
    __shared__ float bvs[DEC_ROWS];                           // beta v_i

    const int bh = blockIdx.x, r0 = blockIdx.y * DEC_ROWS, tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31, sub = lane / LPR, c4 = lane % LPR;
    const int h = bh % p.H, dv = p.dv, R = p.R;
    float *Sb = p.S + ((size_t)bh * dv + r0) * DK;

    // this thread's rows, loaded first so that their latency overlaps the set-up below
    float4 s[PASSES];
#pragma unroll
    for (int ps = 0; ps < PASSES; ++ps) {
        const int i = warp * ROWS_W + ps * RPW + sub;
        s[ps] = *reinterpret_cast<const float4 *>(Sb + (size_t)i * DK + 4 * c4);
    }
    const io_t *kq = reinterpret_cast<const io_t *>(p.k) + (size_t)bh * DK;
    const io_t *qq = reinterpret_cast<const io_t *>(p.q) + (size_t)bh * DK;
    const io_t *uq = reinterpret_cast<const io_t *>(p.u) + (size_t)bh * R * DK;
    for (int e = tid; e < (2 + R) * DK; e += DEC_THREADS)
        vec[e] = e < DK ? ldf(kq + e) : e < 2 * DK ? ldf(qq + e - DK) : ldf(uq + e - 2 * DK);
    const float be = p.beta[bh], al = p.alpha[bh];
    if (tid < DEC_ROWS) {  // channel scalars: anchor, gain, residual chain
        const int c = r0 + tid;
        const io_t *cw = reinterpret_cast<const io_t *>(p.conv_w) + (size_t)h * 4 * dv + c;
        io_t *hp = reinterpret_cast<io_t *>(p.v_hist) + (size_t)bh * 3 * dv + c;
        const io_t v0 = reinterpret_cast<const io_t *>(p.v)[(size_t)bh * dv + c];
        const io_t v3 = hp[0], v2 = hp[dv], v1 = hp[2 * dv];  // v_{-3}, v_{-2}, v_{-1}
        const float vc = ldf(&v0);
        float a = ldf(cw) * vc;
        a = fmaf(ldf(cw + dv), ldf(&v1), a);
        a = fmaf(ldf(cw + 2 * dv), ldf(&v2), a);
        a = fmaf(ldf(cw + 3 * dv), ldf(&v3), a);
        const float Phi = 0.5f * erfcf(-a * 0.70710678118654752f);
        const float phi = 0.39894228040143268f * expf(-0.5f * a * a);
        const float g = fmaf(a, phi, Phi);
        float r = vc - a * Phi;
        bvs[tid] = be * vc;
        const float *gm = p.gamma + (size_t)bh * R, *et = p.eta + (size_t)bh * R;
        for (int l = 0; l < R; ++l) {
            xs[l][tid] = gm[l] * g * r;
            if (l + 1 < R) r *= 1.f - et[l] * g;
        }
        hp[0] = v2;  // the history moves on by one token
        hp[dv] = v1;
        hp[2 * dv] = v0;
    }
    __syncthreads();

    const float4 k4 = *reinterpret_cast<const float4 *>(vec + 4 * c4);
    const float4 q4 = *reinterpret_cast<const float4 *>(vec + DK + 4 * c4);
    out_t *ob = reinterpret_cast<out_t *>(p.out) + (size_t)bh * dv + r0;
#pragma unroll
    for (int ps = 0; ps < PASSES; ++ps) {
        const int i = warp * ROWS_W + ps * RPW + sub;
        float4 x = s[ps];
        float sk = x.x * k4.x + x.y * k4.y + x.z * k4.z + x.w * k4.w;
#pragma unroll
        for (int off = LPR / 2; off > 0; off >>= 1) sk += __shfl_xor_sync(0xffffffffu, sk, off);
        const float ck = bvs[i] - al * be * sk;  // S <- al S + (beta v - al beta S k) k^T
        x.x = fmaf(al, x.x, ck * k4.x);
        x.y = fmaf(al, x.y, ck * k4.y);
        x.z = fmaf(al, x.z, ck * k4.z);
        x.w = fmaf(al, x.w, ck * k4.w);
        for (int l = 0; l < R; ++l) {
            const float4 u4 = *reinterpret_cast<const float4 *>(vec + (2 + l) * DK + 4 * c4);
            const float xl = xs[l][i];
            x.x = fmaf(xl, u4.x, x.x);
            x.y = fmaf(xl, u4.y, x.y);
            x.z = fmaf(xl, u4.z, x.z);
            x.w = fmaf(xl, u4.w, x.w);
        }
        float o = x.x * q4.x + x.y * q4.y + x.z * q4.z + x.w * q4.w;
#pragma unroll
        for (int off = LPR / 2; off > 0; off >>= 1) o += __shfl_xor_sync(0xffffffffu, o, off);
        *reinterpret_cast<float4 *>(Sb + (size_t)i * DK + 4 * c4) = x;
        if (c4 == 0) stf(ob + i, o);
    }
}

template <typename io_t, typename out_t>
cudaError_t decode_t(const Shape &s, const DecodeParams &p, cudaStream_t st)
{
    const dim3 grid(s.BH, s.dv / DEC_ROWS);
    if (s.dk == 64)
        decode_kernel<io_t, out_t, 64><<<grid, DEC_THREADS, 0, st>>>(p);
    else
        decode_kernel<io_t, out_t, 128><<<grid, DEC_THREADS, 0, st>>>(p);
    return cudaGetLastError();
}

}  // namespace state

cudaError_t launch_history(const Shape &s, prism_dtype io, const void *v_hist, const void *v, void *v_hist_out,
                           KernelTimer &tm)
{
    const long long n = (long long)s.BH * s.dv;
    const unsigned blocks = (unsigned)((n + 255) / 256);
    tm.begin("history");
    if (io == PRISM_BF16)
        state::history_kernel<__nv_bfloat16><<<blocks, 256, 0, tm.stream>>>(
            (const __nv_bfloat16 *)v_hist, (const __nv_bfloat16 *)v, (__nv_bfloat16 *)v_hist_out, s.T, s.dv, n);
    else
        state::history_kernel<float><<<blocks, 256, 0, tm.stream>>>((const float *)v_hist, (const float *)v,
                                                                    (float *)v_hist_out, s.T, s.dv, n);
    tm.end();
    return cudaGetLastError();
}

cudaError_t decode_step(const Shape &s, prism_dtype io, prism_dtype out, const DecodeArgs &a, KernelTimer &tm)
{
    state::DecodeParams p;
    p.q = a.q;
    p.k = a.k;
    p.v = a.v;
    p.u = a.u;
    p.conv_w = a.conv_w;
    p.beta = a.beta;
    p.alpha = a.alpha;
    p.gamma = a.gamma;
    p.eta = a.eta;
    p.v_hist = a.v_hist;
    p.S = a.S;
    p.out = a.out;
    p.H = s.H;
    p.dv = s.dv;
    p.R = s.R;
    tm.begin("decode");
    cudaError_t e;
    if (io == PRISM_BF16)
        e = out == PRISM_F32 ? state::decode_t<__nv_bfloat16, float>(s, p, tm.stream)
                             : state::decode_t<__nv_bfloat16, __nv_bfloat16>(s, p, tm.stream);
    else
        e = out == PRISM_F32 ? state::decode_t<float, float>(s, p, tm.stream)
                             : state::decode_t<float, __nv_bfloat16>(s, p, tm.stream);
    tm.end();
    return e;
}

}  // namespace prism
