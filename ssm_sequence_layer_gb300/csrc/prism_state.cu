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
// so the kernel is bound by HBM bandwidth: the state is read once by bulk copies (TMA) into a
// ring of shared-memory stages and written back once with 16-byte stores.
#include "prism_internal.h"
#include "tc_ptx.h"

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
// decode: one token for every (batch, head).  The state streams through shared memory: an item
// is a block of RB value rows of one head (16 KB of S) with what those rows need -- the head's
// k, q and u_l, the block's v, history and convolution taps, the head's gates.  A persistent CTA
// takes items round-robin through a ring of DEC_STAGES stages:
//   warp 8 (producer)   waits until a stage is free, then fills it: the gates with 4-byte
//                       cp.async (each lane's cp.async.mbarrier.arrive tracks them on the
//                       stage's barrier) and everything else with bulk copies (TMA).
//   warps 0-7           each owns RB/8 rows of every item: lanes 0..RB/8-1 compute the anchor,
//                       gain and residual chain of those rows' channels, then the rows are
//                       updated from shared memory, 8 lanes per row, and written back to HBM;
//                       the warp then releases the stage.  No CTA barrier is on this path.
// A CTA owns the rows and history entries of its items, so the in-place updates never race.
constexpr int DEC_CONSUMERS = 8;
constexpr int DEC_THREADS = 32 * (DEC_CONSUMERS + 1);
constexpr int DEC_STAGES = 3;
constexpr int DEC_RMAX = 15;

struct DecodeParams {
    const void *q, *k, *v, *u, *conv_w;
    const float *beta, *alpha, *gamma, *eta;
    void *v_hist;  // [BH][3][dv] io, read and shifted by one token
    float *S;      // [BH][dv][dk] fp32, read and updated
    void *out;     // [BH][dv]
    int *status;
    unsigned long long wait_ns;
    int H, dv, R, n_items;
};

// stage layout (bytes) for head size DK and io element size E
template <int DK, int E>
struct DecStage {
    static constexpr int RB = 16384 / (DK * 4);  // rows per item: 16 KB of fp32 state
    static constexpr int OFF_K = RB * DK * 4;
    static constexpr int OFF_Q = OFF_K + DK * E;
    static constexpr int OFF_U = OFF_Q + DK * E;
    static constexpr int OFF_V = OFF_U + DEC_RMAX * DK * E;
    static constexpr int OFF_H = OFF_V + RB * E;
    static constexpr int OFF_C = OFF_H + 3 * RB * E;
    static constexpr int OFF_G = OFF_C + 4 * RB * E;  // beta, alpha, gamma[R], eta[R] (fp32)
    static constexpr int BYTES = (OFF_G + (2 + 2 * DEC_RMAX) * 4 + 127) / 128 * 128;
    static_assert(OFF_H % 16 == 0 && OFF_C % 16 == 0 && OFF_V % 16 == 0, "bulk copy alignment");
};

// 4 consecutive io values from shared memory as floats
__device__ __forceinline__ float4 lds4(const float *p) { return *reinterpret_cast<const float4 *>(p); }
__device__ __forceinline__ float4 lds4(const __nv_bfloat16 *p)
{
    const uint2 w = *reinterpret_cast<const uint2 *>(p);
    const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&w.x));
    const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&w.y));
    return make_float4(a.x, a.y, b.x, b.y);
}
__device__ __forceinline__ float dot4(const float4 a, const float4 b)
{
    return fmaf(a.x, b.x, fmaf(a.y, b.y, fmaf(a.z, b.z, a.w * b.w)));
}

template <typename io_t, typename out_t, int DK>
__global__ void __launch_bounds__(DEC_THREADS) decode_kernel(const DecodeParams p)
{
    using St = DecStage<DK, (int)sizeof(io_t)>;
    constexpr int RB = St::RB, NJ = DK / 32, RW = RB / DEC_CONSUMERS, PASSES = RW / 4;
    static_assert(PASSES * 4 == RW, "rows per consumer warp");
    extern __shared__ __align__(128) uint8_t dsm[];
    __shared__ __align__(8) uint64_t full[DEC_STAGES], empty[DEC_STAGES];
    __shared__ float xw[DEC_CONSUMERS][DEC_RMAX][RW];  // x_l of each warp's rows
    __shared__ float bvw[DEC_CONSUMERS][RW];           // beta v of each warp's rows
    __shared__ int issued_s;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, sub = lane >> 3, c8 = lane & 7;
    const int dv = p.dv, nblk = dv / RB, R = p.R, G = gridDim.x;
    const int my_n = p.n_items > (int)blockIdx.x ? (p.n_items - 1 - (int)blockIdx.x) / G + 1 : 0;
    if (tid == 0) {
        for (int s = 0; s < DEC_STAGES; ++s) {
            tc::mbar_init(tc::smem_u32(&full[s]), 1);
            tc::mbar_init(tc::smem_u32(&empty[s]), DEC_CONSUMERS);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    int issued = 0;
    if (warp == DEC_CONSUMERS) {  // producer
        const uint32_t bytes = (RB * DK * 4) + (2 * DK + R * DK + 8 * RB) * (uint32_t)sizeof(io_t);
        for (int k = 0; k < my_n; ++k) {
            const int st = k % DEC_STAGES;
            if (k >= DEC_STAGES) {  // the consumers have released item k - DEC_STAGES
                bool ok = true;
                if (lane == 0) ok = tc::mbar_wait(tc::smem_u32(&empty[st]), (uint32_t)((k / DEC_STAGES - 1) & 1), p.wait_ns);
                if (!__shfl_sync(0xffffffffu, ok, 0)) {
                    if (lane == 0) atomicCAS(p.status, 0, kDevTimeout);
                    break;
                }
                tc::fence_async_smem();
            }
            const int it = (int)blockIdx.x + k * G, bh = it / nblk, r0 = (it % nblk) * RB, h = bh % p.H;
            uint8_t *dst = dsm + st * St::BYTES;
            const uint32_t mb = tc::smem_u32(&full[st]);
            if (lane < 2 + 2 * R) {
                const float *src = lane == 0 ? p.beta + bh
                                 : lane == 1 ? p.alpha + bh
                                 : lane < 2 + R ? p.gamma + (size_t)bh * R + (lane - 2)
                                                : p.eta + (size_t)bh * R + (lane - 2 - R);
                asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(tc::smem_u32(dst + St::OFF_G + lane * 4)),
                             "l"(src)
                             : "memory");
            }
            // raises the phase's pending count now and arrives when this lane's copies land; it
            // precedes lane 0's arrival below, so the phase cannot complete without the gates
            asm volatile("cp.async.mbarrier.arrive.shared::cta.b64 [%0];" ::"r"(mb) : "memory");
            __syncwarp();
            if (lane == 0) {
                const io_t *q = reinterpret_cast<const io_t *>(p.q), *kk = reinterpret_cast<const io_t *>(p.k);
                const io_t *u = reinterpret_cast<const io_t *>(p.u), *v = reinterpret_cast<const io_t *>(p.v);
                const io_t *hist = reinterpret_cast<const io_t *>(p.v_hist);
                const io_t *cw = reinterpret_cast<const io_t *>(p.conv_w);
                constexpr uint32_t E = sizeof(io_t);
                tc::mbar_expect_tx(mb, bytes);
                tc::bulk_load(tc::smem_u32(dst), p.S + ((size_t)bh * dv + r0) * DK, RB * DK * 4, mb);
                tc::bulk_load(tc::smem_u32(dst + St::OFF_K), kk + (size_t)bh * DK, DK * E, mb);
                tc::bulk_load(tc::smem_u32(dst + St::OFF_Q), q + (size_t)bh * DK, DK * E, mb);
                if (R > 0) tc::bulk_load(tc::smem_u32(dst + St::OFF_U), u + (size_t)bh * R * DK, R * DK * E, mb);
                tc::bulk_load(tc::smem_u32(dst + St::OFF_V), v + (size_t)bh * dv + r0, RB * E, mb);
                for (int j = 0; j < 3; ++j)
                    tc::bulk_load(tc::smem_u32(dst + St::OFF_H + j * RB * E), hist + ((size_t)bh * 3 + j) * dv + r0, RB * E, mb);
                for (int j = 0; j < 4; ++j)
                    tc::bulk_load(tc::smem_u32(dst + St::OFF_C + j * RB * E), cw + ((size_t)h * 4 + j) * dv + r0, RB * E, mb);
            }
            issued = k + 1;
        }
    } else {  // consumers
        for (int k = 0; k < my_n; ++k) {
            const int st = k % DEC_STAGES;
            const uint8_t *sb = dsm + st * St::BYTES;
            const bool landed = tc::mbar_wait(tc::smem_u32(&full[st]), (uint32_t)((k / DEC_STAGES) & 1), p.wait_ns);
            if (!__all_sync(0xffffffffu, landed)) {
                if (lane == 0) atomicCAS(p.status, 0, kDevTimeout);
                break;
            }
            const int it = (int)blockIdx.x + k * G, bh = it / nblk, r0 = (it % nblk) * RB;
            const float *gs = reinterpret_cast<const float *>(sb + St::OFF_G);
            const float be = gs[0], al = gs[1];
            if (lane < RW) {  // anchor, gain and residual chain of this warp's channels
                const int cl = warp * RW + lane;
                const io_t *vb = reinterpret_cast<const io_t *>(sb + St::OFF_V);
                const io_t *hb = reinterpret_cast<const io_t *>(sb + St::OFF_H);
                const io_t *cb = reinterpret_cast<const io_t *>(sb + St::OFF_C);
                const io_t v0 = vb[cl], v3 = hb[cl], v2 = hb[RB + cl], v1 = hb[2 * RB + cl];  // v, v_{-3}, v_{-2}, v_{-1}
                const float vc = ldf(&v0);
                float a = ldf(cb + cl) * vc;
                a = fmaf(ldf(cb + RB + cl), ldf(&v1), a);
                a = fmaf(ldf(cb + 2 * RB + cl), ldf(&v2), a);
                a = fmaf(ldf(cb + 3 * RB + cl), ldf(&v3), a);
                const float Phi = 0.5f * erfcf(-a * 0.70710678118654752f);
                const float phi = 0.39894228040143268f * expf(-0.5f * a * a);
                const float g = fmaf(a, phi, Phi);
                float r = vc - a * Phi;
                bvw[warp][lane] = be * vc;
                for (int l = 0; l < R; ++l) {
                    xw[warp][l][lane] = gs[2 + l] * g * r;
                    if (l + 1 < R) r *= 1.f - gs[2 + R + l] * g;
                }
                io_t *hp = reinterpret_cast<io_t *>(p.v_hist) + (size_t)bh * 3 * dv + r0 + cl;
                hp[0] = v2;  // the history moves on by one token
                hp[dv] = v1;
                hp[2 * dv] = v0;
            }
            __syncwarp();
            // row update, 8 lanes per row: lane c8 holds columns 4 c8 + 32 j, j < NJ
            const io_t *ks = reinterpret_cast<const io_t *>(sb + St::OFF_K);
            const io_t *qs = reinterpret_cast<const io_t *>(sb + St::OFF_Q);
            const io_t *us = reinterpret_cast<const io_t *>(sb + St::OFF_U);
            float4 k4[NJ], q4[NJ];
#pragma unroll
            for (int j = 0; j < NJ; ++j) {
                k4[j] = lds4(ks + 4 * c8 + 32 * j);
                q4[j] = lds4(qs + 4 * c8 + 32 * j);
            }
            const float *Ss = reinterpret_cast<const float *>(sb);
            float *Sg = p.S + ((size_t)bh * dv + r0) * DK;
            out_t *ob = reinterpret_cast<out_t *>(p.out) + (size_t)bh * dv + r0;
#pragma unroll
            for (int ps = 0; ps < PASSES; ++ps) {
                const int il = ps * 4 + sub, i = warp * RW + il;
                float4 x[NJ];
                float skp[NJ];
#pragma unroll
                for (int j = 0; j < NJ; ++j) {
                    x[j] = *reinterpret_cast<const float4 *>(Ss + i * DK + 4 * c8 + 32 * j);
                    skp[j] = dot4(x[j], k4[j]);
                }
                float sk = skp[0];
#pragma unroll
                for (int j = 1; j < NJ; ++j) sk += skp[j];
                sk += __shfl_xor_sync(0xffffffffu, sk, 4);
                sk += __shfl_xor_sync(0xffffffffu, sk, 2);
                sk += __shfl_xor_sync(0xffffffffu, sk, 1);
                const float ck = bvw[warp][il] - al * be * sk;  // S <- al S + (beta v - al beta S k) k^T
#pragma unroll
                for (int j = 0; j < NJ; ++j) {
                    x[j].x = fmaf(al, x[j].x, ck * k4[j].x);
                    x[j].y = fmaf(al, x[j].y, ck * k4[j].y);
                    x[j].z = fmaf(al, x[j].z, ck * k4[j].z);
                    x[j].w = fmaf(al, x[j].w, ck * k4[j].w);
                }
#pragma unroll 1
                for (int l = 0; l < R; ++l) {  // + sum_l x_l u_l^T
                    const float xl = xw[warp][l][il];
#pragma unroll
                    for (int j = 0; j < NJ; ++j) {
                        const float4 u4 = lds4(us + l * DK + 4 * c8 + 32 * j);
                        x[j].x = fmaf(xl, u4.x, x[j].x);
                        x[j].y = fmaf(xl, u4.y, x[j].y);
                        x[j].z = fmaf(xl, u4.z, x[j].z);
                        x[j].w = fmaf(xl, u4.w, x[j].w);
                    }
                }
                float op[NJ];
#pragma unroll
                for (int j = 0; j < NJ; ++j) {
                    op[j] = dot4(x[j], q4[j]);
                    *reinterpret_cast<float4 *>(Sg + (size_t)i * DK + 4 * c8 + 32 * j) = x[j];
                }
                float o = op[0];
#pragma unroll
                for (int j = 1; j < NJ; ++j) o += op[j];
                o += __shfl_xor_sync(0xffffffffu, o, 4);
                o += __shfl_xor_sync(0xffffffffu, o, 2);
                o += __shfl_xor_sync(0xffffffffu, o, 1);
                if (c8 == 0) stf(ob + i, o);
            }
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(tc::smem_u32(&empty[st]));
        }
    }
    // before the CTA exits: its gate copies and the last bulk copies of each stage have landed
    // (all of them in a normal run; bounded waits after an expired one)
    asm volatile("cp.async.wait_all;" ::: "memory");
    if (tid == 32 * DEC_CONSUMERS) issued_s = issued;
    __syncthreads();
    if (tid == 0)
        for (int j = issued_s - DEC_STAGES; j < issued_s; ++j)
            if (j >= 0) (void)tc::mbar_wait(tc::smem_u32(&full[j % DEC_STAGES]), (uint32_t)((j / DEC_STAGES) & 1), 1000000000ull);
}

template <typename io_t, typename out_t, int DK>
cudaError_t decode_launch(const Shape &s, DecodeParams p, int sm_count, cudaStream_t st)
{
    constexpr int smem = DEC_STAGES * DecStage<DK, (int)sizeof(io_t)>::BYTES;
    static int per_sm = -1;  // resident CTAs per SM (from the occupancy calculator, once)
    if (per_sm < 0) {
        cudaError_t e = cudaFuncSetAttribute(decode_kernel<io_t, out_t, DK>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        int n = 0;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, decode_kernel<io_t, out_t, DK>, DEC_THREADS, smem);
        if (e != cudaSuccess) return e;
        per_sm = n > 0 ? n : 1;
    }
    p.n_items = s.BH * (s.dv / DecStage<DK, (int)sizeof(io_t)>::RB);
    const int grid = p.n_items < per_sm * sm_count ? p.n_items : per_sm * sm_count;
    decode_kernel<io_t, out_t, DK><<<grid, DEC_THREADS, smem, st>>>(p);
    return cudaGetLastError();
}

template <typename io_t, typename out_t>
cudaError_t decode_t(const Shape &s, const DecodeParams &p, int sm_count, cudaStream_t st)
{
    return s.dk == 64 ? decode_launch<io_t, out_t, 64>(s, p, sm_count, st) : decode_launch<io_t, out_t, 128>(s, p, sm_count, st);
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

cudaError_t decode_step(const Shape &s, prism_dtype io, prism_dtype out, const DecodeArgs &a, int sm_count,
                        int *d_status, long long wait_ns, KernelTimer &tm)
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
    p.status = d_status;
    p.wait_ns = wait_ns > 0 ? (unsigned long long)wait_ns : 100000000ull;
    p.H = s.H;
    p.dv = s.dv;
    p.R = s.R;
    p.n_items = 0;
    tm.begin("decode");
    cudaError_t e;
    if (io == PRISM_BF16)
        e = out == PRISM_F32 ? state::decode_t<__nv_bfloat16, float>(s, p, sm_count, tm.stream)
                             : state::decode_t<__nv_bfloat16, __nv_bfloat16>(s, p, sm_count, tm.stream);
    else
        e = out == PRISM_F32 ? state::decode_t<float, float>(s, p, sm_count, tm.stream)
                             : state::decode_t<float, __nv_bfloat16>(s, p, sm_count, tm.stream);
    tm.end();
    return e;
}

}  // namespace prism
