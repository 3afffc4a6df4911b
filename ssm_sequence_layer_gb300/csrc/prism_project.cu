// Input projections of the PRISM block on the tensor cores (sm_103a: TMA + tcgen05).
//
// The reading notes on PRISM (section 2.3, "Input-Anchored Simulation") derive every
// state-independent quantity of the write path from one anchor: a short causal convolution over
// the layer input, followed per refinement level by three projections -- the basis k^(l), the gain
// p^(l) and the gate beta^(l).  Per batch b and token t (X [B,T,D]):
//   a_t = sum_{j=0..3} w_j (.) X_{t-j}                   (zero before t = 0)
//   Y   = a W^T,  W [N, D],  N = H R dk + H R dv + H R
//   u_{t,l} (h) = y / ||y|| over the dk columns of (h, l)  -> u     [B,H,T,R,dk]  bf16
//   p_{t,l} (h) = the dv columns of (h, l)                  -> p     [B,H,T,R,dv]  bf16
//   gamma_{t,l} (h) = sigmoid(column (h, l) of the gates)   -> gamma [B,H,T,R]     fp32
// which are the directions, gains and step gates the recurrence takes.
//
// One CTA computes a 128-token x 128-column tile of Y: per 64-wide slice of D, TMA brings the
// slice of X (with an 8-token halo, zero-filled before the sequence start) and of W; the threads
// form the anchor slice in shared memory (bf16, 128-byte swizzled: the tensor core's A operand);
// one thread issues four tcgen05.mma (M = 128, N = 128, K = 16) into a 128-column fp32
// accumulator in tensor memory.  Two stages: the next slice's copies overlap the current
// slice's convolution and products.  The epilogue (warps 0-3, one token row each) normalises
// the basis columns, applies the gate's logistic and scatters the results into the head-major
// layouts of the recurrence.  Every wait is bounded; an expired one is recorded in the status
// word and the CTA drains its copies and products before it releases tensor memory.
#include <cudaTypedefs.h>

#include "prism_project.h"
#include "tc_ptx.h"

namespace prism {
namespace proj {

using namespace prism::tc;

constexpr int PM = 128, PN = 128, PK = 64, THREADS = 256, STAGES = 2;
constexpr int XROWS = PM + 8;                    // 8-token halo (the window needs 3)
constexpr uint32_t TILE = PM * PK * 2;           // 16 KB: a 128 x 64 bf16 operand tile
constexpr uint32_t XBYTES = XROWS * PK * 2;      // 17 KB: the X slice, unswizzled rows of 128 B
constexpr uint32_t OFF_A = 0;                    // [STAGES] anchor tiles (SW128)
constexpr uint32_t OFF_B = OFF_A + STAGES * TILE;  // [STAGES] W tiles (SW128, by TMA)
constexpr uint32_t OFF_X = OFF_B + STAGES * TILE;  // [STAGES] X slices (by TMA)
constexpr uint32_t SMEM = OFF_X + STAGES * XBYTES + 1024;  // + alignment slack
static_assert(OFF_B % 1024 == 0 && OFF_X % 1024 == 0 && XBYTES % 128 == 0, "layout");

struct ProjParams {
    const __nv_bfloat16 *conv;  // [4][D]
    __nv_bfloat16 *u, *p;
    float *gamma;
    int *status;
    unsigned long long wait_ns;
    int T, D, H, R, dk, dv, N, tiles_t;
};

// K-major 128B-swizzled operand at byte offset off: 16-byte core-matrix rows, 1024-byte 8-row groups
__device__ __forceinline__ uint64_t op_desc(uint64_t base, uint32_t off)
{
    return base + (uint64_t)(off >> 4) + ((uint64_t)(16 >> 4) << 16) + ((uint64_t)(1024 >> 4) << 32);
}

__device__ __forceinline__ uint32_t pack_bf2(float a, float b)
{
    const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<const uint32_t *>(&h);
}

__global__ void __launch_bounds__(THREADS, 2)
    project_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_w, ProjParams p)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    __shared__ uint32_t tmem_base_s;
    __shared__ __align__(8) uint64_t full[STAGES], mmad[STAGES];
    __shared__ int abort_s;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int b = blockIdx.x / p.tiles_t, t0 = (blockIdx.x % p.tiles_t) * PM, n0 = blockIdx.y * PN;
    const int KS = p.D / PK;
    const uint32_t sbase = smem_u32(sm);
    const uint64_t dbase = sdesc(sbase, 0, 0);
    const uint32_t idesc = idesc_bf16(PM, PN, 0, 0);

    if (tid == 0) {
        abort_s = 0;
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(smem_u32(&full[s]), 1);
            mbar_init(smem_u32(&mmad[s]), 1);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        prefetch_tmap(&tm_x);
        prefetch_tmap(&tm_w);
    }
    if (warp == 0) tmem_alloc(smem_u32(&tmem_base_s), PN);
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tmem = tmem_base_s;

    // thread 0's view of the copies and products in flight, for the drain after an expired wait
    int loads_issued = 0, loads_waited = 0, mmas_issued = 0, mmas_waited = 0;
    auto issue = [&](int ks) {  // thread 0: the X and W slices of step ks into stage ks % STAGES
        const int s = ks % STAGES;
        const uint32_t mb = smem_u32(&full[s]);
        mbar_expect_tx(mb, XBYTES + TILE);
        tma_load_3d(sbase + OFF_X + s * XBYTES, &tm_x, mb, ks * PK, t0 - 8, b);
        asm volatile(
            "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], [%2];" ::"r"(
                sbase + OFF_B + s * TILE),
            "l"((uint64_t)&tm_w), "r"(mb), "r"(ks * PK), "r"(n0)
            : "memory");
        ++loads_issued;
    };
    if (tid == 0) issue(0);

    const int cp = tid & 31, rg = tid >> 5;  // convolution: column pair cp, rows rg + 8 r
    for (int ks = 0; ks < KS; ++ks) {
        const int s = ks % STAGES;
        if (tid == 0) {
            bool ok = true;
            if (ks + 1 < KS) {
                // stage s ^ 1 is free once the products of step ks - 1 have read it
                if (ks >= 1) {
                    ok = mbar_wait(smem_u32(&mmad[(ks - 1) % STAGES]), (uint32_t)(((ks - 1) / STAGES) & 1), p.wait_ns);
                    if (ok) ++mmas_waited;
                }
                if (ok) issue(ks + 1);
            }
            if (ok) {
                ok = mbar_wait(smem_u32(&full[s]), (uint32_t)((ks / STAGES) & 1), p.wait_ns);
                if (ok) ++loads_waited;
            }
            if (!ok) {
                abort_s = 1;
                atomicCAS(p.status, 0, kDevTimeout);
            }
        }
        __syncthreads();
        if (abort_s) break;
        // the anchor slice: A[i][c] = sum_j w_j[d0 + c] X[t0 + i - j][d0 + c]  (X row i + 8 - j of the slice)
        {
            const int d0 = ks * PK;
            const __nv_bfloat162 *cw = reinterpret_cast<const __nv_bfloat162 *>(p.conv + d0) + cp;
            const float2 w0 = __bfloat1622float2(cw[0]);
            const float2 w1 = __bfloat1622float2(cw[p.D / 2]);
            const float2 w2 = __bfloat1622float2(cw[2 * (p.D / 2)]);
            const float2 w3 = __bfloat1622float2(cw[3 * (p.D / 2)]);
            const __nv_bfloat162 *xs = reinterpret_cast<const __nv_bfloat162 *>(sm + OFF_X + s * XBYTES) + cp;
            uint8_t *A = sm + OFF_A + s * TILE;
#pragma unroll 4
            for (int r = 0; r < PM / 8; ++r) {
                const int i = rg + 8 * r;
                const float2 x0 = __bfloat1622float2(xs[(i + 8) * 32]);
                const float2 x1 = __bfloat1622float2(xs[(i + 7) * 32]);
                const float2 x2 = __bfloat1622float2(xs[(i + 6) * 32]);
                const float2 x3 = __bfloat1622float2(xs[(i + 5) * 32]);
                const float a0 = fmaf(w0.x, x0.x, fmaf(w1.x, x1.x, fmaf(w2.x, x2.x, w3.x * x3.x)));
                const float a1 = fmaf(w0.y, x0.y, fmaf(w1.y, x1.y, fmaf(w2.y, x2.y, w3.y * x3.y)));
                *reinterpret_cast<uint32_t *>(A + sw128(i, 2 * cp)) = pack_bf2(a0, a1);
            }
        }
        fence_async_smem();  // the anchor tile is read by the tensor core (async proxy)
        fence_before_sync();
        __syncthreads();
        if (tid == 0) {
            fence_after_sync();
#pragma unroll
            for (int j = 0; j < PK / 16; ++j)
                mma_f16(tmem, op_desc(dbase, OFF_A + s * TILE + j * 32), op_desc(dbase, OFF_B + s * TILE + j * 32), idesc,
                        (ks > 0 || j > 0) ? 1u : 0u);
            mma_commit(smem_u32(&mmad[s]));
            ++mmas_issued;
        }
    }
    // all products done (thread 0 waits for the last one), then the epilogue
    if (tid == 0 && !abort_s && mmas_issued > 0) {
        const int last = mmas_issued - 1;
        if (mbar_wait(smem_u32(&mmad[last % STAGES]), (uint32_t)((last / STAGES) & 1), p.wait_ns))
            mmas_waited = mmas_issued;
        else {
            abort_s = 1;
            atomicCAS(p.status, 0, kDevTimeout);
        }
    }
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    if (!abort_s && warp < 4) {
        const int i = warp * 32 + lane, t = t0 + i;
        const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
        const int NU = p.H * p.R * p.dk, NP = p.H * p.R * p.dv;
        const bool live = t < p.T;
        // sum of squares of each basis group in this tile (at most PN / 64 groups, 64-column aligned)
        float ss[PN / 64] = {0.f, 0.f};
        if (n0 < NU) {
#pragma unroll
            for (int ch = 0; ch < PN / 32; ++ch) {
                float v[32];
                tmem_ld(tmem + lane_off + (uint32_t)(32 * ch), v);
                float q = 0.f;
#pragma unroll
                for (int e = 0; e < 32; ++e) q = fmaf(v[e], v[e], q);
                ss[ch / 2] += q;
            }
        }
#pragma unroll
        for (int ch = 0; ch < PN / 32; ++ch) {
            float v[32];
            tmem_ld(tmem + lane_off + (uint32_t)(32 * ch), v);
            const int n = n0 + 32 * ch;
            if (!live || n >= p.N) continue;
            if (n < NU) {  // basis: scale by 1 / ||y|| of its (h, l) group
                const int g = n / p.dk, c = n % p.dk;
                // the group's columns in this tile: dk = 64 -> one 64-column half; dk = 128 -> the whole tile
                float q = (p.dk == 64) ? ss[ch / 2] : ss[0] + ss[1];
                const float f = q > 0.f ? rsqrtf(q) : 0.f;
                __nv_bfloat16 *dst = p.u + ((((size_t)b * p.H + g / p.R) * p.T + t) * p.R + g % p.R) * p.dk + c;
                uint4 *d4 = reinterpret_cast<uint4 *>(dst);
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    d4[e] = make_uint4(pack_bf2(v[8 * e] * f, v[8 * e + 1] * f), pack_bf2(v[8 * e + 2] * f, v[8 * e + 3] * f),
                                       pack_bf2(v[8 * e + 4] * f, v[8 * e + 5] * f), pack_bf2(v[8 * e + 6] * f, v[8 * e + 7] * f));
            } else if (n < NU + NP) {  // gain
                const int m = n - NU, g = m / p.dv, c = m % p.dv;
                __nv_bfloat16 *dst = p.p + ((((size_t)b * p.H + g / p.R) * p.T + t) * p.R + g % p.R) * p.dv + c;
                uint4 *d4 = reinterpret_cast<uint4 *>(dst);
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    d4[e] = make_uint4(pack_bf2(v[8 * e], v[8 * e + 1]), pack_bf2(v[8 * e + 2], v[8 * e + 3]),
                                       pack_bf2(v[8 * e + 4], v[8 * e + 5]), pack_bf2(v[8 * e + 6], v[8 * e + 7]));
            } else {  // gates: logistic, one column each
#pragma unroll
                for (int e = 0; e < 32; ++e) {
                    const int m = n + e - NU - NP;
                    if (n + e < p.N) {
                        const int h = m / p.R, l = m % p.R;
                        p.gamma[(((size_t)b * p.H + h) * p.T + t) * p.R + l] = 1.f / (1.f + __expf(-v[e]));
                    }
                }
            }
        }
    }
    // drain: after an expired wait, the copies and products in flight land before the CTA exits
    if (tid == 0 && abort_s) {
        for (int k = mmas_waited; k < mmas_issued; ++k)
            (void)mbar_wait(smem_u32(&mmad[k % STAGES]), (uint32_t)((k / STAGES) & 1), 1000000000ull);
        for (int k = loads_waited; k < loads_issued; ++k)
            (void)mbar_wait(smem_u32(&full[k % STAGES]), (uint32_t)((k / STAGES) & 1), 1000000000ull);
    }
    fence_before_sync();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, PN);
}

}  // namespace proj

namespace {
bool encode_bf16(CUtensorMap *m, const void *base, int rank, const cuuint64_t *dims, const cuuint64_t *strides,
                 const cuuint32_t *box, CUtensorMapSwizzle sw)
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return false;
        fn = (PFN_cuTensorMapEncodeTiled_v12000)ptr;
    }
    cuuint32_t es[5] = {1, 1, 1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, (cuuint32_t)rank, const_cast<void *>(base), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}
}  // namespace

cudaError_t project_prepare()
{
    return cudaFuncSetAttribute(proj::project_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)proj::SMEM);
}

cudaError_t project_forward(const Shape &s, int D, const ProjectArgs &a, int *d_status, long long wait_ns,
                            KernelTimer &tm)
{
    using namespace proj;
    const int N = s.H * s.R * (s.dk + s.dv + 1);
    CUtensorMap mx, mw;
    {
        cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)s.T, (cuuint64_t)s.B};
        cuuint64_t str[2] = {(cuuint64_t)D * 2, (cuuint64_t)s.T * D * 2};
        cuuint32_t box[3] = {PK, XROWS, 1};
        if (!encode_bf16(&mx, a.X, 3, dims, str, box, CU_TENSOR_MAP_SWIZZLE_NONE)) return cudaErrorInvalidValue;
    }
    {
        cuuint64_t dims[2] = {(cuuint64_t)D, (cuuint64_t)N};
        cuuint64_t str[1] = {(cuuint64_t)D * 2};
        cuuint32_t box[2] = {PK, PN};
        if (!encode_bf16(&mw, a.W, 2, dims, str, box, CU_TENSOR_MAP_SWIZZLE_128B)) return cudaErrorInvalidValue;
    }
    ProjParams p;
    p.conv = (const __nv_bfloat16 *)a.conv;
    p.u = (__nv_bfloat16 *)a.u;
    p.p = (__nv_bfloat16 *)a.p;
    p.gamma = a.gamma;
    p.status = d_status;
    p.wait_ns = wait_ns > 0 ? (unsigned long long)wait_ns : 100000000ull;
    p.T = s.T;
    p.D = D;
    p.H = s.H;
    p.R = s.R;
    p.dk = s.dk;
    p.dv = s.dv;
    p.N = N;
    p.tiles_t = (s.T + PM - 1) / PM;
    const dim3 grid(s.B * p.tiles_t, (N + PN - 1) / PN);
    tm.begin("project");
    project_kernel<<<grid, THREADS, SMEM, tm.stream>>>(mx, mw, p);
    tm.end();
    return cudaGetLastError();
}

}  // namespace prism
