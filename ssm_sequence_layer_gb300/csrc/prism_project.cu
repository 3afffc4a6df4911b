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
// Two kernels.  anchor_kernel forms a = ShortConv(X) once, in bf16 (the tensor core's operand
// type), 8 channels per thread with 16-byte loads.  project_kernel computes a 128-token x
// 128-column tile of Y = a W^T: per 64-wide slice of D, TMA brings the slices of a and W
// (128-byte swizzled) into a ring of STAGES stages and one thread issues four tcgen05.mma
// (M = 128, N = 128, K = 16) into a 128-column fp32 accumulator in tensor memory.  The epilogue
// (each warp a 32-token lane quarter and one 64-column half) normalises the basis columns,
// applies the gate's logistic and scatters the results into the head-major layouts of the
// recurrence.  (Forming the anchor inside the product kernel repeats the convolution for every
// one of the N / 128 column tiles; measured, that made the product kernel instruction- and
// latency-bound.)  Every wait is bounded; an expired one is recorded in the status
// word and the CTA drains its copies and products before it releases tensor memory.
#include <cudaTypedefs.h>

#include "prism_project.h"
#include "tc_ptx.h"

namespace prism {
namespace proj {

using namespace prism::tc;

constexpr int PM = 128, PN = 128, PK = 64, STAGES = 3;
constexpr uint32_t TILE = PM * PK * 2;             // 16 KB: a 128 x 64 bf16 operand tile
constexpr uint32_t OFF_A = 0;                      // [STAGES] anchor tiles (SW128, by TMA)
constexpr uint32_t OFF_B = OFF_A + STAGES * TILE;  // [STAGES] W tiles (SW128, by TMA)
constexpr uint32_t SMEM = OFF_B + STAGES * TILE + 1024;  // + alignment slack: two CTAs per SM
static_assert(OFF_B % 1024 == 0 && 2 * SMEM <= 232448, "layout");

struct ProjParams {
    __nv_bfloat16 *u, *p;
    float *gamma;
    int *status;
    unsigned long long wait_ns;
    int T, D, H, R, dk, dv, N, tiles_t, tiles_bt;
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

// a[b][t][d] = sum_j conv[j][d] X[b][t - j][d] (zero before t = 0), 8 channels per thread
__global__ void __launch_bounds__(256) anchor_kernel(const __nv_bfloat16 *__restrict__ X,
                                                     const __nv_bfloat16 *__restrict__ conv,
                                                     __nv_bfloat16 *__restrict__ a, int T, int D, long long n8)
{
    const long long e = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (e >= n8) return;
    const int d8 = (int)(e % (D / 8)) * 8;
    const long long row = e / (D / 8);  // b T + t
    const int t = (int)(row % T);
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        if (t - j < 0) break;
        const uint4 xv = *reinterpret_cast<const uint4 *>(X + (row - j) * D + d8);
        const uint4 wv = *reinterpret_cast<const uint4 *>(conv + (size_t)j * D + d8);
        const __nv_bfloat162 *x2 = reinterpret_cast<const __nv_bfloat162 *>(&xv);
        const __nv_bfloat162 *w2 = reinterpret_cast<const __nv_bfloat162 *>(&wv);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const float2 xf = __bfloat1622float2(x2[q]), wf = __bfloat1622float2(w2[q]);
            acc[2 * q] = fmaf(wf.x, xf.x, acc[2 * q]);
            acc[2 * q + 1] = fmaf(wf.y, xf.y, acc[2 * q + 1]);
        }
    }
    *reinterpret_cast<uint4 *>(a + row * D + d8) =
        make_uint4(pack_bf2(acc[0], acc[1]), pack_bf2(acc[2], acc[3]), pack_bf2(acc[4], acc[5]), pack_bf2(acc[6], acc[7]));
}

// Persistent product kernel: a CTA takes tiles round-robin (token-tile major, so CTAs running at
// the same time share the anchor tile in L2).  Warp 0 (one thread) runs the main loop: TMA into
// the ring, four MMAs per K-step into one of two accumulators in tensor memory, a commit on the
// accumulator's "full" barrier after a tile's last step.  Warps 1-4 are the epilogue, one TMEM
// lane quarter each (token rows), all 128 columns per thread: they wait for an accumulator,
// drain it and release it on its "empty" barrier, so a tile's epilogue runs under the next
// tile's products.
constexpr int PTHREADS = 192;  // warp 0: products; warp 1: operand loads; warps 2-5: epilogue

__global__ void __launch_bounds__(PTHREADS, 2)
    project_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_w, ProjParams p)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    __shared__ uint32_t tmem_base_s;
    __shared__ __align__(8) uint64_t full[STAGES], mmad[STAGES], acc_full[2], acc_empty[2];
    __shared__ int abort_s;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int KS = p.D / PK;
    const int tiles_n = (p.N + PN - 1) / PN, ntiles = p.tiles_bt * tiles_n;
    const int my_tiles = ntiles > (int)blockIdx.x ? (ntiles - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
    const uint32_t sbase = smem_u32(sm);
    const uint64_t dbase = sdesc(sbase, 0, 0);
    const uint32_t idesc = idesc_bf16(PM, PN, 0, 0);

    if (tid == 0) {
        abort_s = 0;
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(smem_u32(&full[s]), 1);
            mbar_init(smem_u32(&mmad[s]), 1);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(smem_u32(&acc_full[s]), 1);
            mbar_init(smem_u32(&acc_empty[s]), 4);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        prefetch_tmap(&tm_a);
        prefetch_tmap(&tm_w);
    }
    if (warp == 0) tmem_alloc(smem_u32(&tmem_base_s), 2 * PN);
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tmem = tmem_base_s;

    // global step g = tile i * KS + ks uses stage g % STAGES.  Lane 0 of warp 1 refills a stage as
    // soon as the products that read it have completed; lane 0 of warp 0 issues the products as the
    // stages fill, so it never waits for a product before issuing the next.
    const int total = my_tiles * KS;
    auto tile_of = [&](int i, int &b, int &t0, int &n0) {
        const int tile = (int)blockIdx.x + i * (int)gridDim.x;
        const int bt = tile / tiles_n;
        n0 = (tile % tiles_n) * PN;
        b = bt / p.tiles_t;
        t0 = (bt % p.tiles_t) * PM;
    };
    int loads_issued = 0, mmas_issued = 0;  // the producers' counts (for the drain after an expired wait)
    if (tid == 32) {  // ---- operand loads ----
        for (int g = 0; g < total; ++g) {
            const int s = g % STAGES;
            if (g >= STAGES &&
                !mbar_wait(smem_u32(&mmad[s]), (uint32_t)((g / STAGES - 1) & 1), p.wait_ns)) {  // step g - STAGES read it
                abort_s = 1;
                atomicCAS(p.status, 0, kDevTimeout);
                break;
            }
            if (*(volatile int *)&abort_s) break;
            int b, t0, n0;
            tile_of(g / KS, b, t0, n0);
            const int ks = g % KS;
            const uint32_t mb = smem_u32(&full[s]);
            mbar_expect_tx(mb, 2 * TILE);
            tma_load_3d(sbase + OFF_A + s * TILE, &tm_a, mb, ks * PK, t0, b);
            asm volatile(
                "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], [%2];" ::"r"(
                    sbase + OFF_B + s * TILE),
                "l"((uint64_t)&tm_w), "r"(mb), "r"(ks * PK), "r"(n0)
                : "memory");
            loads_issued = g + 1;
        }
    } else if (tid == 0) {  // ---- products ----
        for (int g = 0; g < total; ++g) {
            const int i = g / KS, ks = g % KS, s = g % STAGES, buf = i & 1;
            bool ok = true;
            if (ks == 0 && i >= 2)  // the accumulator's previous tile (i - 2) has been drained
                ok = mbar_wait(smem_u32(&acc_empty[buf]), (uint32_t)(((i - 2) / 2) & 1), p.wait_ns);
            if (ok) ok = mbar_wait(smem_u32(&full[s]), (uint32_t)((g / STAGES) & 1), p.wait_ns);
            if (!ok) {
                abort_s = 1;
                atomicCAS(p.status, 0, kDevTimeout);
                break;
            }
            if (*(volatile int *)&abort_s) break;
            fence_after_sync();
#pragma unroll
            for (int j = 0; j < PK / 16; ++j)
                mma_f16(tmem + buf * PN, op_desc(dbase, OFF_A + s * TILE + j * 32), op_desc(dbase, OFF_B + s * TILE + j * 32),
                        idesc, (ks > 0 || j > 0) ? 1u : 0u);
            mma_commit(smem_u32(&mmad[s]));
            if (ks == KS - 1) mma_commit(smem_u32(&acc_full[buf]));  // the tile's products are in the accumulator
            mmas_issued = g + 1;
        }
    } else if (warp >= 2) {  // epilogue warps 2-5: lane quarter q = warp & 3
        const int q = warp & 3;
        const uint32_t lane_off = (uint32_t)(q * 32) << 16;
        const int NU = p.H * p.R * p.dk, NP = p.H * p.R * p.dv;
        for (int i = 0; i < my_tiles; ++i) {
            const int buf = i & 1;
            const bool done = mbar_wait(smem_u32(&acc_full[buf]), (uint32_t)((i / 2) & 1), p.wait_ns);
            if (!__all_sync(0xffffffffu, done)) {
                if (lane == 0) {
                    atomicCAS(p.status, 0, kDevTimeout);
                    abort_s = 1;  // the products of this tile may still be in flight: drain before the dealloc
                }
                break;
            }
            fence_after_sync();
            const int tile = (int)blockIdx.x + i * (int)gridDim.x;
            const int bt = tile / tiles_n, n0 = (tile % tiles_n) * PN;
            const int b = bt / p.tiles_t, t = (bt % p.tiles_t) * PM + q * 32 + lane;
            const bool live = t < p.T;
            const uint32_t acc = tmem + buf * PN + lane_off;
            float sq[2] = {0.f, 0.f};  // sums of squares of the two 64-column halves
            if (n0 < NU) {
#pragma unroll
                for (int ch = 0; ch < PN / 32; ++ch) {
                    float v[32];
                    tmem_ld(acc + (uint32_t)(32 * ch), v);
#pragma unroll
                    for (int e = 0; e < 32; ++e) sq[ch >> 1] = fmaf(v[e], v[e], sq[ch >> 1]);
                }
            }
#pragma unroll
            for (int ch = 0; ch < PN / 32; ++ch) {
                float v[32];
                tmem_ld(acc + (uint32_t)(32 * ch), v);
                const int n = n0 + 32 * ch;
                if (!live || n >= p.N) continue;
                if (n < NU) {  // basis: a group is one 64-column half (dk = 64) or the whole tile (dk = 128)
                    const int g = n / p.dk, c = n % p.dk;
                    const float gsq = (p.dk == 64) ? sq[ch >> 1] : sq[0] + sq[1];
                    const float f = gsq > 0.f ? rsqrtf(gsq) : 0.f;
                    __nv_bfloat16 *dst = p.u + ((((size_t)b * p.H + g / p.R) * p.T + t) * p.R + g % p.R) * p.dk + c;
                    uint4 *d4 = reinterpret_cast<uint4 *>(dst);
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        d4[e] = make_uint4(pack_bf2(v[8 * e] * f, v[8 * e + 1] * f), pack_bf2(v[8 * e + 2] * f, v[8 * e + 3] * f),
                                           pack_bf2(v[8 * e + 4] * f, v[8 * e + 5] * f),
                                           pack_bf2(v[8 * e + 6] * f, v[8 * e + 7] * f));
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
            fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&acc_empty[buf]));  // this quarter is done with the accumulator
        }
    }
    // drain: after an expired wait, the copies and products in flight land before the CTA exits
    __syncthreads();
    if (abort_s) {
        if (tid == 0 && mmas_issued > 0)  // the last product of each stage (products complete in order)
            (void)mbar_wait(smem_u32(&mmad[(mmas_issued - 1) % STAGES]), (uint32_t)(((mmas_issued - 1) / STAGES) & 1),
                            1000000000ull);
        if (tid == 32)  // the last load of each stage
            for (int g = max(0, loads_issued - STAGES); g < loads_issued; ++g)
                (void)mbar_wait(smem_u32(&full[g % STAGES]), (uint32_t)((g / STAGES) & 1), 1000000000ull);
    }
    fence_before_sync();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, 2 * PN);
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
    CUtensorMap ma, mw;
    {
        cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)s.T, (cuuint64_t)s.B};
        cuuint64_t str[2] = {(cuuint64_t)D * 2, (cuuint64_t)s.T * D * 2};
        cuuint32_t box[3] = {PK, PM, 1};
        if (!encode_bf16(&ma, a.anchor, 3, dims, str, box, CU_TENSOR_MAP_SWIZZLE_128B)) return cudaErrorInvalidValue;
    }
    {
        cuuint64_t dims[2] = {(cuuint64_t)D, (cuuint64_t)N};
        cuuint64_t str[1] = {(cuuint64_t)D * 2};
        cuuint32_t box[2] = {PK, PN};
        if (!encode_bf16(&mw, a.W, 2, dims, str, box, CU_TENSOR_MAP_SWIZZLE_128B)) return cudaErrorInvalidValue;
    }
    ProjParams p;
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
    p.tiles_bt = s.B * p.tiles_t;
    static int sms = 0;
    if (sms == 0) {
        int dev = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (sms <= 0) sms = 1;
    }
    const int ntiles = p.tiles_bt * ((N + PN - 1) / PN);
    const dim3 grid(ntiles < 2 * sms ? ntiles : 2 * sms);
    const long long n8 = (long long)s.B * s.T * (D / 8);
    tm.begin("anchor");
    anchor_kernel<<<(unsigned)((n8 + 255) / 256), 256, 0, tm.stream>>>((const __nv_bfloat16 *)a.X,
                                                                    (const __nv_bfloat16 *)a.conv,
                                                                    (__nv_bfloat16 *)a.anchor, s.T, D, n8);
    tm.end();
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    tm.begin("project");
    project_kernel<<<grid, PTHREADS, SMEM, tm.stream>>>(ma, mw, p);
    tm.end();
    return cudaGetLastError();
}

}  // namespace prism
