// Chunked backward of the PRISM memory recurrence on the tensor cores (sm_103a: tcgen05 + TMA),
// for dk = dv = 64, 1 <= L <= 4, bf16 io.
//
// The two quantities the backward carries -- the state S_c entering chunk c and the cotangent G_c
// flowing into the chunk's last state from later tokens -- follow chunk-level affine recurrences
// with maps that depend on the chunk's inputs only (notes on PRISM, section 2.1: the associative
// A/B form of the state passing; section 2.2: the delta-rule transition alpha (I - beta k k^T),
// symmetric, so the cotangent runs through the transposed chunk map):
//     S_{c+1} = S_c A_c + B_c,          G_{c-1} = G_c A_c^T + Bbar_c.
// Four kernels:
//   maps   one CTA per chunk: the prep (anchor, gain, residual chain -> X), the Grams, the UT
//          solve, the WY factors and the maps A_c, A_c^T, B_c, Bbar_c (fp32); the factors the
//          gradient kernels reuse go to a per-chunk stash (fp16 tiles in their shared-memory image).
//   scan   per sequence, direction and 16 state rows: S_c for every chunk (forward) and G_c
//          (reverse), fp32 SIMT (rows of the state evolve independently).
//   grad   one CTA per chunk, two halves on one set of tiles: the delta-rule values Vt = U' - W
//          S_c^T, z = G_t k_t (Z = Z0 + Wbar G_c^T), the cotangents of the injection factors dX_l,
//          dbeta, dv = beta z and the per-token sum sigma_t = beta_t v_t.z_t + sum_l x_tl.dx_tl;
//          then the masked Grams J = (Vw dO^T) o Dbar, H = (Vw Z^T) o Dbar, the key side dk, du,
//          the query side dq and dalpha (alpha_t dalpha_t = <G_c, S_{c+1}> + the suffix sum over
//          the chunk of q.dq - sigma).
// The token-local chain, gain and convolution backwards then run as in the token-serial pass.
//
// Chunk algebra (local index i, j; lambda_i = sum_{m<=i} ln alpha_m; D_ij = e^{lambda_i - lambda_j};
// Gamma_i = e^{lambda_i}; colf_j = Gamma_63 / Gamma_j; Kw = [K; U_0; ..], Vw = [Vt; X_0; ..]):
//   Akk = (K K^T) o D (j < i),  Mku_l = (K U_l^T) o D (j < i),  P_l = (Q U_l^T) o D (j <= i)
//   T = (I + diag(beta) Akk)^{-1},  E0 = V - sum_l Mku_l X_l,  U' = T diag(beta) E0,
//   W = T diag(beta Gamma) K,  Z0 = T^T ((Q K^T) o D)^T dO,  Wbar = T^T diag(colf) K
//   A_c = Gamma_63 I - W^T diag(colf) K,  B_c = U'^T diag(colf) K + sum_l X_l^T diag(colf) U_l
//   Bbar_c = dO^T diag(Gamma) Q - Z0^T diag(beta Gamma) K
//   dX_l = diag(colf) U_l G^T + P_l^T dO - Mku_l^T diag(beta) Z
//   dKw = diag(colf) Vw G + J Q - H diag(beta) K,  dq = diag(Gamma) dO S + J^T Kw
//   dk = dKw_0 - diag(beta) (diag(Gamma) Z S + H^T Kw),  dbeta = rowsum(Z o (E - Akk Vt)),
//   E = E0 - diag(Gamma) K S^T
// Every product is a tcgen05.mma (kind::f16, M = 128: two 64-row operands stacked, or one with the
// upper rows unused; fp32 accumulators in tensor memory).  The Grams of the maps kernel run on the
// bf16 input tiles; every other product on fp16 operands, the gradient kernels' input tiles
// converted in place (exact for bf16 values within the fp16 range).  Decay factors are all <= 1
// and applied in fp32 before an operand is rounded.
#include <cuda_fp16.h>
#include <cudaTypedefs.h>

#include "prism_internal.h"
#include "tc_ptx.h"
#include "tc_util.h"

namespace prism {
namespace bt {

using namespace tc;
using tcu::dsc;
using tcu::pack_h2;
using tcu::set_status;
using tcu::st_row_h;

constexpr int C = kChunk;
constexpr int D = 64;                 // dk = dv
constexpr int RMAX = 3;               // levels handled (L <= 4)
constexpr int NT = 512;               // threads of the per-chunk kernels: 16 warps, four per TMEM lane quarter
constexpr int CW = 64 / (NT / 128);   // columns of a 64-column accumulator block each thread handles
constexpr int SCAN_NT = 256;          // threads of the scan
constexpr uint32_t PANEL = 8192;      // [64 rows][64 cols] 16-bit SW128
constexpr int STASH = 8;              // stash panels per chunk (maps kernel): U', W, Wbar, Z0, E0, X_0..X_2
enum { ST_UP = 0, ST_W = 1, ST_WB = 2, ST_Z0 = 3, ST_E0 = 4, ST_X = 5 };

// per-token scalars (floats from the scalar region): beta, lambda, Gamma, colf, beta Gamma, gamma, eta
constexpr int SC_BETA = 0, SC_LAM = 64, SC_GAM = 128, SC_COLF = 192, SC_BG = 256, SC_GM = 320,
              SC_ET = 320 + 64 * RMAX, SC_HALO = 320 + 128 * RMAX, SC_RED = SC_HALO + 3 * D;
constexpr int SC_FLOATS = SC_RED + 24 * 64 + 32;  // + per-token partial sums (fixed slots, summed in a fixed order)

struct Params {
    const __nv_bfloat16 *v;          // [BH][T][64]
    const __nv_bfloat16 *conv_w;     // [H][4][64]
    const __nv_bfloat16 *v_hist;     // [BH][3][64] or null
    const float *beta, *alpha, *gamma, *eta;
    const __nv_bfloat16 *p_gain;     // [BH][T][R][64] (the non-linear chain) or null
    const float *dout;               // [BH][T][64]
    float *mapA, *mapAT, *mapB, *mapBb;  // [chunks][64][64]
    __half *stash;                   // [chunks][STASH][4096]
    const float *Sst;                // [BH][NC + 1][64][64]  state entering each chunk (and the final one)
    const float *Gst;                // [BH][NC][64][64]      cotangent flowing into each chunk's last state
    float *dq, *dk, *dv, *dbeta, *dalpha, *du;
    float *dX;                       // [BH T][R][64]
    int *status;
    int H, T, R, NC;
    unsigned long long wait_ns;
};

// ---- small helpers ---------------------------------------------------------------------------------
// barrier over `n` threads (whole warps; id >= 1)
__device__ __forceinline__ void named_bar(int id, int n) { asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory"); }

// barrier over `n` threads (whole warps; id >= 1) that returns whether any of them passed `flag`
__device__ __forceinline__ bool named_bar_or(int id, int n, bool flag)
{
    uint32_t any;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 q, %1, 0;\n\tbar.red.or.pred p, %2, %3, q;\n\tselp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(any)
        : "r"((uint32_t)flag), "r"(id), "r"(n)
        : "memory");
    return any != 0;
}

__device__ __forceinline__ uint64_t km(uint64_t dbase, uint32_t off) { return dsc(dbase, off, 16, 1024); }
__device__ __forceinline__ uint64_t mn(uint64_t dbase, uint32_t off, uint32_t lbo) { return dsc(dbase, off, lbo, 1024); }

// D (M = 128, N) [+]= A B over K = 64 (four steps of 16): a K-major operand advances 32 bytes per
// step, an MN-major one 2048 (16 rows of 128 bytes)
__device__ __forceinline__ void mma_k64(uint32_t d, uint64_t a, bool a_mn, uint64_t b, bool b_mn, uint32_t id, bool acc)
{
#pragma unroll
    for (int s = 0; s < 4; ++s)
        mma_f16(d, a + (uint64_t)((a_mn ? 2048u : 32u) * s >> 4), b + (uint64_t)((b_mn ? 2048u : 32u) * s >> 4), id,
                (acc || s > 0) ? 1u : 0u);
}

// N halves of row `row`, columns col0 .. col0 + N - 1, of an SW128 panel image (shared or global)
template <int N>
__device__ __forceinline__ void ld_row_h(const uint8_t *panel, int row, int col0, float (&v)[N])
{
#pragma unroll
    for (int g = 0; g < N / 8; ++g) {
        const uint4 w = *reinterpret_cast<const uint4 *>(panel + sw128(row, col0 + 8 * g));
        const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int h = 0; h < 4; ++h) {
            const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&ww[h]));
            v[8 * g + 2 * h] = f.x;
            v[8 * g + 2 * h + 1] = f.y;
        }
    }
}

// the raw 16-byte groups of the same row segment (issued early, converted later by h8_to_f)
template <int G>
__device__ __forceinline__ void ld_row_raw(const uint8_t *panel, int row, int col0, uint4 (&w)[G])
{
#pragma unroll
    for (int g = 0; g < G; ++g) w[g] = *reinterpret_cast<const uint4 *>(panel + sw128(row, col0 + 8 * g));
}

template <int G>
__device__ __forceinline__ void h8_to_f(const uint4 (&w)[G], float (&v)[8 * G])
{
#pragma unroll
    for (int g = 0; g < G; ++g) {
        const uint32_t ww[4] = {w[g].x, w[g].y, w[g].z, w[g].w};
#pragma unroll
        for (int h = 0; h < 4; ++h) {
            const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&ww[h]));
            v[8 * g + 2 * h] = f.x;
            v[8 * g + 2 * h + 1] = f.y;
        }
    }
}

// the same from a bf16 panel (TMA image)
template <int N>
__device__ __forceinline__ void ld_row_b(const uint8_t *panel, int row, int col0, float (&v)[N])
{
#pragma unroll
    for (int g = 0; g < N / 8; ++g) {
        const uint4 w = *reinterpret_cast<const uint4 *>(panel + sw128(row, col0 + 8 * g));
        const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int h = 0; h < 4; ++h) {
            const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&ww[h]));
            v[8 * g + 2 * h] = f.x;
            v[8 * g + 2 * h + 1] = f.y;
        }
    }
}

// a bf16 panel (as TMA wrote it) -> fp16 in place; with `copy`, also a copy whose row r is scaled
// by scale[r] (a 16-byte granule at physical offset 128 r + 16 g belongs to row r, whatever column
// group the swizzle put there)
__device__ __forceinline__ void panel_to_f16(uint8_t *panel, uint8_t *copy, const float *scale, float sgn, int tid)
{
    for (int e = tid; e < 512; e += NT) {
        const int r = e >> 3;
        uint4 *p = reinterpret_cast<uint4 *>(panel + 16 * e);
        const uint4 w = *p;
        const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
        float f[8];
#pragma unroll
        for (int h = 0; h < 4; ++h) {
            const float2 x = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&ww[h]));
            f[2 * h] = x.x;
            f[2 * h + 1] = x.y;
        }
        uint4 o;
        o.x = pack_h2(f[0], f[1]);
        o.y = pack_h2(f[2], f[3]);
        o.z = pack_h2(f[4], f[5]);
        o.w = pack_h2(f[6], f[7]);
        *p = o;
        if (copy) {
            const float s = sgn * scale[r];
            o.x = pack_h2(s * f[0], s * f[1]);
            o.y = pack_h2(s * f[2], s * f[3]);
            o.z = pack_h2(s * f[4], s * f[5]);
            o.w = pack_h2(s * f[6], s * f[7]);
            *reinterpret_cast<uint4 *>(copy + 16 * e) = o;
        }
    }
}

// an fp16 panel scaled in place, row r by scale[r]
__device__ __forceinline__ void panel_scale(uint8_t *panel, const float *scale, int tid)
{
    for (int e = tid; e < 512; e += NT) {
        const float s = scale[e >> 3];
        uint4 *p = reinterpret_cast<uint4 *>(panel + 16 * e);
        uint4 w = *p;
        uint32_t *ww = reinterpret_cast<uint32_t *>(&w);
#pragma unroll
        for (int h = 0; h < 4; ++h) {
            const float2 x = __half22float2(*reinterpret_cast<const __half2 *>(&ww[h]));
            ww[h] = pack_h2(s * x.x, s * x.y);
        }
        *p = w;
    }
}

// per-token scalars of one chunk (n tokens from tok0; the rest identity tokens: beta = 0,
// alpha = 1, gamma = eta = 0): warp 0 the gates and the inclusive scan of ln alpha, the other
// warps gamma and eta (eta of the last level is never read)
__device__ __forceinline__ void load_scalars(float *sc, const Params &p, size_t tok0, int n, int tid)
{
    const int warp = tid >> 5, lane = tid & 31, R = p.R;
    if (warp == 0) {
        const int i0 = 2 * lane, i1 = i0 + 1;
        const float b0 = i0 < n ? p.beta[tok0 + i0] : 0.f, b1 = i1 < n ? p.beta[tok0 + i1] : 0.f;
        const float la0 = i0 < n ? logf(p.alpha[tok0 + i0]) : 0.f, la1 = i1 < n ? logf(p.alpha[tok0 + i1]) : 0.f;
        float s = la0 + la1;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const float y = __shfl_up_sync(0xffffffffu, s, off);
            if (lane >= off) s += y;
        }
        const float l1 = s, l0 = s - la1, lc = __shfl_sync(0xffffffffu, s, 31);
        sc[SC_BETA + i0] = b0;
        sc[SC_BETA + i1] = b1;
        sc[SC_LAM + i0] = l0;
        sc[SC_LAM + i1] = l1;
        sc[SC_GAM + i0] = __expf(l0);
        sc[SC_GAM + i1] = __expf(l1);
        sc[SC_COLF + i0] = __expf(lc - l0);
        sc[SC_COLF + i1] = __expf(lc - l1);
        sc[SC_BG + i0] = b0 * __expf(l0);
        sc[SC_BG + i1] = b1 * __expf(l1);
    } else {
        for (int e = tid - 32; e < 64 * RMAX; e += NT - 32) {
            const int i = e / RMAX, l = e % RMAX;
            const bool ok = i < n && l < R;
            sc[SC_GM + e] = ok ? p.gamma[(tok0 + i) * R + l] : 0.f;
            sc[SC_ET + e] = (ok && l + 1 < R && p.eta) ? p.eta[(tok0 + i) * R + l] : 0.f;
        }
    }
}

// decayed, masked scores of row i, columns j0 .. j0 + N - 1: v[q] *= D_{i, j} for j <= i (incl) or
// j < i; 0 elsewhere
// The pair decay D_{i,j} = e^{lambda_i - lambda_j} of the kept elements: while the chunk's total
// decay keeps the per-token factors in fp32 range (-lambda_63 <= 80, the usual case) as a product
// of two factors from the scalar region (Gamma = e^lambda, colf = e^{lambda_63 - lambda}), else one
// exponential per element.  `lam` is the scalar region's lambda row.
template <int N>
__device__ __forceinline__ void decay_row(float (&v)[N], const float *lam, int i, int j0, bool incl)
{
    const float *gam = lam + (SC_GAM - SC_LAM), *colf = lam + (SC_COLF - SC_LAM);
    if (-lam[63] <= 80.f) {
        const float ri = gam[i] / gam[63];  // e^{lambda_i - lambda_63}
#pragma unroll
        for (int q = 0; q < N; ++q) {
            const int j = j0 + q;
            const bool keep = incl ? j <= i : j < i;
            v[q] = keep ? v[q] * (ri * colf[j]) : 0.f;
        }
        return;
    }
    const float li = lam[i];
#pragma unroll
    for (int q = 0; q < N; ++q) {
        const int j = j0 + q;
        const bool keep = incl ? j <= i : j < i;
        v[q] = keep ? v[q] * __expf(fminf(li - lam[j], 0.f)) : 0.f;
    }
}

// the transposed mask: v[q] (row m, column j = j0 + q) *= D_{j, m} for j >= m (incl) or j > m
template <int N>
__device__ __forceinline__ void decay_col(float (&v)[N], const float *lam, int m, int j0, bool incl)
{
    const float *gam = lam + (SC_GAM - SC_LAM), *colf = lam + (SC_COLF - SC_LAM);
    if (-lam[63] <= 80.f) {
        const float cm = colf[m] / gam[63];  // e^{-lambda_m}
#pragma unroll
        for (int q = 0; q < N; ++q) {
            const int j = j0 + q;
            const bool keep = incl ? j >= m : j > m;
            v[q] = keep ? v[q] * (gam[j] * cm) : 0.f;
        }
        return;
    }
    const float lm = lam[m];
#pragma unroll
    for (int q = 0; q < N; ++q) {
        const int j = j0 + q;
        const bool keep = incl ? j >= m : j > m;
        v[q] = keep ? v[q] * __expf(fminf(lam[j] - lm, 0.f)) : 0.f;
    }
}

template <int N>
__device__ __forceinline__ void st_row_f(float *dst, const float (&v)[N])
{
#pragma unroll
    for (int g = 0; g < N / 4; ++g)
        reinterpret_cast<float4 *>(dst)[g] = make_float4(v[4 * g], v[4 * g + 1], v[4 * g + 2], v[4 * g + 3]);
}

// An fp32 [64][64] output tile staged for TMA stores: two panels (columns 0-31 and 32-63), each 64
// rows of 128 B in the 128B-swizzled layout of the fp32 output tensor maps' boxes.  A row's 16
// columns from n0 (a multiple of 16) are four 16-byte granules; the rows of a warp hit distinct
// banks.
__device__ __forceinline__ uint32_t tile_f_off(int row, int col)
{
    return (uint32_t)(col >> 5) * PANEL + sw128(row, 2 * (col & 31));
}
__device__ __forceinline__ void st_tile_f(uint8_t *tile, int row, int n0, const float (&v)[16])
{
#pragma unroll
    for (int g = 0; g < 4; ++g)
        *reinterpret_cast<float4 *>(tile + tile_f_off(row, n0 + 4 * g)) =
            make_float4(v[4 * g], v[4 * g + 1], v[4 * g + 2], v[4 * g + 3]);
}
__device__ __forceinline__ void ld_tile_f(const uint8_t *tile, int row, int n0, float (&v)[16])
{
#pragma unroll
    for (int g = 0; g < 4; ++g) {
        const float4 f = *reinterpret_cast<const float4 *>(tile + tile_f_off(row, n0 + 4 * g));
        v[4 * g] = f.x;
        v[4 * g + 1] = f.y;
        v[4 * g + 2] = f.z;
        v[4 * g + 3] = f.w;
    }
}
__device__ __forceinline__ void tma_store_4d(const CUtensorMap *map, uint32_t src, int c0, int c1, int c2, int c3)
{
    asm volatile("cp.async.bulk.tensor.4d.global.shared::cta.bulk_group [%0, {%2, %3, %4, %5}], [%1];" ::"l"(
                     (uint64_t)map),
                 "r"(src), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
                 : "memory");
}

// untiled bulk copy shared -> global (bulk-group completion); both addresses 16-byte aligned, bytes
// a multiple of 16
__device__ __forceinline__ void bulk_store(void *dst, uint32_t src, uint32_t bytes)
{
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst), "r"(src), "r"(bytes)
                 : "memory");
}

// =====================================================================================================
// maps kernel: shared-memory panels (index x PANEL from a 1024-aligned base)
namespace mk {
enum {
    Q = 0, K = 1, U0 = 2, V = 5, ZERO = 6, X0 = 7, DO = 10, Z0 = 11, MKU0 = 12, PK = 15, TF = 16, W = 17, UP = 18,
    F = 19,  // solve region (A, T fp32 + scratch), then:
    BE = 19, BGK = 20, Y = 21, CK = 22, NBGK = 23, NPANELS = 24,
    // the fp32 maps staged for their TMA stores once the last products have read these tiles (none
    // of them is the source of a stash copy): A_c, A_c^T, B_c, Bbar_c
    MA = 12, MAT = 14, MB = 19, MBB = 21
};
// later tenants: colf U_l in MKU0 + l (after the E product), Gamma Q in PK (after the Y product)
constexpr uint32_t SC_OFF = NPANELS * PANEL;
constexpr uint32_t SMEM = SC_OFF + SC_FLOATS * 4 + 1024;
static_assert(2 * 64 * tcu::LDA * 4 + tcu::SOLVE_SCRATCH * 4 <= 5 * PANEL, "solve region");
static_assert(MA == MKU0 && MAT == MKU0 + 2 && MAT + 1 == PK && MB == BE && MBB == Y && MBB + 1 == CK,
              "map staging over tiles the last products read");
static_assert(SMEM <= 232448, "shared memory budget");
// tensor memory columns (512)
constexpr uint32_t TM_G1 = 0, TM_E = 256, TM_Y = 320, TM_WY = 384, TM_ZW = 0, TM_MAP = 128, TM_BAR = 192;
}  // namespace mk

__global__ void __launch_bounds__(NT, 1)
    maps_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_u,
                const __grid_constant__ CUtensorMap tm_ma, const __grid_constant__ CUtensorMap tm_mat,
                const __grid_constant__ CUtensorMap tm_mb, const __grid_constant__ CUtensorMap tm_mbb, Params p)
{
    using namespace mk;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    __shared__ uint32_t tmem_base_s;
    __shared__ __align__(8) uint64_t mbar[6];  // 0 loads, 1 Gram, 2 E/Y, 3 WY/ZW, 4 maps, 5 drain
    __shared__ int abort_s;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, quad = warp & 3, sub = warp >> 2;
    const int row = quad * 32 + lane;
    const int R = p.R;
    const int chunk = blockIdx.x, bh = chunk / p.NC, c = chunk % p.NC, h = bh % p.H;
    const int t0 = c * C, n = min(C, p.T - t0);
    const size_t tok0 = (size_t)bh * p.T + t0;
    float *sc = reinterpret_cast<float *>(sm + SC_OFF);
    const float *s_beta = sc + SC_BETA, *s_lam = sc + SC_LAM, *s_gam = sc + SC_GAM, *s_colf = sc + SC_COLF,
                *s_bg = sc + SC_BG;
    auto P = [&](int idx) { return sm + (uint32_t)idx * PANEL; };
    const uint32_t sbase = smem_u32(sm);
    const uint64_t dbase = sdesc(sbase, 0, 0);
    uint8_t *stash = reinterpret_cast<uint8_t *>(p.stash) + (size_t)chunk * STASH * PANEL;

    if (tid == 0) {
        abort_s = 0;
        for (int i = 0; i < 6; ++i) mbar_init(smem_u32(&mbar[i]), 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 0) tmem_alloc(smem_u32(&tmem_base_s), 512);
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tmem = tmem_base_s, lane_off = (uint32_t)(quad * 32) << 16;
    grid_dependency_wait();
    allow_dependent_launch();
    const uint32_t mb_ld = smem_u32(&mbar[0]);
    bool pend_ld = false;
    if (tid == 0) {
        mbar_expect_tx(mb_ld, (uint32_t)(3 + R) * PANEL);
        tma_load_3d(sbase + Q * PANEL, &tm_q, mb_ld, 0, t0, bh);
        tma_load_3d(sbase + K * PANEL, &tm_k, mb_ld, 0, t0, bh);
        for (int l = 0; l < R; ++l) tma_load_4d(sbase + (U0 + l) * PANEL, &tm_u, mb_ld, 0, l, t0, bh);
        tma_load_3d(sbase + V * PANEL, &tm_v, mb_ld, 0, t0, bh);
        pend_ld = true;
    }
    auto expired = [&]() {
        abort_s = 1;
        set_status(p.status, kDevTimeout);
    };
    auto wait_all = [&](int b, uint32_t ph) {
        if (!mbar_wait(smem_u32(&mbar[b]), ph, p.wait_ns)) expired();
    };
    // this thread's dout granules (row tid / 8; 0 past the end) and halo value, loaded before
    // anything else so that their loads are in flight together: the three tokens before the chunk
    // are history or earlier tokens of the sequence (zero before it)
    static_assert(NT == 64 * 8 && 3 * D <= NT, "one row granule pair and one halo value per thread");
    const int cr = tid >> 3, cg = tid & 7;
    float4 d0 = make_float4(0.f, 0.f, 0.f, 0.f), d1 = d0;
    if (cr < n) {
        const float4 *d4 = reinterpret_cast<const float4 *>(p.dout + (tok0 + cr) * D + 8 * cg);
        d0 = d4[0];
        d1 = d4[1];
    }
    float hx = 0.f;
    if (tid < 3 * D) {
        const int j = tid / D, ch = tid % D, t = t0 - 3 + j;
        if (t >= 0) hx = __bfloat162float(p.v[((size_t)bh * p.T + t) * D + ch]);
        else if (p.v_hist) hx = __bfloat162float(p.v_hist[((size_t)bh * 3 + (3 + t)) * D + ch]);
    }
    // thread 0 waits for the tiles at once (the first product needs them); the others stage
    if (tid == 0) {
        if (mbar_wait(mb_ld, 0, p.wait_ns)) pend_ld = false;
        else expired();
    }
    load_scalars(sc, p, tok0, n, tid);
    if (tid < 3 * D) sc[SC_HALO + tid] = hx;
    {
        uint4 w;
        w.x = pack_h2(d0.x, d0.y);
        w.y = pack_h2(d0.z, d0.w);
        w.z = pack_h2(d1.x, d1.y);
        w.w = pack_h2(d1.z, d1.w);
        *reinterpret_cast<uint4 *>(P(DO) + sw128(cr, 8 * cg)) = w;
    }
    for (int e = tid; e < 512; e += NT) reinterpret_cast<uint4 *>(P(ZERO))[e] = make_uint4(0, 0, 0, 0);
    __syncthreads();

    do {
        // ---- the Grams [Q; K] [K | U_l]^T on the bf16 tiles --------------------------------------------
        if (tid == 0) {
            if (!abort_s) {
                const uint32_t id = idesc_bf16(128, 64, 0, 0);
                for (int b = 0; b <= R; ++b)
                    mma_k64(tmem + TM_G1 + 64 * b, km(dbase, Q * PANEL), false,
                            km(dbase, (b == 0 ? K : U0 + b - 1) * PANEL), false, id, false);
            }
            mma_commit(smem_u32(&mbar[1]));
        }
        if (tid != 0) wait_all(0, 0);  // V has landed
        __syncthreads();
        if (abort_s) break;
        // ---- prep: x_{i,l} = gamma_il g_i r_il (two channels, eight tokens per thread) -> X_l; the
        // non-linear chain x_{i,l} = gamma_il GELU(p_il r_il), r_{i,l+1} = r_il - GELU(p_il r_il) ------
        if (R > 0) {
            const int cp = tid & 31, tg = tid >> 5;  // channel pair; tokens tg + 16 k
            const __nv_bfloat162 *cw = reinterpret_cast<const __nv_bfloat162 *>(p.conv_w) + (size_t)h * 4 * (D / 2) + cp;
            float2 w[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) w[j] = __bfloat1622float2(cw[j * (D / 2)]);
            const uint8_t *vp = P(V);
            auto vat = [&](int i) -> float2 {  // v of local token i (i >= -3)
                if (i >= 0) return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(vp + sw128(i, 2 * cp)));
                return make_float2(sc[SC_HALO + (3 + i) * D + 2 * cp], sc[SC_HALO + (3 + i) * D + 2 * cp + 1]);
            };
#pragma unroll 2
            for (int k = 0; k < 64 / (NT / 32); ++k) {
                const int i = tg + (NT / 32) * k;
                const float2 v0 = vat(i), v1 = vat(i - 1), v2 = vat(i - 2), v3 = vat(i - 3);
                const float a0 = fmaf(w[0].x, v0.x, fmaf(w[1].x, v1.x, fmaf(w[2].x, v2.x, w[3].x * v3.x)));
                const float a1 = fmaf(w[0].y, v0.y, fmaf(w[1].y, v1.y, fmaf(w[2].y, v2.y, w[3].y * v3.y)));
                float g0, g1, Phi0, Phi1;
                tcu::gelu_gain(a0, g0, Phi0);
                tcu::gelu_gain(a1, g1, Phi1);
                float r0 = v0.x - a0 * Phi0, r1 = v0.y - a1 * Phi1;
                // the gains of every level loaded before the first is used (tokens past the end: 0,
                // so delta = 0)
                float2 pv[RMAX];
                if (p.p_gain) {
                    const __nv_bfloat162 *pg = reinterpret_cast<const __nv_bfloat162 *>(p.p_gain + (tok0 + i) * R * D) + cp;
#pragma unroll
                    for (int l = 0; l < RMAX; ++l)
                        pv[l] = (i < n && l < R) ? __bfloat1622float2(pg[l * (D / 2)]) : make_float2(0.f, 0.f);
                }
#pragma unroll
                for (int l = 0; l < RMAX; ++l) {
                    if (l >= R) break;
                    const float gm = sc[SC_GM + i * RMAX + l], et = sc[SC_ET + i * RMAX + l];
                    float x0, x1;
                    if (p.p_gain) {
                        const float d0 = tcu::gelu_value(pv[l].x * r0), d1 = tcu::gelu_value(pv[l].y * r1);
                        x0 = gm * d0;
                        x1 = gm * d1;
                        r0 -= d0;
                        r1 -= d1;
                    } else {
                        x0 = gm * g0 * r0;
                        x1 = gm * g1 * r1;
                        r0 *= 1.f - et * g0;
                        r1 *= 1.f - et * g1;
                    }
                    const uint32_t xv = pack_h2(x0, x1);
                    *reinterpret_cast<uint32_t *>(P(X0 + l) + sw128(i, 2 * cp)) = xv;
                }
            }
            fence_async_smem();
        }
        wait_all(1, 0);
        fence_after_sync();
        // ---- Gram epilogue: P_k = (Q K^T) o D (j <= i); A = diag(beta) (K K^T) o D (j < i) (fp32, for
        // the solve); Mku_l = (K U_l^T) o D (j < i) --------------------------------------------------------
        float *sA = reinterpret_cast<float *>(P(F)), *sT32 = sA + 64 * tcu::LDA, *sX = sT32 + 64 * tcu::LDA;
        {
            const int j0 = CW * sub;
            float v[CW];
            if (row < 64) {
                tmem_ld(tmem + TM_G1 + lane_off + (uint32_t)j0, v);
                decay_row(v, s_lam, row, j0, true);
                st_row_h(P(PK), row, j0, v);
            } else {
                const int i = row - 64;
                tmem_ld(tmem + TM_G1 + lane_off + (uint32_t)j0, v);
                decay_row(v, s_lam, i, j0, false);
                const float b = s_beta[i];
#pragma unroll
                for (int q = 0; q < CW; ++q) v[q] *= b;
                st_row_f(sA + i * tcu::LDA + j0, v);
                for (int l = 0; l < R; ++l) {
                    tmem_ld(tmem + TM_G1 + 64 * (l + 1) + lane_off + (uint32_t)j0, v);
                    decay_row(v, s_lam, i, j0, false);
                    st_row_h(P(MKU0 + l), i, j0, v);
                }
            }
        }
        fence_async_smem();
        fence_before_sync();
        __syncthreads();
        // ---- E = Mku X and Y = P_k^T dO on the tensor core while the warps solve T -------------------
        if (tid == 0) {
            fence_after_sync();
            for (int l = 0; l < R; ++l)
                mma_k64(tmem + TM_E, km(dbase, (MKU0 + l) * PANEL), false, mn(dbase, (X0 + l) * PANEL, PANEL), true,
                        idesc_f16(128, 64, 0, 1), l > 0);
            mma_k64(tmem + TM_Y, mn(dbase, PK * PANEL, PANEL), true, mn(dbase, DO * PANEL, PANEL), true,
                    idesc_f16(128, 64, 1, 1), false);
            mma_commit(smem_u32(&mbar[2]));
            for (int l = 0; l < R; ++l) bulk_store(stash + (ST_X + l) * PANEL, sbase + (X0 + l) * PANEL, PANEL);
            bulk_commit();
        }
        if (tid < tcu::SOLVE_THREADS) tcu::ut_solve(sA, sT32, sX, P(TF), tid, 1);
        fence_async_smem();
        wait_all(2, 0);
        fence_after_sync();
        __syncthreads();  // the solve region is free from here on
        // ---- E0 = V - Mku X, beta E0, Y (rows < 64); the scaled key and query copies (rows >= 64) ------
        {
            const int c0 = CW * sub;
            float v[CW], e[CW];
            if (row < 64) {
                const int i = row;
                if (R > 0) {
                    tmem_ld(tmem + TM_E + lane_off + (uint32_t)c0, e);
                } else {
#pragma unroll
                    for (int q = 0; q < CW; ++q) e[q] = 0.f;
                }
                ld_row_b(P(V), i, c0, v);
#pragma unroll
                for (int q = 0; q < CW; ++q) v[q] -= e[q];
                st_row_h(P(V), i, c0, v);  // E0 in place of the values (their last reader), for the stash
                const float b = s_beta[i];
#pragma unroll
                for (int q = 0; q < CW; ++q) v[q] *= b;
                st_row_h(P(BE), i, c0, v);
                tmem_ld(tmem + TM_Y + lane_off + (uint32_t)c0, v);
                st_row_h(P(Y), i, c0, v);
            } else {
                const int i = row - 64;
                ld_row_b(P(K), i, c0, v);
                const float bg = s_bg[i], cf = s_colf[i];
#pragma unroll
                for (int q = 0; q < CW; ++q) e[q] = bg * v[q];
                st_row_h(P(BGK), i, c0, e);
#pragma unroll
                for (int q = 0; q < CW; ++q) e[q] = -e[q];
                st_row_h(P(NBGK), i, c0, e);
#pragma unroll
                for (int q = 0; q < CW; ++q) e[q] = cf * v[q];
                st_row_h(P(CK), i, c0, e);
                ld_row_b(P(Q), i, c0, v);
                const float gi = s_gam[i];
#pragma unroll
                for (int q = 0; q < CW; ++q) v[q] *= gi;
                st_row_h(P(PK), i, c0, v);
                for (int l = 0; l < R; ++l) {
                    ld_row_b(P(U0 + l), i, c0, v);
#pragma unroll
                    for (int q = 0; q < CW; ++q) v[q] *= cf;
                    st_row_h(P(MKU0 + l), i, c0, v);
                }
            }
        }
        fence_async_smem();
        fence_before_sync();
        __syncthreads();
        // ---- [U' | W] = T [beta E0 | beta Gamma K];  [Z0 | Wbar] = T^T [Y | colf K] ----------------------
        if (tid == 0) {
            fence_after_sync();
            mma_k64(tmem + TM_WY, km(dbase, TF * PANEL), false, mn(dbase, BE * PANEL, PANEL), true,
                    idesc_f16(128, 128, 0, 1), false);
            mma_k64(tmem + TM_ZW, mn(dbase, TF * PANEL, PANEL), true, mn(dbase, Y * PANEL, PANEL), true,
                    idesc_f16(128, 128, 1, 1), false);
            mma_commit(smem_u32(&mbar[3]));
            bulk_store(stash + ST_E0 * PANEL, sbase + V * PANEL, PANEL);
            bulk_commit();
        }
        wait_all(3, 0);
        fence_after_sync();
        if (row < 64) {
            const int i = row, c0 = CW * sub;
            float v[CW];
            tmem_ld(tmem + TM_WY + lane_off + (uint32_t)c0, v);
            st_row_h(P(UP), i, c0, v);
            tmem_ld(tmem + TM_WY + 64 + lane_off + (uint32_t)c0, v);
            st_row_h(P(W), i, c0, v);
            tmem_ld(tmem + TM_ZW + lane_off + (uint32_t)c0, v);
            st_row_h(P(Z0), i, c0, v);
            tmem_ld(tmem + TM_ZW + 64 + lane_off + (uint32_t)c0, v);
            st_row_h(P(TF), i, c0, v);  // Wbar, for the stash only, over T (read by the products above)
        }
        fence_async_smem();
        fence_before_sync();
        __syncthreads();
        // ---- maps: [W^T; U'^T] colf K + [0; X_l^T] colf U_l;  [0; dO^T] Gamma Q - [0; Z0^T] beta Gamma K ---
        if (tid == 0) {
            fence_after_sync();
            const uint32_t id = idesc_f16(128, 64, 1, 1);
            mma_k64(tmem + TM_MAP, mn(dbase, W * PANEL, (UP - W) * PANEL), true, mn(dbase, CK * PANEL, PANEL), true, id,
                    false);
            for (int l = 0; l < R; ++l)
                mma_k64(tmem + TM_MAP, mn(dbase, ZERO * PANEL, (X0 + l - ZERO) * PANEL), true,
                        mn(dbase, (MKU0 + l) * PANEL, PANEL), true, id, true);
            mma_k64(tmem + TM_BAR, mn(dbase, ZERO * PANEL, (DO - ZERO) * PANEL), true, mn(dbase, PK * PANEL, PANEL),
                    true, id, false);
            mma_k64(tmem + TM_BAR, mn(dbase, ZERO * PANEL, (Z0 - ZERO) * PANEL), true, mn(dbase, NBGK * PANEL, PANEL),
                    true, id, true);
            mma_commit(smem_u32(&mbar[4]));
            bulk_store(stash + ST_UP * PANEL, sbase + UP * PANEL, PANEL);
            bulk_store(stash + ST_W * PANEL, sbase + W * PANEL, PANEL);
            bulk_store(stash + ST_Z0 * PANEL, sbase + Z0 * PANEL, PANEL);
            bulk_store(stash + ST_WB * PANEL, sbase + TF * PANEL, PANEL);
            bulk_commit();
        }
        wait_all(4, 0);
        fence_after_sync();
        {
            const int n0 = CW * sub;
            float v[CW];
            tmem_ld(tmem + TM_MAP + lane_off + (uint32_t)n0, v);
            if (row < 64) {  // A_c [m][n] = Gamma_63 [m == n] - (W^T colf K)[m][n], and its transpose
                const float g63 = s_gam[63];
#pragma unroll
                for (int q = 0; q < CW; ++q) v[q] = (n0 + q == row ? g63 : 0.f) - v[q];
                st_tile_f(P(MA), row, n0, v);
#pragma unroll
                for (int q = 0; q < CW; ++q) *reinterpret_cast<float *>(P(MAT) + tile_f_off(n0 + q, row)) = v[q];
            } else {
                st_tile_f(P(MB), row - 64, n0, v);
                tmem_ld(tmem + TM_BAR + lane_off + (uint32_t)n0, v);
                st_tile_f(P(MBB), row - 64, n0, v);
            }
        }
        fence_async_smem();
        fence_before_sync();
        __syncthreads();
        if (tid == 0) {
            for (int h2 = 0; h2 < 2; ++h2) {
                tma_store_2d(&tm_ma, sbase + (MA + h2) * PANEL, 32 * h2, chunk * 64);
                tma_store_2d(&tm_mat, sbase + (MAT + h2) * PANEL, 32 * h2, chunk * 64);
                tma_store_2d(&tm_mb, sbase + (MB + h2) * PANEL, 32 * h2, chunk * 64);
                tma_store_2d(&tm_mbb, sbase + (MBB + h2) * PANEL, 32 * h2, chunk * 64);
            }
            bulk_commit();
        }
    } while (0);

    // drain (after an expired wait): let the copies and products in flight land, bounded
    if (tid == 0 && abort_s) {
        const uint64_t drain_ns = 1000000000ull;
        if (pend_ld) (void)mbar_wait(mb_ld, 0, drain_ns);
        const uint32_t mb_drain = smem_u32(&mbar[5]);
        mma_commit(mb_drain);
        (void)mbar_wait(mb_drain, 0, drain_ns);
    }
    if (tid == 0) bulk_wait_read();  // the stash and map stores have read their tiles
    fence_before_sync();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, 512);
}

// =====================================================================================================
// scan: grid (64 / SC_ROWS row blocks, BH, 2 directions), 256 + 32 threads.  Forward: S_{c+1} = S_c A_c + B_c
// from S_init (or 0), storing S_c for c = 0 .. NC.  Reverse: G_{c-1} = G_c A_c^T + Bbar_c from
// dS_final (or 0), storing G_c for c = NC-1 .. 0, the last value being dS_init.  Thread (q, c)
// forms the partial sums over m in [16 q, 16 q + 16) of all the block's rows of column c, so each
// map element is read from shared memory once per step and used for every row from a register; the
// four partials meet through shared memory.  Four rows a block: two blocks share an SM, which hides
// the step's latencies better than one block of eight rows.  The maps stream through a ring of bulk
// copies issued by one lane of a producer warp, off the steps' critical path: every consumer waits
// on the stage's `full` mbarrier, each consumer warp arrives on its `empty` mbarrier once it has
// read the stage, and the producer waits for that before refilling it (every wait bounded).
constexpr int SC_ROWS = 4, SC_STAGES = 4;
constexpr int SC_OUTS = SC_ROWS * D / SCAN_NT;  // outputs a thread forms in the reduction (consecutive columns)
static_assert(SC_OUTS >= 1 && SC_OUTS <= 4, "scan layout");
constexpr int SC_STAGE_FLOATS = D * D + SC_ROWS * D;
constexpr size_t SCAN_SMEM = (size_t)(SC_STAGES * SC_STAGE_FLOATS + SC_ROWS * D + 4 * SC_ROWS * D) * 4 + 128;
// The shared memory the scan's launch requests: more than the scan uses, so that at most two of its
// blocks fit an SM.  Launched while the maps kernel drains (programmatic dependent launch), the
// blocks are placed on SMs as they free up; with room for three, the first SMs freed took three
// and the steps of their chains ran slower (0.78 against 0.72 ms per backward pass at 16K tokens).
constexpr size_t SCAN_SMEM_LAUNCH = 100 * 1024;
static_assert(SCAN_SMEM <= SCAN_SMEM_LAUNCH && 3 * (SCAN_SMEM_LAUNCH + 1024) > 228 * 1024, "two scan blocks per SM");
static_assert(SC_OUTS * SCAN_NT == SC_ROWS * D && SCAN_NT % 64 == 0, "the consumers' roles");

__global__ void __launch_bounds__(SCAN_NT + 32) scan_kernel(const float *__restrict__ mapA, const float *__restrict__ mapAT,
                                                       const float *__restrict__ mapB, const float *__restrict__ mapBb,
                                                       const float *__restrict__ S_init, const float *__restrict__ dS_final,
                                                       float *__restrict__ Sst, float *__restrict__ Gst,
                                                       float *__restrict__ dS_init, int NC, int *status,
                                                       unsigned long long wait_ns)
{
    extern __shared__ __align__(128) float ssm[];
    float *st = ssm + SC_STAGES * SC_STAGE_FLOATS;  // the state rows [SC_ROWS][64]
    float *red = st + SC_ROWS * D;                  // partial sums [4][SC_ROWS][64]
    __shared__ __align__(8) uint64_t full[SC_STAGES], empty[SC_STAGES];
    const int tid = threadIdx.x, col = tid & 63, qm = tid >> 6;  // partial-sum role
    const int orow = tid / (D / SC_OUTS), oc = (tid % (D / SC_OUTS)) * SC_OUTS;  // output role
    const int rb = blockIdx.x * SC_ROWS, bh = blockIdx.y;
    const bool rev = blockIdx.z == 1;
    const float *M = rev ? mapAT : mapA, *Bv = rev ? mapBb : mapB;
    const float *init = rev ? dS_final : S_init;
    if (tid == 0) {
        for (int i = 0; i < SC_STAGES; ++i) {
            mbar_init(smem_u32(&full[i]), 1);
            mbar_init(smem_u32(&empty[i]), SCAN_NT / 32);  // one arrival per consumer warp
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    grid_dependency_wait();
    allow_dependent_launch();
    float s[SC_OUTS];
    if (tid < SCAN_NT) {
#pragma unroll
        for (int e = 0; e < SC_OUTS; ++e) s[e] = init ? init[((size_t)bh * D + rb + orow) * D + oc + e] : 0.f;
#pragma unroll
        for (int e = 0; e < SC_OUTS; ++e) st[orow * D + oc + e] = s[e];
    }
    __syncthreads();

    if (tid >= SCAN_NT) {  // ---- producer: one lane of the last warp streams the maps -------------------
        if (tid == SCAN_NT) {
            int issued = 0;
            for (int k = 0; k < NC; ++k) {
                const int slot = k % SC_STAGES;
                if (k >= SC_STAGES &&
                    !mbar_wait(smem_u32(&empty[slot]), (uint32_t)(k / SC_STAGES - 1) & 1u, wait_ns)) {
                    set_status(status, kDevTimeout);
                    break;
                }
                const int cc = rev ? NC - 1 - k : k;
                const size_t mo = ((size_t)bh * NC + cc) * D * D;
                const uint32_t mb = smem_u32(&full[slot]);
                const uint32_t dst = smem_u32(ssm + slot * SC_STAGE_FLOATS);
                mbar_expect_tx(mb, SC_STAGE_FLOATS * 4);
                bulk_load(dst, M + mo, D * D * 4, mb);
                bulk_load(dst + D * D * 4, Bv + mo + (size_t)rb * D, SC_ROWS * D * 4, mb);
                issued = k + 1;
            }
            // every copy issued lands before the CTA exits (bounded): only the last SC_STAGES
            // stages can still be in flight
            for (int j = max(0, issued - SC_STAGES); j < issued; ++j)
                (void)mbar_wait(smem_u32(&full[j % SC_STAGES]), (uint32_t)(j / SC_STAGES) & 1u, 1000000000ull);
        }
        return;
    }

    // ---- consumers (the first SCAN_NT threads); their barriers leave the producer warp out.  An
    // expired wait is recorded per thread and OR-reduced at the step's last barrier, so every
    // consumer leaves the loop at the same step.
    bool expired = false, stop = false;
    for (int k = 0; k < NC; ++k) {
        const int cc = rev ? NC - 1 - k : k;
        float *out = rev ? Gst + ((size_t)bh * NC + cc) * D * D : Sst + ((size_t)bh * (NC + 1) + cc) * D * D;
#pragma unroll
        for (int e = 0; e < SC_OUTS; ++e) out[(size_t)(rb + orow) * D + oc + e] = s[e];
        const int slot = k % SC_STAGES;
        if (!mbar_wait(smem_u32(&full[slot]), (uint32_t)(k / SC_STAGES) & 1u, wait_ns)) {
            expired = true;
            set_status(status, kDevTimeout);
        }
        const float *mm = ssm + slot * SC_STAGE_FLOATS;
        float part[SC_ROWS];
#pragma unroll
        for (int r = 0; r < SC_ROWS; ++r) part[r] = 0.f;
#pragma unroll
        for (int m4 = 0; m4 < 4; ++m4) {
            const int m0 = 16 * qm + 4 * m4;
            float w[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) w[q] = mm[(m0 + q) * D + col];
#pragma unroll
            for (int r = 0; r < SC_ROWS; ++r) {
                const float4 a = *reinterpret_cast<const float4 *>(st + r * D + m0);
                part[r] = fmaf(a.x, w[0], fmaf(a.y, w[1], fmaf(a.z, w[2], fmaf(a.w, w[3], part[r]))));
            }
        }
#pragma unroll
        for (int r = 0; r < SC_ROWS; ++r) red[(qm * SC_ROWS + r) * D + col] = part[r];
        named_bar(1, SCAN_NT);  // partials complete; the state rows of step k are no longer read
        float bv[SC_OUTS];
#pragma unroll
        for (int e = 0; e < SC_OUTS; ++e) bv[e] = mm[D * D + orow * D + oc + e];
        __syncwarp();
        if ((tid & 31) == 0) mbar_arrive(smem_u32(&empty[slot]));  // this warp is done with the stage
#pragma unroll
        for (int e = 0; e < SC_OUTS; ++e) {
            float acc = bv[e];
#pragma unroll
            for (int q = 0; q < 4; ++q) acc += red[(q * SC_ROWS + orow) * D + oc + e];
            st[orow * D + oc + e] = acc;
            s[e] = acc;
        }
        // the new state is written and the partials are free; leave together after an expired wait
        if ((stop = named_bar_or(1, SCAN_NT, expired))) break;
    }
    if (stop) return;
#pragma unroll
    for (int e = 0; e < SC_OUTS; ++e) {
        if (!rev) Sst[((size_t)bh * (NC + 1) + NC) * D * D + (size_t)(rb + orow) * D + oc + e] = s[e];
        else if (dS_init) dS_init[((size_t)bh * D + rb + orow) * D + oc + e] = s[e];
    }
}

// =====================================================================================================
// grad: the cotangents of one chunk, one CTA per chunk.  Two halves on one set of tiles:
//   values   [K; W] S^T -> E and Vt;  [Wbar; colf U_0] G^T -> z, then + [0; P_0^T] dO - [0; Mku_0^T]
//            beta Z -> dX_0 (likewise dX_1, dX_2);  Akk Vt -> dbeta;  dv = beta z;
//            sigma_t = beta_t v_t.z_t + sum_l x_tl.dx_tl
//   keys     [Vt; X_0] [dO | Z]^T, [X_1; X_2] [dO | Z]^T -> J, H;  [colf Vt; colf X_0] G + [J_0; J_1] Q
//            - [H_0; H_1] beta K -> dk's write part and du_0 (likewise du_1, du_2);
//            [Gamma dO; Gamma Z] S + sum_b [J_b^T; H_b^T] Kw_b -> dq and dk's state part; dalpha.
// Vt, Z, X and dO stay in shared memory between the halves; E stays in the registers of the
// threads (rows < 64) that form dbeta.  Shared-memory panels (index x PANEL from a 1024-aligned
// base); the second half's tiles take the first half's dead ones.
namespace gk {
enum {
    Q = 0, K = 1, W = 2, U0 = 3, VT = 6, X0 = 7, DO = 10, Z = 11, S0 = 12, GB = 13, WB = 14, CU0 = 15, ZERO = 18,
    P0 = 19, AKK = 22, MKU0 = 23, NPANELS = 26,
    NBK = 2,    // -beta K, in W's place (W is read by the first products only)
    J0 = 14,    // J_0..J_3 over Wbar and colf U_l
    H0 = 18,    // H_0..H_3 over the zero tile and P_l (H_b = J_b + 4 panels)
    DKW = 22,   // dk's write part, then dk, fp32 [64][64] staged for its TMA store, over Akk and Mku_0
    DQS = 6,    // dq, staged (fp32, two panels) over Vt and X_0 once the last products have read them
    DUS = 8,    // du_0 .. du_2, staged at DUS + 2 l (X_1 .. GB)
    DVS = 14,   // dv, staged over Wbar and colf U_0 (read by the first products only)
    DXS = 22    // dX_0, dX_1 over Akk and Mku (read by the second products); dX_2 at DXS2
};
constexpr int DXS2 = 16;  // over colf U_1, U_2
__host__ __device__ constexpr int dx_stage(int l) { return l < 2 ? DXS + 2 * l : DXS2; }
constexpr uint32_t SC_OFF = NPANELS * PANEL;
constexpr uint32_t SMEM = SC_OFF + SC_FLOATS * 4 + 1024;
static_assert(SMEM <= 232448, "shared memory budget");
static_assert(H0 - J0 == 4 && X0 == VT + 1 && Z == DO + 1 && W == K + 1 && CU0 == WB + 1, "stacked operands");
static_assert(DQS + 2 <= DUS && DUS + 2 * RMAX <= J0 && DQS > Q, "output staging over tiles the last products read");
static_assert(DVS == WB && DVS + 2 == DXS2 && DXS2 + 2 == ZERO && DXS == AKK && DXS + 4 == NPANELS && RMAX <= 3,
              "dv and dX staging over tiles dead after the first / second products");
// tensor memory columns (512): first half, then the second half over the dead first-half columns
constexpr uint32_t TM_G1 = 0, TM_D1 = 256, TM_D2 = 320, TM_D3 = 384, TM_DF = 448;
constexpr uint32_t TM_C = 0, TM_D = 256, TM_E = 384;
}  // namespace gk

__global__ void __launch_bounds__(NT, 1)
    grad_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                const __grid_constant__ CUtensorMap tm_u, const __grid_constant__ CUtensorMap tm_dq,
                const __grid_constant__ CUtensorMap tm_dk, const __grid_constant__ CUtensorMap tm_du,
                const __grid_constant__ CUtensorMap tm_dv, const __grid_constant__ CUtensorMap tm_dx, Params p)
{
    using namespace gk;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    __shared__ uint32_t tmem_base_s;
    __shared__ __align__(8) uint64_t mbar[6];  // 0 loads, 1-4 products, 5 drain
    __shared__ int abort_s;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, quad = warp & 3, sub = warp >> 2;
    const int row = quad * 32 + lane;
    const int R = p.R;
    const int chunk = blockIdx.x, bh = chunk / p.NC, c = chunk % p.NC;
    const int t0 = c * C, n = min(C, p.T - t0);
    const size_t tok0 = (size_t)bh * p.T + t0;
    float *sc = reinterpret_cast<float *>(sm + SC_OFF);
    const float *s_beta = sc + SC_BETA, *s_lam = sc + SC_LAM, *s_gam = sc + SC_GAM, *s_colf = sc + SC_COLF;
    // per-token partial sums in fixed slots (summed in a fixed order, so the pass is deterministic):
    // sigma [16][64] (slots 0-3: beta v.z by column part; 4 + 4 l + part: x_l.dx_l), dbeta [4][64],
    // q.dq [4][64]; <G, S'> per warp [16]
    float *s_sig = sc + SC_RED, *s_db = s_sig + 16 * 64, *s_qdq = s_db + 4 * 64, *s_Fw = s_qdq + 4 * 64;
    auto P = [&](int idx) { return sm + (uint32_t)idx * PANEL; };
    const uint32_t sbase = smem_u32(sm);
    const uint64_t dbase = sdesc(sbase, 0, 0);
    const uint8_t *stash = reinterpret_cast<const uint8_t *>(p.stash) + (size_t)chunk * STASH * PANEL;
    const float *Gc = p.Gst + ((size_t)bh * p.NC + c) * D * D;
    const float *Sc = p.Sst + ((size_t)bh * (p.NC + 1) + c) * D * D;

    if (tid == 0) {
        abort_s = 0;
        for (int i = 0; i < 6; ++i) mbar_init(smem_u32(&mbar[i]), 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 0) tmem_alloc(smem_u32(&tmem_base_s), 512);
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tmem = tmem_base_s, lane_off = (uint32_t)(quad * 32) << 16;
    grid_dependency_wait();  // the scan's states
    allow_dependent_launch();
    const uint32_t mb_ld = smem_u32(&mbar[0]);
    bool pend_ld = false;
    if (tid == 0) {
        mbar_expect_tx(mb_ld, (uint32_t)(4 + 2 * R) * PANEL);
        tma_load_3d(sbase + Q * PANEL, &tm_q, mb_ld, 0, t0, bh);
        tma_load_3d(sbase + K * PANEL, &tm_k, mb_ld, 0, t0, bh);
        for (int l = 0; l < R; ++l) tma_load_4d(sbase + (U0 + l) * PANEL, &tm_u, mb_ld, 0, l, t0, bh);
        bulk_load(sbase + W * PANEL, stash + ST_W * PANEL, PANEL, mb_ld);
        bulk_load(sbase + WB * PANEL, stash + ST_WB * PANEL, PANEL, mb_ld);
        for (int l = 0; l < R; ++l) bulk_load(sbase + (X0 + l) * PANEL, stash + (ST_X + l) * PANEL, PANEL, mb_ld);
        pend_ld = true;
    }
    auto expired = [&]() {
        abort_s = 1;
        set_status(p.status, kDevTimeout);
    };
    auto wait_all = [&](int b, uint32_t ph) {
        if (!mbar_wait(smem_u32(&mbar[b]), ph, p.wait_ns)) expired();
    };
    // the chunk's fp32 operands into registers before anything else: S_c, G_c, dout (0 past the
    // end) and S_{c+1}, granules 2 cg, 2 cg + 1 of row cr, so that their loads are in flight together
    static_assert(NT == 64 * 8, "one row granule pair per thread");
    const int cr = tid >> 3, cg = tid & 7;
    float4 fv[8];
    {
        const float4 *s4 = reinterpret_cast<const float4 *>(Sc + cr * D + 8 * cg);
        const float4 *g4 = reinterpret_cast<const float4 *>(Gc + cr * D + 8 * cg);
        const float4 *n4 = reinterpret_cast<const float4 *>(Sc + D * D + cr * D + 8 * cg);
        fv[0] = s4[0];
        fv[1] = s4[1];
        fv[2] = g4[0];
        fv[3] = g4[1];
        fv[6] = n4[0];
        fv[7] = n4[1];
        fv[4] = fv[5] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (cr < n) {
            const float4 *d4 = reinterpret_cast<const float4 *>(p.dout + (tok0 + cr) * D + 8 * cg);
            fv[4] = d4[0];
            fv[5] = d4[1];
        }
    }
    if (tid == 0) {  // thread 0 waits for the tiles at once; the others stage
        if (mbar_wait(mb_ld, 0, p.wait_ns)) pend_ld = false;
        else expired();
    }
    load_scalars(sc, p, tok0, n, tid);
    for (int e = tid; e < 24 * 64; e += NT) s_sig[e] = 0.f;  // sigma, dbeta, q.dq slots
    {
        auto put = [&](int panel, const float4 &a, const float4 &b) {
            uint4 w;
            w.x = pack_h2(a.x, a.y);
            w.y = pack_h2(a.z, a.w);
            w.z = pack_h2(b.x, b.y);
            w.w = pack_h2(b.z, b.w);
            *reinterpret_cast<uint4 *>(P(panel) + sw128(cr, 8 * cg)) = w;
        };
        put(S0, fv[0], fv[1]);
        put(GB, fv[2], fv[3]);
        put(DO, fv[4], fv[5]);
    }
    for (int e = tid; e < 512; e += NT) reinterpret_cast<uint4 *>(P(ZERO))[e] = make_uint4(0, 0, 0, 0);
    {  // F0 = <G_c, S_{c+1}> (for dalpha), partial per warp
        float part = 0.f;
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            const float4 a = fv[2 + q], b = fv[6 + q];
            part = fmaf(a.x, b.x, fmaf(a.y, b.y, fmaf(a.z, b.z, fmaf(a.w, b.w, part))));
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) part += __shfl_xor_sync(0xffffffffu, part, off);
        if (lane == 0) s_Fw[warp] = part;
    }
    __syncthreads();

    float z[CW], Ev[CW];  // rows < 64: this thread's columns of z_i and of E_i (kept for dbeta)
    do {
        if (abort_s) break;
        // ---- the input tiles to fp16 in place; colf U_l copies ----------------------------------------------
        panel_to_f16(P(Q), nullptr, nullptr, 1.f, tid);
        panel_to_f16(P(K), nullptr, nullptr, 1.f, tid);
        for (int l = 0; l < R; ++l) panel_to_f16(P(U0 + l), P(CU0 + l), s_colf, 1.f, tid);
        fence_async_smem();
        __syncthreads();
        // ---- values: Grams [Q; K] [K | U_l]^T;  [K; W] S^T;  [Wbar; colf U_0] G^T;  [colf U_1; colf U_2] G^T ----
        if (tid == 0) {
            const uint32_t id = idesc_f16(128, 64, 0, 0);
            for (int b = 0; b <= R; ++b)
                mma_k64(tmem + TM_G1 + 64 * b, km(dbase, Q * PANEL), false, km(dbase, (b == 0 ? K : U0 + b - 1) * PANEL),
                        false, id, false);
            mma_k64(tmem + TM_D1, km(dbase, K * PANEL), false, km(dbase, S0 * PANEL), false, id, false);
            mma_k64(tmem + TM_D2, km(dbase, WB * PANEL), false, km(dbase, GB * PANEL), false, id, false);
            if (R >= 2) mma_k64(tmem + TM_D3, km(dbase, (CU0 + 1) * PANEL), false, km(dbase, GB * PANEL), false, id, false);
            mma_commit(smem_u32(&mbar[1]));
        }
        // this thread's rows of the stash and of v, loaded while the products run
        uint4 pre[3][CW / 8];
        {
            const int j0 = CW * sub, i = row & 63;
            if (row < 64) {
                ld_row_raw(stash + ST_E0 * PANEL, i, j0, pre[0]);
                ld_row_raw(stash + ST_Z0 * PANEL, i, j0, pre[1]);
                if (i < n) {
#pragma unroll
                    for (int g = 0; g < CW / 8; ++g) pre[2][g] = reinterpret_cast<const uint4 *>(p.v + (tok0 + i) * D + j0)[g];
                }
            } else {
                ld_row_raw(stash + ST_UP * PANEL, i, j0, pre[0]);
            }
        }
        wait_all(1, 0);
        fence_after_sync();
        {
            const int j0 = CW * sub;
            float v[CW], s2[CW];
            if (row < 64) {
                const int i = row;
                // P_l = (Q U_l^T) o D (j <= i)
                for (int l = 0; l < R; ++l) {
                    tmem_ld(tmem + TM_G1 + 64 * (l + 1) + lane_off + (uint32_t)j0, v);
                    decay_row(v, s_lam, i, j0, true);
                    st_row_h(P(P0 + l), i, j0, v);
                }
                // E = E0 - Gamma_i (K S^T)_i  (fp32, kept in registers for dbeta)
                tmem_ld(tmem + TM_D1 + lane_off + (uint32_t)j0, v);
                h8_to_f(pre[0], Ev);
                const float gi = s_gam[i];
#pragma unroll
                for (int q = 0; q < CW; ++q) Ev[q] -= gi * v[q];
                // z = Z0 + (Wbar G^T)_i;  Z (fp16);  dv = beta z;  sigma += beta v.z
                tmem_ld(tmem + TM_D2 + lane_off + (uint32_t)j0, v);
                h8_to_f(pre[1], s2);
                const float b = s_beta[i];
#pragma unroll
                for (int q = 0; q < CW; ++q) z[q] = s2[q] + v[q];
                st_row_h(P(Z), i, j0, z);
                {
                    float dvv[CW];
#pragma unroll
                    for (int q = 0; q < CW; ++q) dvv[q] = b * z[q];
                    st_tile_f(P(DVS), i, j0, dvv);
                }
                if (i < n) {
                    const __nv_bfloat162 *vr = reinterpret_cast<const __nv_bfloat162 *>(pre[2]);
                    float part = 0.f;
#pragma unroll
                    for (int q = 0; q < CW / 2; ++q) {
                        const float2 f = __bfloat1622float2(vr[q]);
                        part = fmaf(f.x, z[2 * q], fmaf(f.y, z[2 * q + 1], part));
                    }
                    s_sig[sub * 64 + i] = b * part;
                }
            } else {
                const int i = row - 64;
                const float nb = -s_beta[i];
                // Akk = (K K^T) o D (j < i);  -beta_i Mku_l = -beta_i (K U_l^T) o D (j < i)
                tmem_ld(tmem + TM_G1 + lane_off + (uint32_t)j0, v);
                decay_row(v, s_lam, i, j0, false);
                st_row_h(P(AKK), i, j0, v);
                for (int l = 0; l < R; ++l) {
                    tmem_ld(tmem + TM_G1 + 64 * (l + 1) + lane_off + (uint32_t)j0, v);
                    decay_row(v, s_lam, i, j0, false);
#pragma unroll
                    for (int q = 0; q < CW; ++q) v[q] *= nb;
                    st_row_h(P(MKU0 + l), i, j0, v);
                }
                // Vt = U' - (W S^T)_i
                tmem_ld(tmem + TM_D1 + lane_off + (uint32_t)j0, v);
                h8_to_f(pre[0], s2);
#pragma unroll
                for (int q = 0; q < CW; ++q) s2[q] -= v[q];
                st_row_h(P(VT), i, j0, s2);
                // -beta K (for the keys half), in W's place: the products that read W are complete
                ld_row_h(P(K), i, j0, s2);
#pragma unroll
                for (int q = 0; q < CW; ++q) s2[q] *= nb;
                st_row_h(P(NBK), i, j0, s2);
            }
        }
        fence_async_smem();
        fence_before_sync();
        __syncthreads();
        // ---- dX_l += P_l^T dO + (-beta Mku_l)^T Z;  Akk Vt ---------------------------------------------------
        if (tid == 0) {
            fence_after_sync();
            const uint32_t id = idesc_f16(128, 64, 1, 1);
            if (R >= 1) {
                mma_k64(tmem + TM_D2, mn(dbase, ZERO * PANEL, (P0 - ZERO) * PANEL), true, mn(dbase, DO * PANEL, PANEL),
                        true, id, true);
                mma_k64(tmem + TM_D2, mn(dbase, ZERO * PANEL, (MKU0 - ZERO) * PANEL), true, mn(dbase, Z * PANEL, PANEL),
                        true, id, true);
            }
            if (R >= 2) {
                mma_k64(tmem + TM_D3, mn(dbase, (P0 + 1) * PANEL, PANEL), true, mn(dbase, DO * PANEL, PANEL), true, id,
                        true);
                mma_k64(tmem + TM_D3, mn(dbase, (MKU0 + 1) * PANEL, PANEL), true, mn(dbase, Z * PANEL, PANEL), true, id,
                        true);
            }
            mma_k64(tmem + TM_DF, km(dbase, AKK * PANEL), false, mn(dbase, VT * PANEL, PANEL), true,
                    idesc_f16(128, 64, 0, 1), false);
            mma_commit(smem_u32(&mbar[2]));
            for (int h = 0; h < 2; ++h) tma_store_3d(&tm_dv, sbase + (DVS + h) * PANEL, 32 * h, t0, bh);
            bulk_commit();
        }
        wait_all(2, 0);
        fence_after_sync();
        {
            const int j0 = CW * sub;
            float v[CW], x[CW];
            auto dx_out = [&](uint32_t col, int l, int i) {  // dX_l row i -> staged, sigma += x.dx
                tmem_ld(tmem + col + lane_off + (uint32_t)j0, v);
                st_tile_f(P(dx_stage(l)), i, j0, v);
                if (i < n) {
                    ld_row_h(P(X0 + l), i, j0, x);
                    float part = 0.f;
#pragma unroll
                    for (int q = 0; q < CW; ++q) part = fmaf(x[q], v[q], part);
                    s_sig[(4 + 4 * l + sub) * 64 + i] = part;
                }
            };
            if (row < 64) {
                const int i = row;
                if (R >= 2) dx_out(TM_D3, 1, i);
                // dbeta_i = sum_c z_ic (E_ic - (Akk Vt)_ic)
                tmem_ld(tmem + TM_DF + lane_off + (uint32_t)j0, v);
                float part = 0.f;
#pragma unroll
                for (int q = 0; q < CW; ++q) part = fmaf(z[q], Ev[q] - v[q], part);
                s_db[sub * 64 + i] = part;
            } else {
                const int i = row - 64;
                if (R >= 1) dx_out(TM_D2, 0, i);
                if (R >= 3) dx_out(TM_D3, 2, i);
            }
        }
        fence_async_smem();
        fence_before_sync();
        __syncthreads();
        if (tid < n) p.dbeta[tok0 + tid] = (s_db[tid] + s_db[64 + tid]) + (s_db[128 + tid] + s_db[192 + tid]);
        // ---- keys: [Vt; X_0] [dO | Z]^T and [X_1; X_2] [dO | Z]^T -------------------------------------------
        if (tid == 0) {
            fence_after_sync();
            const uint32_t id = idesc_f16(128, 128, 0, 0);
            mma_k64(tmem + TM_C, km(dbase, VT * PANEL), false, km(dbase, DO * PANEL), false, id, false);
            if (R >= 2) mma_k64(tmem + TM_C + 128, km(dbase, (X0 + 1) * PANEL), false, km(dbase, DO * PANEL), false, id, false);
            for (int h = 0; h < 2; ++h)
                for (int l = 0; l < R; ++l) tma_store_4d(&tm_dx, sbase + (dx_stage(l) + h) * PANEL, 32 * h, l, t0, bh);
            bulk_commit();
            // J and H (next) take the dv and dX staging tiles: their stores must have read them
            // before the products' completion releases the epilogue
            bulk_wait_read();
            mma_commit(smem_u32(&mbar[3]));
        }
        wait_all(3, 0);
        fence_after_sync();
        // J_b[m][j] = (w_m . dout_j) D_{j,m} (j >= m), H_b[m][j] = (w_m . z_j) D_{j,m} (j > m); thread
        // (quad, sub): row `row` of group sub & 1 (block b = 2 (sub & 1) + row / 64), the 32 columns
        // of half sub >> 1
        {
            const int g = sub & 1, h2 = sub >> 1, b = 2 * g + (row >> 6), m = row & 63;
            if ((g == 0 || R >= 2) && b <= R) {
                float v[32];
                const uint32_t col = TM_C + 128 * g + (uint32_t)(h2 * 32);
                tmem_ld(tmem + col + lane_off, v);
                decay_col(v, s_lam, m, 32 * h2, true);
                st_row_h(P(J0 + b), m, 32 * h2, v);
                tmem_ld(tmem + col + 64 + lane_off, v);
                decay_col(v, s_lam, m, 32 * h2, false);
                st_row_h(P(H0 + b), m, 32 * h2, v);
            }
        }
        // the operands of the next products, scaled in place (the Grams have read them)
        panel_scale(P(VT), s_colf, tid);
        for (int l = 0; l < R; ++l) panel_scale(P(X0 + l), s_colf, tid);
        panel_scale(P(DO), s_gam, tid);
        panel_scale(P(Z), s_gam, tid);
        fence_async_smem();
        fence_before_sync();
        __syncthreads();
        // ---- dKw = diag(colf) Vw G + J Q - H diag(beta) K;  [dq; extra] = [Gamma dO; Gamma Z] S + [J^T; H^T] Kw --
        if (tid == 0) {
            fence_after_sync();
            const uint32_t id = idesc_f16(128, 64, 0, 1);
            for (int g = 0; g < (R >= 2 ? 2 : 1); ++g) {
                const uint32_t d = tmem + TM_D + 64 * g;
                mma_k64(d, km(dbase, (g == 0 ? VT : X0 + 1) * PANEL), false, mn(dbase, GB * PANEL, PANEL), true, id, false);
                mma_k64(d, km(dbase, (J0 + 2 * g) * PANEL), false, mn(dbase, Q * PANEL, PANEL), true, id, true);
                mma_k64(d, km(dbase, (H0 + 2 * g) * PANEL), false, mn(dbase, NBK * PANEL, PANEL), true, id, true);
            }
            mma_k64(tmem + TM_E, km(dbase, DO * PANEL), false, mn(dbase, S0 * PANEL, PANEL), true, id, false);
            for (int b = 0; b <= R; ++b)
                mma_k64(tmem + TM_E, mn(dbase, (J0 + b) * PANEL, (H0 - J0) * PANEL), true,
                        mn(dbase, (b == 0 ? K : U0 + b - 1) * PANEL, PANEL), true, idesc_f16(128, 64, 1, 1), true);
            mma_commit(smem_u32(&mbar[4]));
        }
        wait_all(4, 0);
        fence_after_sync();
        // the outputs go out by TMA stores of fp32 tiles staged in the tiles the products have read
        // (rows past the sequence's end are clipped by the tensor maps)
        {
            const int n0 = CW * sub;
            float v[CW];
            if (row < 64) {
                const int i = row;
                tmem_ld(tmem + TM_D + lane_off + (uint32_t)n0, v);  // the write part of dk
                st_tile_f(P(DKW), i, n0, v);
                if (R >= 2) {
                    tmem_ld(tmem + TM_D + 64 + lane_off + (uint32_t)n0, v);
                    st_tile_f(P(DUS + 2), i, n0, v);
                }
                tmem_ld(tmem + TM_E + lane_off + (uint32_t)n0, v);  // dq
                st_tile_f(P(DQS), i, n0, v);
                if (i < n) {
                    float qv[CW];
                    ld_row_h(P(Q), i, n0, qv);
                    float part = 0.f;
#pragma unroll
                    for (int q = 0; q < CW; ++q) part = fmaf(qv[q], v[q], part);
                    s_qdq[sub * 64 + i] = part;
                }
            } else {
                const int i = row - 64;
                if (R >= 1) {
                    tmem_ld(tmem + TM_D + lane_off + (uint32_t)n0, v);
                    st_tile_f(P(DUS), i, n0, v);
                }
                if (R >= 3) {
                    tmem_ld(tmem + TM_D + 64 + lane_off + (uint32_t)n0, v);
                    st_tile_f(P(DUS + 4), i, n0, v);
                }
            }
        }
        fence_async_smem();
        __syncthreads();
        if (tid == 0) {
            for (int h = 0; h < 2; ++h) {
                tma_store_3d(&tm_dq, sbase + (DQS + h) * PANEL, 32 * h, t0, bh);
                for (int l = 0; l < R; ++l) tma_store_4d(&tm_du, sbase + (DUS + 2 * l + h) * PANEL, 32 * h, l, t0, bh);
            }
            bulk_commit();
        }
        if (row >= 64) {  // dk = (dKw)_0 - beta (Gamma Z S + H^T Kw), in place
            const int i = row - 64, n0 = CW * sub;
            float v[CW], w[CW];
            tmem_ld(tmem + TM_E + lane_off + (uint32_t)n0, v);
            ld_tile_f(P(DKW), i, n0, w);
            const float b = s_beta[i];
#pragma unroll
            for (int q = 0; q < CW; ++q) v[q] = w[q] - b * v[q];
            st_tile_f(P(DKW), i, n0, v);
        }
        fence_async_smem();
        __syncthreads();
        if (tid == 0) {
            for (int h = 0; h < 2; ++h) tma_store_3d(&tm_dk, sbase + (DKW + h) * PANEL, 32 * h, t0, bh);
            bulk_commit();
        }
        // alpha_i dalpha_i = F0 + sum_{j >= i} (q_j.dq_j - sigma_j)
        if (warp == 0) {
            auto term = [&](int i) {
                float sg = 0.f;
#pragma unroll
                for (int k = 0; k < 16; ++k) sg += s_sig[k * 64 + i];
                return (s_qdq[i] + s_qdq[64 + i]) + (s_qdq[128 + i] + s_qdq[192 + i]) - sg;
            };
            const int i0 = 2 * lane, i1 = i0 + 1;
            const float a0 = i0 < n ? term(i0) : 0.f;
            const float a1 = i1 < n ? term(i1) : 0.f;
            float x = a0 + a1;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const float y = __shfl_down_sync(0xffffffffu, x, off);
                if (lane + off < 32) x += y;
            }
            float F0 = 0.f;
#pragma unroll
            for (int k = 0; k < NT / 32; ++k) F0 += s_Fw[k];
            if (i0 < n) p.dalpha[tok0 + i0] = (F0 + x) / p.alpha[tok0 + i0];
            if (i1 < n) p.dalpha[tok0 + i1] = (F0 + x - a0) / p.alpha[tok0 + i1];
        }
    } while (0);

    // drain (after an expired wait): let the copies and products in flight land, bounded
    if (tid == 0 && abort_s) {
        const uint64_t drain_ns = 1000000000ull;
        if (pend_ld) (void)mbar_wait(mb_ld, 0, drain_ns);
        const uint32_t mb_drain = smem_u32(&mbar[5]);
        mma_commit(mb_drain);
        (void)mbar_wait(mb_drain, 0, drain_ns);
    }
    if (tid == 0) bulk_wait_read();  // the output stores have read their tiles
    fence_before_sync();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, 512);
}

}  // namespace bt

// ---------------------------------------------------------------------------------------------------------
namespace {

PFN_cuTensorMapEncodeTiled_v12000 bt_encoder()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = (PFN_cuTensorMapEncodeTiled_v12000)ptr;
    }
    return fn;
}

bool bt_encode(CUtensorMap *m, const void *base, int rank, const cuuint64_t *dims, const cuuint64_t *strides_bytes,
               const cuuint32_t *box, CUtensorMapDataType type = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16)
{
    auto fn = bt_encoder();
    if (!fn) return false;
    cuuint32_t es[5] = {1, 1, 1, 1, 1};
    return fn(m, type, (cuuint32_t)rank, const_cast<void *>(base), dims, strides_bytes, box,
              es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// workspace of the chunked backward: maps (4 x fp32 64 x 64 per chunk), the stash (8 fp16 panels per
// chunk), the chunk states and cotangents, dX, and the convolution scratch of the token-local kernels
struct BtCarve {
    float *mapA, *mapAT, *mapB, *mapBb, *Sst, *Gst, *dX, *dH, *dWp;
    __half *stash;
};

size_t bt_carve(const Shape &s, void *base, BtCarve *out)
{
    BtCarve scratch{};
    BtCarve *w = out ? out : &scratch;
    const size_t chunks = (size_t)s.BH * s.NC, dd = (size_t)s.dk * s.dv, th = (size_t)s.BH * s.T;
    const int ntile = backward_conv_tiles(s.T);
    const size_t bytes[10] = {chunks * dd * 4, chunks * dd * 4, chunks * dd * 4, chunks * dd * 4,
                              (size_t)s.BH * (s.NC + 1) * dd * 4, chunks * dd * 4,
                              th * (size_t)(s.R > 0 ? s.R : 1) * s.dv * 4, th * s.dv * 4,
                              (size_t)s.BH * ntile * 4 * s.dv * 4, chunks * bt::STASH * bt::PANEL};
    void **dst[10] = {(void **)&w->mapA, (void **)&w->mapAT, (void **)&w->mapB, (void **)&w->mapBb, (void **)&w->Sst,
                      (void **)&w->Gst, (void **)&w->dX, (void **)&w->dH, (void **)&w->dWp, (void **)&w->stash};
    size_t off = 0;
    for (int i = 0; i < 10; ++i) {
        if (base) *dst[i] = static_cast<char *>(base) + off;
        off += (bytes[i] + 1023) & ~(size_t)1023;
    }
    return off;
}

}  // namespace

bool backward_tc_supported(const Shape &s, prism_dtype io)
{
    return io == PRISM_BF16 && s.dk == bt::D && s.dv == bt::D && s.L >= 1 && s.L <= 1 + bt::RMAX;
}

size_t backward_tc_workspace_bytes(const Shape &s) { return bt_carve(s, nullptr, nullptr); }

cudaError_t backward_tc_prepare()
{
    cudaError_t e;
    if ((e = cudaFuncSetAttribute(bt::maps_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bt::mk::SMEM)) !=
        cudaSuccess)
        return e;
    if ((e = cudaFuncSetAttribute(bt::scan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bt::SCAN_SMEM_LAUNCH)) !=
        cudaSuccess)
        return e;
    return cudaFuncSetAttribute(bt::grad_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bt::gk::SMEM);
}

cudaError_t backward_tc(const Shape &s, const BackwardArgs &a, void *ws, int *d_status, long long wait_ns,
                        KernelTimer &tm)
{
    using namespace bt;
    BtCarve w{};
    bt_carve(s, ws, &w);
    cudaStream_t st = tm.stream;
    CUtensorMap mq, mk_, mv, mu;
    {
        const cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)s.T, (cuuint64_t)s.BH};
        const cuuint64_t str[2] = {(cuuint64_t)D * 2, (cuuint64_t)s.T * D * 2};
        const cuuint32_t box[3] = {64, 64, 1};
        if (!bt_encode(&mq, a.q, 3, dims, str, box) || !bt_encode(&mk_, a.k, 3, dims, str, box) ||
            !bt_encode(&mv, a.v, 3, dims, str, box))
            return cudaErrorInvalidValue;
    }
    if (s.R > 0) {
        const cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)s.R, (cuuint64_t)s.T, (cuuint64_t)s.BH};
        const cuuint64_t str[3] = {(cuuint64_t)D * 2, (cuuint64_t)s.R * D * 2, (cuuint64_t)s.T * s.R * D * 2};
        const cuuint32_t box[4] = {64, 1, 64, 1};
        if (!bt_encode(&mu, a.u, 4, dims, str, box)) return cudaErrorInvalidValue;
    } else {
        mu = mk_;  // never read with L = 1
    }
    // the fp32 outputs the gradient kernel writes by TMA stores: 32-column boxes of one chunk
    CUtensorMap mdq, mdk, mdu, mdv, mdx;
    {
        const cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)s.T, (cuuint64_t)s.BH};
        const cuuint64_t str[2] = {(cuuint64_t)D * 4, (cuuint64_t)s.T * D * 4};
        const cuuint32_t box[3] = {32, 64, 1};
        if (!bt_encode(&mdq, a.dq, 3, dims, str, box, CU_TENSOR_MAP_DATA_TYPE_FLOAT32) ||
            !bt_encode(&mdk, a.dk, 3, dims, str, box, CU_TENSOR_MAP_DATA_TYPE_FLOAT32) ||
            !bt_encode(&mdv, a.dv, 3, dims, str, box, CU_TENSOR_MAP_DATA_TYPE_FLOAT32))
            return cudaErrorInvalidValue;
    }
    if (s.R > 0) {
        const cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)s.R, (cuuint64_t)s.T, (cuuint64_t)s.BH};
        const cuuint64_t str[3] = {(cuuint64_t)D * 4, (cuuint64_t)s.R * D * 4, (cuuint64_t)s.T * s.R * D * 4};
        const cuuint32_t box[4] = {32, 1, 64, 1};
        if (!bt_encode(&mdu, a.du, 4, dims, str, box, CU_TENSOR_MAP_DATA_TYPE_FLOAT32) ||
            !bt_encode(&mdx, w.dX, 4, dims, str, box, CU_TENSOR_MAP_DATA_TYPE_FLOAT32))
            return cudaErrorInvalidValue;
    } else {
        mdu = mdx = mdq;  // never written with L = 1
    }
    // the maps kernel's fp32 chunk maps, [chunks x 64][64]
    CUtensorMap mma_, mmat, mmb, mmbb;
    {
        const cuuint64_t dims[2] = {(cuuint64_t)D, (cuuint64_t)s.BH * s.NC * 64};
        const cuuint64_t str[1] = {(cuuint64_t)D * 4};
        const cuuint32_t box[2] = {32, 64};
        if (!bt_encode(&mma_, w.mapA, 2, dims, str, box, CU_TENSOR_MAP_DATA_TYPE_FLOAT32) ||
            !bt_encode(&mmat, w.mapAT, 2, dims, str, box, CU_TENSOR_MAP_DATA_TYPE_FLOAT32) ||
            !bt_encode(&mmb, w.mapB, 2, dims, str, box, CU_TENSOR_MAP_DATA_TYPE_FLOAT32) ||
            !bt_encode(&mmbb, w.mapBb, 2, dims, str, box, CU_TENSOR_MAP_DATA_TYPE_FLOAT32))
            return cudaErrorInvalidValue;
    }
    Params p{};
    p.v = (const __nv_bfloat16 *)a.v;
    p.conv_w = (const __nv_bfloat16 *)a.conv_w;
    p.v_hist = (const __nv_bfloat16 *)a.v_hist;
    p.beta = a.beta;
    p.alpha = a.alpha;
    p.gamma = a.gamma;
    p.eta = a.eta;
    p.p_gain = static_cast<const __nv_bfloat16 *>(a.p_gain);
    p.dout = a.dout;
    p.mapA = w.mapA;
    p.mapAT = w.mapAT;
    p.mapB = w.mapB;
    p.mapBb = w.mapBb;
    p.stash = w.stash;
    p.Sst = w.Sst;
    p.Gst = w.Gst;
    p.dq = a.dq;
    p.dk = a.dk;
    p.dv = a.dv;
    p.dbeta = a.dbeta;
    p.dalpha = a.dalpha;
    p.du = a.du;
    p.dX = w.dX;
    p.status = d_status;
    p.H = s.H;
    p.T = s.T;
    p.R = s.R;
    p.NC = s.NC;
    p.wait_ns = wait_ns > 0 ? (unsigned long long)wait_ns : 100000000ull;
    const unsigned nchunks = (unsigned)(s.BH * s.NC);

    cudaLaunchAttribute pdl[1];
    pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    pdl[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.stream = st;
    cfg.attrs = pdl;
    cfg.numAttrs = 1;
    cudaError_t e;

    tm.begin("bwd_maps");
    cfg.gridDim = dim3(nchunks);
    cfg.blockDim = dim3(NT);
    cfg.dynamicSmemBytes = mk::SMEM;
    cfg.numAttrs = 0;  // the previous kernel on the stream may be anything
    e = cudaLaunchKernelEx(&cfg, maps_kernel, mq, mk_, mv, mu, mma_, mmat, mmb, mmbb, p);
    tm.end();
    if (e != cudaSuccess) return e;
    cfg.numAttrs = 1;
    tm.begin("bwd_chunk_scan");
    cfg.gridDim = dim3(D / SC_ROWS, s.BH, 2);
    cfg.blockDim = dim3(SCAN_NT + 32);
    cfg.dynamicSmemBytes = SCAN_SMEM_LAUNCH;
    e = cudaLaunchKernelEx(&cfg, scan_kernel, (const float *)w.mapA, (const float *)w.mapAT, (const float *)w.mapB,
                           (const float *)w.mapBb, a.S_init, a.dS_final, w.Sst, w.Gst, a.dS_init, s.NC, d_status,
                           p.wait_ns);
    tm.end();
    if (e != cudaSuccess) return e;
    tm.begin("bwd_grad");
    cfg.gridDim = dim3(nchunks);
    cfg.blockDim = dim3(NT);
    cfg.dynamicSmemBytes = gk::SMEM;
    e = cudaLaunchKernelEx(&cfg, grad_kernel, mq, mk_, mu, mdq, mdk, mdu, mdv, mdx, p);
    tm.end();
    if (e != cudaSuccess) return e;
    return backward_token_local(s, PRISM_BF16, a, w.dX, w.dH, w.dWp, tm);
}

}  // namespace prism
