// Tensor-core path of the PRISM memory-recurrence forward (sm_103a: tcgen05 + TMA).
//
// Shapes: dk = dv = 64, 1 <= L <= 4, bf16 io, chunks of C = 64 tokens.
//
// Three kernels:
//   segment  one CTA per (sequence, segment of consecutive chunks).  For every chunk it runs
//            the prep (anchor, gain, residual chain), the Gram tiles, the UT/WY solve, the WY
//            factors and the chunk's state map S -> S M_c + N_c, and carries the augmented state
//            Z = [N; M] (the segment's map S_start -> S_start M + N) through the segment.  The
//            output of a chunk is o = o0 + Qhat S_start^T: o0 and Qhat are exact given Z, so the
//            first segment of a sequence that starts from S = 0 writes o directly and the others
//            stash (o0, Qhat) for the fix-up.  A sequence continued from an earlier call starts
//            from S_init, with the anchor's left context v_{-3..-1} in place of the zero halo.
//   combine  per sequence, S_start of segment p from S_init (or 0) and the maps of segments
//            0..p-1 (associative combine of the input-only affine maps, notes on PRISM
//            section 2.1); optionally the state after the last token.
//   fixup    o = o0 + Qhat S_start^T for the chunks of the stashing segments (tcgen05, one CTA per chunk pair).
//
// Chunk algebra (local index i, j; lambda_i = sum_{m<=i} ln alpha_m; lc = lambda_{C-1};
// D_ij = e^{lambda_i - lambda_j} (j <= i), colf_j = e^{lc - lambda_j} <= 1, Gamma_i = e^{lambda_i}):
//   A_ij  = beta_i D_ij k_i.k_j                        (j < i)   -> T = (I + A)^{-1}   (fp32 solve)
//   PK_l  = D_ij k_i.u_{j,l} (j < i);  PQ_l = D_ij q_i.u_{j,l}, G = D_ij q_i.k_j (j <= i)  (decayed
//           scores, computed and stored transposed, [j][i], from Grams with key/direction rows)
//   X_l   = x_{j,l}                                    (x = gamma g (.) r, the prep)
//   K'    = diag(colf) K,  U'_l = diag(colf) U_l       (the state-side key and direction tiles)
//   RHS   = diag(beta) (V - sum_l PK_l X_l)
//   [U'^T; W^T] = [RHS | diag(beta Gamma) K]^T T^T  = UW
//   D4    = UW G^T + [X^T; 0] PQ^T = [O_loc^T ; (G W)^T]
//   D5    = UW K' + [X^T; 0] U'   = [N_c ; W^T K']
//   Qt    = Q~^T = diag(Gamma) Q^T - (G W)^T,   M_c = Gamma_C I - W^T K'
//   Z    <- Z M_c + [N_c; 0],   [o0^T ; Qhat^T] = Z Qt + [O_loc^T ; 0]   (Z before the update)
// Every decay that a product needs is applied in fp32 before an operand is rounded: D_ij on the
// score tiles (as e^{lambda_i - lc} e^{lc - lambda_j} while the chunk's total decay is within fp32
// range, else one exponential per element), colf on the state side.  No fp16 operand carries a
// factor that a later step multiplies back up, so an operand that underflows only drops a
// contribution below fp16's range, however strong the decay.
// All matrix products above run on tcgen05.mma (fp16 operands in 128B-swizzled shared memory,
// fp32 accumulators in tensor memory); operands come from TMA or from the epilogues.  The Gram
// runs on the bf16 input tiles; K and U are then converted to fp16 in place, scaled by colf, for
// the state-side products: fp16's 10-bit mantissa keeps the computed operands (scores, X, T,
// U'/W, Q~, M_c, Z) 8x closer to fp32 than bf16 would, at the same tensor-core rate.
#include <cuda_fp16.h>
#include <cudaTypedefs.h>

#include "prism_internal.h"
#include "tc_ptx.h"

// Developer tracing: with -DPRISM_PHASE_TIMERS the segment kernel accumulates clock64()
// cycles per phase of its chunk loop (thread 0 of every CTA) into prism_tc_phase_cycles.
#ifdef PRISM_PHASE_TIMERS
constexpr int kPhaseSlots = 24;
__device__ unsigned long long prism_tc_phase_cycles[kPhaseSlots];
#define PHASE_MARK(k)                                         \
    do {                                                      \
        if (threadIdx.x == 0) {                               \
            const long long now_ = clock64();                 \
            ph_acc_s[k] += (unsigned long long)(now_ - ph_last); \
            ph_last = now_;                                   \
        }                                                     \
    } while (0)
#else
#define PHASE_MARK(k) \
    do {              \
    } while (0)
#endif

namespace prism {
namespace tc {

constexpr int C = kChunk;
constexpr int D = 64;       // dk = dv
constexpr int RMAX = 3;     // refinement levels handled (L <= 4)
constexpr int NT = 512;     // threads per CTA: 16 warps, 4 per TMEM lane quarter
constexpr int CW = 64 / (NT / 128);  // columns of a 64-column TMEM block each thread handles
constexpr uint32_t TILE = 8192;  // 64 rows x 128 B

// shared memory map (bytes from a 1024-aligned base)
constexpr uint32_t OFF_V0 = 0;                   // two V stages, 72 rows x 128 B (8-row halo), unswizzled
constexpr uint32_t VBYTES = 72 * 128;
constexpr uint32_t OFF_V1 = OFF_V0 + 10240;
constexpr uint32_t OFF_Q = OFF_V1 + 10240;        // Q tile, then K, U0..U2 (contiguous: [Q;K] and [K;U] operands;
constexpr uint32_t OFF_K = OFF_Q + TILE;          // the tile below Q is the first atom of the Q^T copy)
constexpr uint32_t OFF_U = OFF_K + TILE;
constexpr uint32_t OFF_E = OFF_U + RMAX * TILE;   // [PK0|PQ0^T|PK1|PQ1^T|PK2|PQ2^T|G^T]; later Qt, Mc
constexpr uint32_t OFF_G = OFF_E + 6 * TILE;
constexpr uint32_t OFF_AKK = OFF_E + 7 * TILE;    // A (fp32, row stride LDA); later UW
constexpr uint32_t LDA = 68;    // row stride (floats) of A and T32 (float4 rows, conflict-free fragments)
constexpr uint32_t OFF_T32 = OFF_AKK + 64 * LDA * 4;
constexpr uint32_t OFF_TB = OFF_T32 + 64 * LDA * 4;  // bf16 identity (written once): B of the Q^T copy
constexpr uint32_t OFF_TF = OFF_E + 2 * TILE;        // T (fp16), over PK_1^T (free once MX completed)
constexpr uint32_t OFF_XS = OFF_TB + TILE;            // X0..X2
constexpr uint32_t OFF_ZERO = OFF_XS + RMAX * TILE;   // zero tile
constexpr uint32_t OFF_ZA = OFF_ZERO + TILE;          // Z (128 rows, bf16, K-major)
constexpr uint32_t OFF_BGK = OFF_ZA + 2 * TILE;       // diag(beta Gamma) K (fp16 tile)
constexpr uint32_t OFF_SC = OFF_BGK + TILE;           // per-token scalars
constexpr uint32_t SC_SET = 64 * 6 + 64 * RMAX * 2;         // per-token scalars of one chunk
constexpr uint32_t XTMP_FLOATS = 4 * 256;                     // solve scratch: 4 warps x 32 x 8
constexpr uint32_t SC_FLOATS = 2 * SC_SET + XTMP_FLOATS;       // two chunks' sets + solve scratch
constexpr uint32_t SMEM_BYTES = OFF_SC + SC_FLOATS * 4 + 1024;  // + alignment slack

static_assert(OFF_Q % 1024 == 0 && OFF_Q >= TILE && OFF_E % 1024 == 0 && OFF_AKK % 1024 == 0 && OFF_TB % 1024 == 0 &&
                  OFF_XS % 1024 == 0 && OFF_ZA % 1024 == 0 &&
                  OFF_BGK % 1024 == 0,
              "align");
static_assert(SMEM_BYTES <= 232448, "shared memory budget");
// the solve's scratch: level 1 uses 4 warps x 16 x 8 floats, level 2 4 warps x 32 x 8 floats
static_assert(4 * 128 <= XTMP_FLOATS && 4 * 256 <= XTMP_FLOATS, "solve scratch");

// TMEM column map
constexpr uint32_t TM_D1 = 0, TM_D2 = 256, TM_D3 = 320, TM_D5 = 384, TM_D4 = 448, TM_D7 = 0, TM_D6 = 64;
constexpr uint32_t TM_QT = 128;  // Q^T (lanes 64..127), copied from P3 to E4 in the Gram's upper columns
static_assert(TM_D4 == TM_D5 + 64 && TM_D6 == TM_D7 + 64, "D5|D4 and D7|D6 are written by one N = 128 MMA each");

struct SegParams {
    const float *beta, *alpha, *gamma, *eta;
    const __nv_bfloat16 *conv_w;
    void *out;              // bf16, or fp32 when out_f32
    float *zsum;            // [BH][P][128][64]
    void *stash_o;          // [BH][NC][64][64]  o0 (token-major; fp32 for fp32 output, else fp16)
    __half *stash_q;        // [BH][NC][64][64]  Qhat (token-major)
    const __nv_bfloat16 *v_hist;  // [BH][3][64] v_{-3..-1} of the sequence, or null (zeros)
    const __nv_bfloat16 *p_gain;  // [BH][T][R][64] gains of the non-linear residual chain, or null (linear)
    int *status;
    int H, T, R, NC, P;
    int out_f32;
    int has_init;           // the sequence starts from a given state: segment 0 is tracked too
    unsigned long long wait_ns;  // bound of every wait on an mbarrier
};

__device__ __forceinline__ void set_status(int *st, int code) { atomicCAS(st, 0, code); }

// compile-time flag for code paths chosen by a uniform runtime branch
template <bool B>
struct BoolTag {
    static constexpr bool value = B;
};

__device__ __forceinline__ uint32_t pack2(float a, float b)
{
    const __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<const uint32_t *>(&h);
}

// write N consecutive fp32 values (columns col0..col0+N-1 of row `row`, col0 a multiple of 8)
// as fp16 into a [rows][64] SW128 tile
template <int N>
__device__ __forceinline__ void st_row(uint8_t *tile, int row, int col0, const float (&v)[N])
{
#pragma unroll
    for (int g = 0; g < N / 8; ++g) {
        uint4 w;
        w.x = pack2(v[8 * g + 0], v[8 * g + 1]);
        w.y = pack2(v[8 * g + 2], v[8 * g + 3]);
        w.z = pack2(v[8 * g + 4], v[8 * g + 5]);
        w.w = pack2(v[8 * g + 6], v[8 * g + 7]);
        *reinterpret_cast<uint4 *>(tile + sw128(row, col0 + 8 * g)) = w;
    }
}

// Descriptor of the tile at byte offset `off` of the CTA's 1024-aligned shared-memory base,
// built by adding the offset fields to a descriptor of the base (all fields stay in range).
__device__ __forceinline__ uint64_t dsc(uint64_t base, uint32_t off, uint32_t lbo, uint32_t sbo)
{
    return base + (uint64_t)(off >> 4) + ((uint64_t)(lbo >> 4) << 16) + ((uint64_t)(sbo >> 4) << 32);
}

__device__ __forceinline__ float ld_bf(const uint8_t *tile, int row, int col)
{
    return __bfloat162float(*reinterpret_cast<const __nv_bfloat16 *>(tile + sw128(row, col)));
}

// Gain g = GELU'(a) = Phi(a) + a phi(a) and Phi(a), for the exact-erf GELU.  Phi uses the
// rational approximation of erf from Abramowitz & Stegun, Handbook of Mathematical Functions,
// formula 7.1.26 (|error| <= 1.5e-7), which shares the Gaussian factor e^{-a^2/2} with phi.
__device__ __forceinline__ void gelu_gain(float a, float &g, float &Phi)
{
    const float x = fabsf(a) * 0.70710678118654752f;
    const float t = __fdividef(1.f, fmaf(0.3275911f, x, 1.f));
    const float E = __expf(-0.5f * a * a);
    float poly = fmaf(t, 1.061405429f, -1.453152027f);
    poly = fmaf(t, poly, 1.421413741f);
    poly = fmaf(t, poly, -0.284496736f);
    poly = fmaf(t, poly, 0.254829592f);
    const float erfx = 1.f - poly * t * E;
    Phi = 0.5f + copysignf(0.5f * erfx, a);
    g = fmaf(a, 0.39894228040143268f * E, Phi);
}

// GELU(z) = z Phi(z), Phi from the same approximation of erf as gelu_gain
__device__ __forceinline__ float gelu_value(float z)
{
    float g, Phi;
    gelu_gain(z, g, Phi);
    return z * Phi;
}

// The lane's fragment coordinates of a warp-level m16n8 MMA: row group gq = lane / 4, column
// pair index tq = lane % 4.
struct Frag {
    int gq, tq;  // lane / 4, lane % 4
};
// m16n8k16 fp16 fragments of fp32 matrices in shared memory (row-major, row stride ld; A: 16 rows
// from r0, 16 columns from k0; B: 16 rows (k) from k0, 8 columns (n) from n0), rounded to fp16
// (T enters the tensor-core products as fp16 anyway, and fp16 keeps tf32's 10 mantissa bits), and
// D += A B with fp32 accumulation.  The C fragment: rows gq and gq + 8, columns 2 tq, 2 tq + 1.
__device__ __forceinline__ void frag_a16(const Frag &f, const float *M, int ld, int r0, int k0, uint32_t (&a)[4])
{
    const float *p = M + (r0 + f.gq) * ld + k0 + 2 * f.tq;
    a[0] = pack2(p[0], p[1]);
    a[1] = pack2(p[8 * ld], p[8 * ld + 1]);
    a[2] = pack2(p[8], p[9]);
    a[3] = pack2(p[8 * ld + 8], p[8 * ld + 9]);
}
__device__ __forceinline__ void frag_b16(const Frag &f, const float *M, int ld, int k0, int n0, uint32_t &b0, uint32_t &b1)
{
    const float *p = M + (k0 + 2 * f.tq) * ld + n0 + f.gq;
    b0 = pack2(p[0], p[ld]);
    b1 = pack2(p[8 * ld], p[9 * ld]);
}
__device__ __forceinline__ void mma_h16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1)
{
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void frag_c_store(const Frag &f, float *M, int ld, int r0, int n0, const float (&c)[4], float sgn)
{
    float *p = M + (r0 + f.gq) * ld + n0 + 2 * f.tq;
    p[0] = sgn * c[0];
    p[1] = sgn * c[1];
    p[8 * ld] = sgn * c[2];
    p[8 * ld + 1] = sgn * c[3];
}

// in-place bf16 -> fp16 conversion of `bytes` bytes of [64][64] tiles (layout unchanged), each
// row r of every tile scaled by scale[r] (a 16-byte group never leaves its row under the swizzle)
__device__ __forceinline__ void tiles_bf16_to_f16(uint8_t *base, uint32_t bytes, int t, int nthreads,
                                                  const float *scale)
{
    for (uint32_t e = t; e < bytes / 16; e += nthreads) {
        uint4 w = reinterpret_cast<uint4 *>(base)[e];
        const float sc = scale[(e >> 3) & 63];
        uint32_t *pw = &w.x;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162 *>(&pw[q]);
            const float2 f = __bfloat1622float2(b);
            pw[q] = pack2(sc * f.x, sc * f.y);
        }
        reinterpret_cast<uint4 *>(base)[e] = w;
    }
}

// prep of one chunk (P1): anchor, gain and residual chain -> X tiles, two channels x 4 tokens per
// thread, from V stage `stg` and the chunk's per-token scalars `pset`.  Kept out of line: the
// segment kernel calls it at two places, and one copy of its code keeps the loop body smaller.
template <bool kNonlinear>
__device__ __noinline__ void prep_chunk(uint8_t *sm, const float *pset, const __nv_bfloat162 *cw2, int stg, int R,
                                        const uint32_t *pg, int n)
{
    const int tid = threadIdx.x;
    const float2 w0 = __bfloat1622float2(cw2[0 * (D / 2)]);
    const float2 w1 = __bfloat1622float2(cw2[1 * (D / 2)]);
    const float2 w2 = __bfloat1622float2(cw2[2 * (D / 2)]);
    const float2 w3 = __bfloat1622float2(cw2[3 * (D / 2)]);
    const float *p_gc = pset + 384, *p_eta = pset + 384 + 64 * RMAX;
    const __nv_bfloat162 *vb = reinterpret_cast<const __nv_bfloat162 *>(sm + (stg ? OFF_V1 : OFF_V0));
    const int cp = tid & 31, tg = tid >> 5;  // channel pair, token group
    constexpr int TPT = 64 / (NT / 32);     // tokens per thread
    // the non-linear chain's gains of this thread's tokens, all loads issued before any is used
    uint32_t pz[TPT][RMAX];
    if constexpr (kNonlinear) {
#pragma unroll
        for (int k = 0; k < TPT; ++k) {
            const int i = tg + (NT / 32) * k;
#pragma unroll
            for (int l = 0; l < RMAX; ++l) pz[k][l] = (i < n && l < R) ? pg[(size_t)(i * R + l) * (D / 2) + cp] : 0u;
        }
    }
#pragma unroll
    for (int k = 0; k < TPT; ++k) {
        const int i = tg + (NT / 32) * k;
        const float2 v0 = __bfloat1622float2(vb[(i + 8) * 32 + cp]);
        const float2 v1 = __bfloat1622float2(vb[(i + 7) * 32 + cp]);
        const float2 v2 = __bfloat1622float2(vb[(i + 6) * 32 + cp]);
        const float2 v3 = __bfloat1622float2(vb[(i + 5) * 32 + cp]);
        float gcl[RMAX], etl[RMAX];
#pragma unroll
        for (int l = 0; l < RMAX; ++l) {
            gcl[l] = p_gc[i * RMAX + l];
            etl[l] = p_eta[i * RMAX + l];
        }
        const float a0 = fmaf(w0.x, v0.x, fmaf(w1.x, v1.x, fmaf(w2.x, v2.x, w3.x * v3.x)));
        const float a1 = fmaf(w0.y, v0.y, fmaf(w1.y, v1.y, fmaf(w2.y, v2.y, w3.y * v3.y)));
        float g0, g1, Phi0, Phi1;
        gelu_gain(a0, g0, Phi0);
        gelu_gain(a1, g1, Phi1);
        float r0 = v0.x - a0 * Phi0, r1 = v0.y - a1 * Phi1;
        uint8_t *xs = sm + OFF_XS + sw128(i, 2 * cp);
        if constexpr (kNonlinear) {  // non-linear chain: delta = GELU(p r), x = gamma delta, r <- r - delta
#pragma unroll
            for (int l = 0; l < RMAX; ++l) {
                if (l < R) {
                    const float2 pf = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&pz[k][l]));
                    const float d0 = gelu_value(pf.x * r0), d1 = gelu_value(pf.y * r1);
                    *reinterpret_cast<uint32_t *>(xs + l * TILE) = pack2(gcl[l] * d0, gcl[l] * d1);
                    r0 -= d0;
                    r1 -= d1;
                }
            }
        } else {
#pragma unroll
            for (int l = 0; l < RMAX; ++l) {
                if (l < R) *reinterpret_cast<uint32_t *>(xs + l * TILE) = pack2(gcl[l] * g0 * r0, gcl[l] * g1 * r1);
                r0 *= 1.f - etl[l] * g0;
                r1 *= 1.f - etl[l] * g1;
            }
        }
    }
}

// barrier over `n` threads (whole warps) of the CTA; ids 1.. (0 is __syncthreads')
__device__ __forceinline__ void named_bar(int id, int n) { asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory"); }

// ---------------------------------------------------------------------------------------------
__global__ void __launch_bounds__(NT, 1)
    segment_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_u, SegParams p)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    __shared__ uint32_t tmem_base_s;
    __shared__ __align__(8) uint64_t mbar[4];  // 0: MMA, 1: Q/K/U, 2,3: V stages
    __shared__ int abort_s;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int quad = warp & 3, sub = warp >> 2;  // TMEM lane quarter, epilogue column slice
    const int row = quad * 32 + lane;  // TMEM lane owned in epilogues
    const int bh = blockIdx.x / p.P, seg = blockIdx.x % p.P;
    const int h = bh % p.H;
    const int R = p.R;
    const int c_begin = (int)(((long long)seg * p.NC) / p.P);
    const int c_end = (int)(((long long)(seg + 1) * p.NC) / p.P);
    // a tracked segment carries M (the map's linear part) and stashes o0/Qhat for the fix-up;
    // only the first segment of a sequence that starts from S = 0 can write o directly
    const bool tracked = seg > 0 || p.has_init;

    float *sc = reinterpret_cast<float *>(sm + OFF_SC);
    // per-token scalars, one set per chunk parity (the next chunk's set is filled while the
    // state-side MMAs of the current one run):
    //   beta | lambda | rowf = e^{lambda_i - lc} | colf = e^{lc - lambda_i} | Gamma_i | beta_i Gamma_i
    //   | gamma [64][RMAX] | eta [64][RMAX]
    float *s_xtmp = sc + 2 * SC_SET;  // XTMP_FLOATS of scratch for the solve

    const uint32_t sbase = smem_u32(sm);
    const uint64_t dbase = sdesc(sbase, 0, 0);
    const uint32_t mb_mma = smem_u32(&mbar[0]), mb_qku = smem_u32(&mbar[1]);
    const uint32_t mb_v[2] = {smem_u32(&mbar[2]), smem_u32(&mbar[3])};

    if (tid == 0) {
        abort_s = 0;
        mbar_init(mb_mma, 1);
        mbar_init(mb_qku, 1);
        mbar_init(mb_v[0], 1);
        mbar_init(mb_v[1], 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        prefetch_tmap(&tm_q);
        prefetch_tmap(&tm_k);
        prefetch_tmap(&tm_v);
        prefetch_tmap(&tm_u);
    }
    // zero tile, bf16 identity, and Z = [0; I] (tracked segments) or 0
    for (int e = tid; e < (int)(TILE / 16); e += NT) reinterpret_cast<uint4 *>(sm + OFF_ZERO)[e] = make_uint4(0, 0, 0, 0);
    {
        const int i = tid >> 3, g = tid & 7;  // row i, 16-byte group g (8 columns)
        uint4 w = make_uint4(0, 0, 0, 0);
        if ((i >> 3) == g) reinterpret_cast<__nv_bfloat16 *>(&w)[i & 7] = __float2bfloat16_rn(1.f);
        *reinterpret_cast<uint4 *>(sm + OFF_TB + sw128(i, 8 * g)) = w;
    }
    for (int e = tid; e < 128 * 64; e += NT) {
        const int r = e >> 6, m = e & 63;
        const float z = (tracked && r >= 64 && (r - 64) == m) ? 1.f : 0.f;
        *reinterpret_cast<__half *>(sm + OFF_ZA + sw128(r, m)) = __float2half_rn(z);
    }
    if (warp == 0) tmem_alloc(smem_u32(&tmem_base_s), 512);
    fence_async_smem();
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tmem = tmem_base_s;
    // the set-up above touches no global memory; everything below may depend on the previous
    // kernel in the stream (inputs, or the workspace a previous forward's fix-up still reads)
    grid_dependency_wait();
    allow_dependent_launch();

    // the inputs stream through once: let their L2 lines go first, so that the per-chunk stash
    // (read back by the fix-up) stays in L2
    const uint64_t l2ef = l2_evict_first_policy();
    uint32_t ph_mma = 0, ph_qku = 0, ph_v[2] = {0, 0};
    uint32_t pending = 0;  // issuer's view (thread 0): 1 MMA, 2 Q/K/U load, 4/8 V loads in flight
    const uint32_t qku_bytes = (2 + R) * TILE;

    auto issue_qku = [&](int c) {
        mbar_expect_tx(mb_qku, qku_bytes);
        tma_load_3d_hint(sbase + OFF_Q, &tm_q, mb_qku, 0, c * C, bh, l2ef);
        tma_load_3d_hint(sbase + OFF_K, &tm_k, mb_qku, 0, c * C, bh, l2ef);
        for (int l = 0; l < R; ++l) tma_load_4d_hint(sbase + OFF_U + l * TILE, &tm_u, mb_qku, 0, l, c * C, bh, l2ef);
        pending |= 2u;
    };
    auto issue_v = [&](int c, int stage) {
        mbar_expect_tx(mb_v[stage], VBYTES);
        tma_load_3d_hint(sbase + (stage ? OFF_V1 : OFF_V0), &tm_v, mb_v[stage], 0, c * C - 8, bh, l2ef);
        pending |= 4u << stage;
        if (p.p_gain && R > 0) {  // the non-linear chain's gains of the chunk, read by its prep: into L2 now
            const uint32_t bytes = (uint32_t)min(C, p.T - c * C) * R * D * 2;
            const __nv_bfloat16 *src = p.p_gain + ((size_t)bh * p.T + (size_t)c * C) * R * D;
            asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
        }
    };
    // collective bounded wait on one mbarrier phase (thread 0 polls, then a CTA barrier)
    auto wait_one = [&](uint32_t mb, uint32_t &phase, uint32_t bit) -> bool {
        if (tid == 0) {
            if (mbar_wait(mb, phase, p.wait_ns)) {
                phase ^= 1u;
                pending &= ~bit;
            } else {
                abort_s = 1;
                set_status(p.status, kDevTimeout);
            }
        }
        __syncthreads();
        return abort_s == 0;
    };
    // every thread waits for the MMA barrier itself, so no CTA barrier follows; an expired wait
    // is recorded and the CTA leaves the chunk loop at its next barrier (thread 0 keeps the MMA
    // pending for the drain)
    auto wait_mma = [&]() {
        if (mbar_wait(mb_mma, ph_mma, p.wait_ns)) {
            ph_mma ^= 1u;
            if (tid == 0) pending &= ~1u;
        } else {
            abort_s = 1;
            set_status(p.status, kDevTimeout);
        }
    };

    // the Gram tiles D1 = [K; U_0] [Q; K]^T and D1' = [U_1; U_2] [Q; K]^T on the bf16 input tiles
    // (exact values), committed to the MMA barrier (thread 0)
    auto issue_gram = [&]() {
        const uint32_t id = idesc_bf16(128, 128, 0, 0);
#pragma unroll
        for (int s = 0; s < 4; ++s)
            mma_f16(tmem + TM_D1, dsc(dbase, OFF_K + s * 32, 16, 1024), dsc(dbase, OFF_Q + s * 32, 16, 1024), id,
                    s > 0);
        if (R >= 2)
#pragma unroll
            for (int s = 0; s < 4; ++s)
                mma_f16(tmem + TM_D1 + 128, dsc(dbase, OFF_U + TILE + s * 32, 16, 1024),
                        dsc(dbase, OFF_Q + s * 32, 16, 1024), id, s > 0);
        mma_commit(mb_mma);
        pending |= 1u;
    };

    if (tid == 0 && c_begin < c_end) {
        issue_v(c_begin, 0);
        issue_qku(c_begin);
    }
    // this thread's two conv channels (re-read from L1 by every prep: no registers held across the loop)
    const __nv_bfloat162 *cw2 = reinterpret_cast<const __nv_bfloat162 *>(p.conv_w) + (size_t)h * 4 * (D / 2) + (tid & 31);

    // gates of one chunk: lane l of warp 1 holds beta/alpha of tokens 2l, 2l+1; thread
    // 256 + s (s < 192) holds gamma/eta slot s.  Warp 0 (thread 0 issues the MMAs) is left out,
    // so the next chunk's scalars are not held up behind an MMA issue sequence.
    constexpr int SCAN_WARP = 1, GATE_T0 = 256;
    static_assert(GATE_T0 + 64 * RMAX <= NT, "gate threads");
    const int gt = tid - GATE_T0;
    float pf_b0 = 0.f, pf_b1 = 0.f, pf_a0 = 1.f, pf_a1 = 1.f, pf_gam = 0.f, pf_eta = 0.f;
    auto load_gates = [&](int c) {
        const int n = min(C, p.T - c * C);
        const size_t tok0 = (size_t)bh * p.T + (size_t)c * C;
        if (warp == SCAN_WARP) {
            const int i0 = 2 * lane, i1 = 2 * lane + 1;
            pf_b0 = i0 < n ? p.beta[tok0 + i0] : 0.f;
            pf_b1 = i1 < n ? p.beta[tok0 + i1] : 0.f;
            pf_a0 = i0 < n ? p.alpha[tok0 + i0] : 1.f;
            pf_a1 = i1 < n ? p.alpha[tok0 + i1] : 1.f;
        }
        if (gt >= 0 && gt < 64 * RMAX) {
            const int i = gt / RMAX, l = gt % RMAX;
            const bool valid = (i < n) && (l < R);
            pf_gam = valid ? p.gamma[(tok0 + i) * R + l] : 0.f;
            pf_eta = (valid && p.eta) ? p.eta[(tok0 + i) * R + l] : 0.f;
        }
    };
    if (c_begin < c_end) load_gates(c_begin);
    // gates in registers -> one set of per-token scalars (no barrier inside)
    auto fill_scalars = [&](float *set) {
        if (warp == SCAN_WARP) {  // inclusive scan of the 64 log-decays, two per lane, in registers
            const float la0 = logf(pf_a0), la1 = logf(pf_a1);
            float s = la0 + la1;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const float y = __shfl_up_sync(0xffffffffu, s, off);
                if (lane >= off) s += y;
            }
            const float l1 = s, l0 = s - la1;
            const float lcw = __shfl_sync(0xffffffffu, s, 31);
            const int i0 = 2 * lane, i1 = i0 + 1;
            set[i0] = pf_b0;
            set[i1] = pf_b1;
            set[64 + i0] = l0;
            set[64 + i1] = l1;
            set[128 + i0] = __expf(l0 - lcw);
            set[128 + i1] = __expf(l1 - lcw);
            set[192 + i0] = __expf(lcw - l0);
            set[192 + i1] = __expf(lcw - l1);
            set[256 + i0] = __expf(l0);
            set[256 + i1] = __expf(l1);
            set[320 + i0] = pf_b0 * __expf(l0);
            set[320 + i1] = pf_b1 * __expf(l1);
        }
        if (gt >= 0 && gt < 64 * RMAX) {
            set[384 + gt] = pf_gam;
            set[384 + 64 * RMAX + gt] = pf_eta;
        }
    };

    // prep of chunk cc (P1): anchor, gain and residual chain -> X tiles, two channels x 4 tokens
    // per thread, from the V stage stg and the chunk's per-token scalars.  It runs in the
    // previous chunk's tail, while that chunk's last MMAs are in flight.
    auto prep = [&](int cc, int stg) {
        const uint32_t *pg = p.p_gain ? reinterpret_cast<const uint32_t *>(p.p_gain) +
                                            ((size_t)bh * p.T + (size_t)cc * C) * R * (D / 2)
                                      : nullptr;
        if (pg)
            prep_chunk<true>(sm, sc + (cc & 1) * SC_SET, cw2, stg, R, pg, min(C, p.T - cc * C));
        else
            prep_chunk<false>(sm, sc + (cc & 1) * SC_SET, cw2, stg, R, nullptr, 0);
    };

#ifdef PRISM_PHASE_TIMERS
    // per-phase totals in shared memory (registers would crowd the kernel's own)
    __shared__ unsigned long long ph_acc_s[kPhaseSlots];
    if (tid == 0)
        for (int k = 0; k < kPhaseSlots; ++k) ph_acc_s[k] = 0;
    long long ph_last = clock64();
#endif
    bool alive = true;
    for (int c = c_begin; c < c_end && alive; ++c) {
        const int stage = (c - c_begin) & 1;
        const int t0 = c * C;
        const int n = min(C, p.T - t0);
        const size_t tok0 = (size_t)bh * p.T + t0;

        float *const set = sc + (c & 1) * SC_SET;
        float *const s_beta = set, *const s_lam = set + 64, *const s_rowf = set + 128, *const s_colf = set + 192;
        float *const s_gam = set + 256, *const s_bg = set + 320;  // (gamma, eta at 384.. are the prep's)
        if (c == c_begin) {  // the first chunk's scalars and prep; later ones run in the previous chunk
            fill_scalars(set);
            if (c + 1 < c_end) load_gates(c + 1);
            if (!wait_one(mb_v[stage], ph_v[stage], 4u << stage)) break;
            if (seg == 0 && p.v_hist != nullptr) {  // the convolution's left context replaces the zero halo
                if (tid < 24) {  // 3 rows (tokens -3..-1) x 8 groups of 16 bytes
                    const uint4 hv = reinterpret_cast<const uint4 *>(p.v_hist + (size_t)bh * 3 * D)[tid];
                    *reinterpret_cast<uint4 *>(sm + (stage ? OFF_V1 : OFF_V0) + (5 + (tid >> 3)) * 128 + (tid & 7) * 16) = hv;
                    fence_async_smem();  // the stage is refilled by TMA later
                }
                __syncthreads();
            }
            prep(c, stage);
            fence_async_smem();
        }
        const float lc = s_lam[63];

        PHASE_MARK(0);
        // ---- P2: Gram tiles  D1 = [K; U_0] [Q; K]^T,  D1' = [U_1; U_2] [Q; K]^T ------------------
        // (rows are key/direction tokens j, columns query/key tokens i: the score tiles come out
        // transposed, [j][i], which is the operand form the later products read)
        // The first chunk of the segment waits for its tiles and issues its Gram here; every later
        // chunk's Gram was issued at the end of the chunk before it, under that chunk's output
        // stores, so only its completion is waited for.
        if (c == c_begin && !wait_one(mb_qku, ph_qku, 2u)) break;
        if (tid == 0 && c + 1 < c_end) issue_v(c + 1, stage ^ 1);
        if (tid == 0) {
            if (c == c_begin) {
                fence_after_sync();
                issue_gram();
            }
            if (mbar_wait(mb_mma, ph_mma, p.wait_ns)) {
                pending &= ~1u;
            } else {
                abort_s = 1;
                set_status(p.status, kDevTimeout);
            }
        }

        PHASE_MARK(1);
        {  // diag(beta Gamma) K, one 16-byte group of 8 per thread (K still bf16)
            const int j = tid >> 3, m0 = (tid & 7) * 8;
            uint4 w = *reinterpret_cast<const uint4 *>(sm + OFF_K + sw128(j, m0));
            uint32_t *pw = &w.x;
            const float sbg = s_bg[j];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&pw[q]));
                pw[q] = pack2(sbg * f.x, sbg * f.y);
            }
            *reinterpret_cast<uint4 *>(sm + OFF_BGK + sw128(j, m0)) = w;
        }
        fence_async_smem();
        __syncthreads();
        if (abort_s) break;
        ph_mma ^= 1u;  // every thread's copy of the MMA barrier phase (thread 0 waited for it)
        fence_after_sync();

        PHASE_MARK(2);
        // ---- E1: masks and decays -> A (fp32), PK_l^T, PQ_l^T, G^T (fp16 tiles) --------------------
        // TMEM lanes 0..63 hold key rows k_j, 64..127 direction rows u_{j,0} (D1) and u_{j,1},
        // u_{j,2} (D1'); column block 0/2 holds the query side q_i, 1/3 the key side k_i.  Each
        // kept element takes its pair decay D_ij = e^{lambda_i - lambda_j} in fp32: the product
        // rowf_i colf_j while the chunk's total decay keeps both factors in fp32 range (the usual
        // case), else one exponential per element.
        {
            const int r = row & 63;
            const bool upper = row >= 64;
            const int nblk = R >= 2 ? 4 : 2;
            const bool skip = upper && R == 0;  // u_0 rows do not exist
            const float lr = s_lam[r];
            const float rf_r = s_rowf[r], cf_r = s_colf[r];
            const float br = s_beta[r];
            const int j0 = sub * CW;
            // one copy of the epilogue per decay form (a uniform branch: no per-element select)
            auto e1 = [&](auto form) {
                constexpr bool kFactored = decltype(form)::value;
                // decay of row token r (a key / direction token j) to column token i = j0 + q, i >= r
                float dq[CW];
                if constexpr (kFactored) {
#pragma unroll
                    for (int g = 0; g < CW / 4; ++g) {
                        const float4 f = reinterpret_cast<const float4 *>(s_rowf + j0)[g];
                        dq[4 * g + 0] = f.x * cf_r;
                        dq[4 * g + 1] = f.y * cf_r;
                        dq[4 * g + 2] = f.z * cf_r;
                        dq[4 * g + 3] = f.w * cf_r;
                    }
                } else {
#pragma unroll
                    for (int q = 0; q < CW; ++q) dq[q] = __expf(fminf(s_lam[j0 + q] - lr, 0.f));
                }
#pragma unroll
                for (int b2 = 0; b2 < 4; b2 += 2) {  // two 64-column blocks per TMEM wait
                    if (b2 >= nblk || skip) break;
                    if (b2 == 2 && upper && R < 3) break;  // u_2 rows do not exist
                    uint32_t rr[2][CW];
#pragma unroll
                    for (int u = 0; u < 2; ++u)
                        tmem_ld_nowait(tmem + TM_D1 + ((uint32_t)(quad * 32) << 16) + (uint32_t)((b2 + u) * 64 + j0),
                                       rr[u]);
                    tmem_wait_ld();
                    const int l = b2 ? (upper ? 2 : 1) : 0;  // direction level of an upper / D1' row
                    const bool keyrow = b2 == 0 && !upper;
#pragma unroll
                    for (int u = 0; u < 2; ++u) {
                        float v[CW];
                        u2f(rr[u], v);
                        if (u == 0) {  // query side: G^T (key rows) or PQ_l^T, kept where i >= j
#pragma unroll
                            for (int q = 0; q < CW; ++q) v[q] = (j0 + q >= r) ? v[q] * dq[q] : 0.f;
                            st_row(sm + (keyrow ? OFF_G : OFF_E + (2 * l + 1) * TILE), r, j0, v);
                        } else if (keyrow) {  // A_ij = beta_i D_ij k_i.k_j (j < i), row i = r, from k_j.k_i
                            float4 *A4 = reinterpret_cast<float4 *>(sm + OFF_AKK + (r * LDA + j0) * 4);
#pragma unroll
                            for (int g = 0; g < CW / 4; ++g) {
                                float d[4];
                                if constexpr (kFactored) {
                                    const float4 cf = reinterpret_cast<const float4 *>(s_colf + j0)[g];
                                    const float b = br * rf_r;
                                    d[0] = b * cf.x;
                                    d[1] = b * cf.y;
                                    d[2] = b * cf.z;
                                    d[3] = b * cf.w;
                                } else {
#pragma unroll
                                    for (int e = 0; e < 4; ++e) d[e] = br * __expf(fminf(lr - s_lam[j0 + 4 * g + e], 0.f));
                                }
                                const int j = j0 + 4 * g;
                                A4[g] = make_float4(j + 0 < r ? v[4 * g + 0] * d[0] : 0.f, j + 1 < r ? v[4 * g + 1] * d[1] : 0.f,
                                                    j + 2 < r ? v[4 * g + 2] * d[2] : 0.f, j + 3 < r ? v[4 * g + 3] * d[3] : 0.f);
                            }
                        } else {  // PK_l^T, kept where i > j
#pragma unroll
                            for (int q = 0; q < CW; ++q) v[q] = (j0 + q > r) ? v[q] * dq[q] : 0.f;
                            st_row(sm + OFF_E + 2 * l * TILE, r, j0, v);
                        }
                    }
                }
            };
            if (-lc <= 80.f)
                e1(BoolTag<true>{});
            else
                e1(BoolTag<false>{});
        }
        fence_async_smem();
        fence_before_sync();
        __syncthreads();

        PHASE_MARK(3);
        // ---- P3: MX = sum_l PK_l X_l on the tensor core.  Meanwhile the warps of TMEM lane
        // quarters 2-3 solve T = (I + A)^{-1}, and those of quarters 0-1 (thread 0 among them)
        // wait for MX, form the RHS (E2) and convert K and U to fp16.  The two groups of 256
        // threads sync on named barriers 1 and 2 and meet again at the CTA barrier before P4.
        if (tid == 0) {
            fence_after_sync();
            // A = PK_l^T in MN-major form; its second 64-row atom (lanes 64..127, never read)
            // points at the next tile
            const uint32_t id = idesc_f16(128, 64, 1, 1);
            for (int l = 0; l < R; ++l)
#pragma unroll
                for (int s = 0; s < 4; ++s)
                    mma_f16(tmem + TM_D2, dsc(dbase, OFF_E + l * 2 * TILE + s * 2048, TILE, 1024),
                             dsc(dbase, OFF_XS + l * TILE + s * 2048, TILE, 1024), id, (l | s) != 0);
            mma_commit(mb_mma);
            pending |= 1u;
        }
        PHASE_MARK(11);
        if (quad >= 2) {
            {
                // T = (I + A)^{-1} by 16x16 blocks: diagonal blocks by forward substitution, then the
                // block diagonals below them, T[bi][bj] = -T[bi][bi] sum_{k=bj..bi-1} A[bi][k] T[k][bj]
                const int sw = ((warp >> 2) << 1) | (warp & 1);  // solver warp 0..7: warps 2,3,6,7,10,11,14,15
                const int stid = sw * 32 + lane;
                const float *A = reinterpret_cast<const float *>(sm + OFF_AKK);
                float *T32 = reinterpret_cast<float *>(sm + OFF_T32);
                const Frag fr{lane >> 2, lane & 3};
                if (tid >= 64 && tid < 128) {  // diagonal 16x16 blocks by forward substitution, one
                    // column per thread (warps 2-3)
                    const int o = 16 * ((tid - 64) >> 4), cc = tid & 15;
                    float t[16];
                    // the block's row r of A as four 16-byte loads, the next row's in flight while a
                    // row is summed; T's column is stored after the whole column (a store between
                    // the rows would keep every later row's loads of A, which it may alias, behind it)
                    auto arow = [&](int r, float (&a)[16]) {
                        const float4 *src = reinterpret_cast<const float4 *>(A + (o + r) * LDA + o);
#pragma unroll
                        for (int g = 0; g < 4; ++g) {
                            const float4 f = src[g];
                            a[4 * g] = f.x;
                            a[4 * g + 1] = f.y;
                            a[4 * g + 2] = f.z;
                            a[4 * g + 3] = f.w;
                        }
                    };
                    float ar[2][16];  // row 0 reads none of A
#pragma unroll
                    for (int r = 0; r < 16; ++r) {
                        if (r + 1 < 16) arow(r + 1, ar[(r + 1) & 1]);
                        const float *a = ar[r & 1];
                        // t[j] = 0 for j < cc, so the sum may run over all j < r
                        float s0 = 0.f, s1 = 0.f;
#pragma unroll
                        for (int j = 0; j + 1 < r; j += 2) {
                            s0 = fmaf(a[j], t[j], s0);
                            s1 = fmaf(a[j + 1], t[j + 1], s1);
                        }
                        if (r & 1) s0 = fmaf(a[r - 1], t[r - 1], s0);
                        t[r] = (r == cc) ? 1.f : (r < cc ? 0.f : -(s0 + s1));
                    }
#pragma unroll
                    for (int r = 0; r < 16; ++r) T32[(o + r) * LDA + o + cc] = t[r];
                }
                named_bar(1, NT / 2);
                if (sw < 4) {
                    // 16 -> 32: T[1][0] = -T[1][1] A[1][0] T[0][0], T[3][2] likewise; solver warp sw
                    // owns one 8-column tile of one block
                    const int pb = sw >> 1, nt = sw & 1;         // block pair (0: rows 16.., 1: rows 48..)
                    const int ri = 16 + 32 * pb, cj = 32 * pb;        // block (ri, cj) below the diagonal
                    float x[4] = {0.f, 0.f, 0.f, 0.f};
                    {                                                 // X = A[ri][cj] T[cj][cj] (cols 8 nt..)
                        uint32_t a[4], b0, b1;
                        frag_a16(fr, A, LDA, ri, cj, a);
                        frag_b16(fr, T32, LDA, cj, cj + 8 * nt, b0, b1);
                        mma_h16(x, a, b0, b1);
                    }
                    float *X = s_xtmp + sw * 128;                     // 16 x 8
                    X[fr.gq * 8 + 2 * fr.tq] = x[0];
                    X[fr.gq * 8 + 2 * fr.tq + 1] = x[1];
                    X[(fr.gq + 8) * 8 + 2 * fr.tq] = x[2];
                    X[(fr.gq + 8) * 8 + 2 * fr.tq + 1] = x[3];
                    __syncwarp();
                    float y[4] = {0.f, 0.f, 0.f, 0.f};
                    {                                                 // T[ri][cj] = -T[ri][ri] X
                        uint32_t a[4], b0, b1;
                        frag_a16(fr, T32, LDA, ri, ri, a);
                        frag_b16(fr, X, 8, 0, 0, b0, b1);
                        mma_h16(y, a, b0, b1);
                    }
                    frag_c_store(fr, T32, LDA, ri, cj + 8 * nt, y, -1.f);
                }
                named_bar(1, NT / 2);
                {
                    // 32 -> 64: T[32:64][0:32] = -T[32:64][32:64] A[32:64][0:32] T[0:32][0:32]; solver
                    // warp sw owns the 16-row half mt = sw / 4 of the 8-column tile nt = sw % 4 (n0 = 8 nt):
                    // its rows of X = A_lo T_lo, then (once all of X is in) its rows of -T_hi X
                    const int nt = sw & 3, mt = sw >> 2, n0 = 8 * nt;
                    float x[4] = {0.f, 0.f, 0.f, 0.f};
                    // T_lo[k][n] = 0 for k < 16 <= n: block (0,1) of T32 is never written, so skip it
#pragma unroll
                    for (int ks = 0; ks < 2; ++ks) {                 // X = A_lo T_lo, 16 of k a step
                        if (n0 >= 16 && ks == 0) continue;
                        uint32_t a[4], b0, b1;
                        frag_b16(fr, T32, LDA, 16 * ks, n0, b0, b1);
                        frag_a16(fr, A, LDA, 32 + 16 * mt, 16 * ks, a);
                        mma_h16(x, a, b0, b1);
                    }
                    float *X = s_xtmp + nt * 256;                     // 32 x 8
                    X[(16 * mt + fr.gq) * 8 + 2 * fr.tq] = x[0];
                    X[(16 * mt + fr.gq) * 8 + 2 * fr.tq + 1] = x[1];
                    X[(16 * mt + fr.gq + 8) * 8 + 2 * fr.tq] = x[2];
                    X[(16 * mt + fr.gq + 8) * 8 + 2 * fr.tq + 1] = x[3];
                    named_bar(1, NT / 2);  // both halves of every X tile are in
                    float y[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                    for (int ks = 0; ks < 2; ++ks) {                 // T_lower = -T_hi X, 16 of k a step
                        if (mt == 0 && ks == 1) continue;  // T_hi[0:16][16:32] = 0 (block (2,3) is never written)
                        uint32_t a[4], b0, b1;
                        frag_b16(fr, X, 8, 16 * ks, 0, b0, b1);
                        frag_a16(fr, T32, LDA, 32 + 16 * mt, 32 + 16 * ks, a);
                        mma_h16(y, a, b0, b1);
                    }
                    frag_c_store(fr, T32, LDA, 32 + 16 * mt, n0, y, -1.f);
                }
                if (tid == 64 && !mbar_wait(mb_mma, ph_mma, p.wait_ns)) {  // MX has read PK_1^T (T's slot)
                    abort_s = 1;
                    set_status(p.status, kDevTimeout);
                }
                named_bar(1, NT / 2);
                // T as an fp16 operand ([i][j], zero above the diagonal)
                for (int e = stid; e < 64 * 8; e += NT / 2) {
                    const int i = e >> 3, g = e & 7;
                    const float4 lo = *reinterpret_cast<const float4 *>(T32 + i * LDA + 8 * g);
                    const float4 hi = *reinterpret_cast<const float4 *>(T32 + i * LDA + 8 * g + 4);
                    const float v[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
                    float m[8];
#pragma unroll
                    for (int q = 0; q < 8; ++q) m[q] = (8 * g + q <= i) ? v[q] : 0.f;
                    uint4 w;
                    w.x = pack2(m[0], m[1]);
                    w.y = pack2(m[2], m[3]);
                    w.z = pack2(m[4], m[5]);
                    w.w = pack2(m[6], m[7]);
                    *reinterpret_cast<uint4 *>(sm + OFF_TF + sw128(i, 8 * g)) = w;
                }
            }
        } else {
            if (tid == 0) {
                if (mbar_wait(mb_mma, ph_mma, p.wait_ns)) {
                    pending &= ~1u;
                } else {
                    abort_s = 1;
                    set_status(p.status, kDevTimeout);
                }
            }
            named_bar(2, NT / 2);
            PHASE_MARK(4);
            if (abort_s == 0) {
                fence_after_sync();
                // ---- E2: RHS = diag(beta) (V - MX) (diag(beta Gamma) K was formed during the prep) ---
                // (lanes 0..63 hold the MX rows)
                const __nv_bfloat16 *vb = reinterpret_cast<const __nv_bfloat16 *>(sm + (stage ? OFF_V1 : OFF_V0));
                const int i = row, j0 = sub * CW;
                float v[CW];
                if (R > 0) {
                    tmem_ld(tmem + TM_D2 + ((uint32_t)(quad * 32) << 16) + (uint32_t)j0, v);
                } else {
#pragma unroll
                    for (int q = 0; q < CW; ++q) v[q] = 0.f;  // no levels: M X = 0 (D2 is never written)
                }
                const float bi = s_beta[i];
#pragma unroll
                for (int q = 0; q < CW; ++q) v[q] = bi * (__bfloat162float(vb[(i + 8) * 64 + j0 + q]) - v[q]);
                st_row(sm + OFF_E, i, j0, v);  // RHS tile, over PK_0^T (MX, its reader, is complete)
                PHASE_MARK(12);
                // K' = diag(colf) K and U'_l = diag(colf) U_l in fp16, in place, for the state-side
                // products (the Gram has read K and U)
                tiles_bf16_to_f16(sm + OFF_K, (1 + R) * TILE, (warp >> 2) * 64 + (warp & 1) * 32 + lane, NT / 2, s_colf);
                PHASE_MARK(13);
            }
        }
        fence_async_smem();
        fence_before_sync();
        __syncthreads();
        if (abort_s) break;
        ph_mma ^= 1u;  // MX completed (thread 0 waited for it)

        PHASE_MARK(5);
        // ---- P4: [U'^T ; W^T] = [RHS | BGK]^T T^T -------------------------------------------------
        if (tid == 0) {
            fence_after_sync();
            const uint32_t id = idesc_f16(128, 64, 1, 0);
#pragma unroll
            for (int s = 0; s < 4; ++s)
                mma_f16(tmem + TM_D3, dsc(dbase, OFF_E + s * 2048, OFF_BGK - OFF_E, 1024),
                        dsc(dbase, OFF_TF + s * 32, 16, 1024),
                         id, s > 0);
            mma_commit(mb_mma);
            pending |= 1u;
            // [Y; Q^T] I -> Q^T in lanes 64..127 (exact: bf16 times one), so that E4 needs no Q tile
            // and Q's buffer can take the next chunk's tile after P5.  The first atom Y is the tile
            // below Q (V data); lanes 0..63 of these columns are never read.  Issued here, behind
            // P4 and outside P3 (where MX and the solve's warp MMAs share the tensor pipe); P5's
            // commit covers it.
            const uint32_t idq = idesc_bf16(128, 64, 1, 0);
#pragma unroll
            for (int s = 0; s < 4; ++s)
                mma_f16(tmem + TM_QT, dsc(dbase, OFF_Q - TILE + s * 2048, TILE, 1024),
                        dsc(dbase, OFF_TB + s * 32, 16, 1024), idq, s > 0);
        }
        wait_mma();
        fence_after_sync();

        PHASE_MARK(6);
        // ---- E3: UW = [U'^T; W^T] -> fp16 --------------------------------------------------------
        {
            const int j0 = sub * CW;
            float v[CW];
            tmem_ld(tmem + TM_D3 + ((uint32_t)(quad * 32) << 16) + (uint32_t)j0, v);
            st_row(sm + OFF_AKK, row, j0, v);  // over A (the solve is complete)
        }
        fence_async_smem();
        fence_before_sync();
        __syncthreads();
        if (abort_s) break;

        PHASE_MARK(7);
        // ---- P5: [D5 | D4] = UW [K' | G^T] + sum_l [X_l^T; 0] [U'_l | PQ_l^T]  (N = 128) ----------
        if (tid == 0) {
            fence_after_sync();
            const uint32_t idk = idesc_f16(128, 128, 0, 1), idx = idesc_f16(128, 128, 1, 1);
#pragma unroll
            for (int s = 0; s < 4; ++s)
                mma_f16(tmem + TM_D5, dsc(dbase, OFF_AKK + s * 32, 16, 1024),
                        dsc(dbase, OFF_K + s * 2048, OFF_G - OFF_K, 1024), idk, s > 0);
            for (int l = 0; l < R; ++l) {
                const uint32_t xs = OFF_XS + l * TILE, ub = OFF_U + l * TILE, pq = OFF_E + l * 2 * TILE + TILE;
#pragma unroll
                for (int s = 0; s < 4; ++s)
                    mma_f16(tmem + TM_D5, dsc(dbase, xs + s * 2048, OFF_ZERO - xs, 1024),
                            dsc(dbase, ub + s * 2048, pq - ub, 1024), idx, 1);
            }
            mma_commit(mb_mma);
            pending |= 1u;
        }
        if (c + 1 < c_end) {  // next chunk's per-token scalars while the MMAs run
            fill_scalars(sc + ((c + 1) & 1) * SC_SET);
            if (c + 2 < c_end) load_gates(c + 2);
        }
        wait_mma();
        fence_after_sync();

        // the next chunk's Q, K and U: this chunk's Q was last read by the Q^T copy (complete with P5),
        // K and U by P5
        if (tid == 0 && c + 1 < c_end && abort_s == 0) issue_qku(c + 1);
        PHASE_MARK(8);
        // ---- E4: Qt = diag(Gamma) Q^T - (G W)^T ;  Mc = Gamma_C I - W^T K' --------------------------
        if (quad >= 2) {
            const int m = row - 64, j0 = sub * CW;
            float v[CW], v5[CW];
            {
                uint32_t r4[CW], r5[CW], rq[CW];
                tmem_ld_nowait(tmem + TM_D4 + ((uint32_t)(quad * 32) << 16) + (uint32_t)j0, r4);
                tmem_ld_nowait(tmem + TM_D5 + ((uint32_t)(quad * 32) << 16) + (uint32_t)j0, r5);
                tmem_ld_nowait(tmem + TM_QT + ((uint32_t)(quad * 32) << 16) + (uint32_t)j0, rq);
                tmem_wait_ld();
                u2f(r4, v);
                u2f(r5, v5);
#pragma unroll
                for (int q = 0; q < CW; ++q) v[q] = s_gam[j0 + q] * __uint_as_float(rq[q]) - v[q];
            }
            st_row(sm + OFF_E, m, j0, v);  // Qt [m][i]
#pragma unroll
            for (int q = 0; q < CW; ++q) v[q] = v5[q];
            const float gC = __expf(lc);
#pragma unroll
            for (int q = 0; q < CW; ++q) v[q] = ((j0 + q) == m ? gC : 0.f) - v[q];
            st_row(sm + OFF_E + TILE, m, j0, v);  // Mc [m][m']
        }
        if (tid == 0 && c + 1 < c_end) {  // the next chunk's V (issued at this chunk's start) for its prep
            if (mbar_wait(mb_v[stage ^ 1], ph_v[stage ^ 1], p.wait_ns)) {
                ph_v[stage ^ 1] ^= 1u;
                pending &= ~(4u << (stage ^ 1));
            } else {
                abort_s = 1;
                set_status(p.status, kDevTimeout);
            }
        }
        fence_async_smem();
        fence_before_sync();
        __syncthreads();
        if (abort_s) break;
        if (tid == 0) {
            fence_after_sync();
            // ---- P6: [D7 | D6] = Z [Qt | Mc]  (N = 128) ------------------------------------------
            const uint32_t id = idesc_f16(128, 128, 0, 1);
#pragma unroll
            for (int s = 0; s < 4; ++s)
                mma_f16(tmem + TM_D7, dsc(dbase, OFF_ZA + s * 32, 16, 1024), dsc(dbase, OFF_E + s * 2048, TILE, 1024),
                        id, s > 0);
            mma_commit(mb_mma);
            pending |= 1u;
        }
        if (c + 1 < c_end) {  // the next chunk's prep while MMA6 runs (X of this chunk is dead)
            prep(c + 1, stage ^ 1);
            fence_async_smem();
        }
        PHASE_MARK(14);
        wait_mma();
        fence_after_sync();

        PHASE_MARK(9);
        // ---- E5: Z <- Z Mc + [N_c; 0];  o0 / Qhat ------------------------------------------------
        {
            const int j0 = sub * CW;
            const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
            float z[CW], nc[CW], o[CW], ol[CW];
            {
                uint32_t r0[CW], r1[CW], r2[CW], r3[CW];
                tmem_ld_nowait(tmem + TM_D6 + lane_off + (uint32_t)j0, r0);
                tmem_ld_nowait(tmem + TM_D5 + lane_off + (uint32_t)j0, r1);
                tmem_ld_nowait(tmem + TM_D7 + lane_off + (uint32_t)j0, r2);
                tmem_ld_nowait(tmem + TM_D4 + lane_off + (uint32_t)j0, r3);
                tmem_wait_ld();
                u2f(r0, z);
                u2f(r1, nc);
                u2f(r2, o);
                u2f(r3, ol);
            }
            if (row < 64) {
#pragma unroll
                for (int q = 0; q < CW; ++q) z[q] += nc[q];
            }
            // ZA and the region holding Qt/Mc are rewritten below: MMA6/7, their readers, are complete
            PHASE_MARK(15);
            st_row(sm + OFF_ZA, row, j0, z);
            fence_async_smem();  // ZA is the next chunk's MMA operand; nothing after this needs the fence
            if (c + 1 == c_end) {
                float *zs = p.zsum + (((size_t)bh * p.P + seg) * 128 + row) * 64 + j0;
#pragma unroll
                for (int q = 0; q < CW; ++q) zs[q] = z[q];
            }
            // outputs: row < 64 -> o0^T[c][i] = D7 + O_loc^T ; row >= 64 -> Qhat^T[m][i].  They are
            // transposed through shared memory (region E: Qt and Mc are no longer read) and
            // written with 16-byte stores: o0 as [i][c] fp32, Qhat as [i][m] fp16.
            float *so = reinterpret_cast<float *>(sm + OFF_E);                // [64][64] fp32
            __half *sq = reinterpret_cast<__half *>(sm + OFF_E + 2 * TILE);   // [64][64] fp16
            if (row < 64) {
#pragma unroll
                for (int q = 0; q < CW; ++q) so[(j0 + q) * 64 + row] = o[q] + ol[q];
            } else if (tracked) {
#pragma unroll
                for (int q = 0; q < CW; ++q) sq[(j0 + q) * 64 + row - 64] = __float2half_rn(o[q]);
            }
        }
        PHASE_MARK(16);
        fence_before_sync();  // the tensor-memory reads of this chunk precede the next chunk's Gram
        __syncthreads();
        PHASE_MARK(17);
        // the next chunk's Gram, under this chunk's output stores: its tiles were requested during
        // this chunk (Q after the Q^T copy, K and U after the state-side products), and tensor
        // memory columns 0..255 are free (D7 and D6 were read above)
        if (tid == 0 && c + 1 < c_end && abort_s == 0) {
            if (mbar_wait(mb_qku, ph_qku, p.wait_ns)) {
                ph_qku ^= 1u;
                pending &= ~2u;
                fence_after_sync();
                issue_gram();
            } else {
                abort_s = 1;
                set_status(p.status, kDevTimeout);
            }
        }
        {
            const float *so = reinterpret_cast<const float *>(sm + OFF_E);
            bool finite = true;
            for (int e = tid; e < 64 * 16; e += NT) {  // 16-byte groups of 4 outputs
                const int i = e >> 4, c4 = (e & 15) * 4;
                if (i >= n) continue;
                const float4 v = *reinterpret_cast<const float4 *>(so + i * 64 + c4);
                finite = finite && isfinite(v.x) && isfinite(v.y) && isfinite(v.z) && isfinite(v.w);
                const size_t o = (tok0 + i) * D + c4;
                if (!tracked) {
                    if (p.out_f32) {
                        *reinterpret_cast<float4 *>(reinterpret_cast<float *>(p.out) + o) = v;
                    } else {
                        __nv_bfloat162 lo = __floats2bfloat162_rn(v.x, v.y), hi = __floats2bfloat162_rn(v.z, v.w);
                        uint2 w;
                        w.x = *reinterpret_cast<uint32_t *>(&lo);
                        w.y = *reinterpret_cast<uint32_t *>(&hi);
                        *reinterpret_cast<uint2 *>(reinterpret_cast<__nv_bfloat16 *>(p.out) + o) = w;
                    }
                } else if (p.out_f32) {
                    *reinterpret_cast<float4 *>(reinterpret_cast<float *>(p.stash_o) +
                                                (((size_t)bh * p.NC + c) * 64 + i) * 64 + c4) = v;
                } else {
                    __half2 lo = __floats2half2_rn(v.x, v.y), hi = __floats2half2_rn(v.z, v.w);
                    uint2 w;
                    w.x = *reinterpret_cast<uint32_t *>(&lo);
                    w.y = *reinterpret_cast<uint32_t *>(&hi);
                    *reinterpret_cast<uint2 *>(reinterpret_cast<__half *>(p.stash_o) +
                                               (((size_t)bh * p.NC + c) * 64 + i) * 64 + c4) = w;
                }
            }
            PHASE_MARK(18);
            if (tracked) {
                const uint4 *sq = reinterpret_cast<const uint4 *>(sm + OFF_E + 2 * TILE);
                uint4 *dq = reinterpret_cast<uint4 *>(p.stash_q + ((size_t)bh * p.NC + c) * 4096);
                for (int e = tid; e < 512; e += NT) dq[e] = sq[e];
            }
            if (!finite) set_status(p.status, kDevBounds);  // outside the fp16 operand range
            PHASE_MARK(19);
        }
        fence_before_sync();
        __syncthreads();
        alive = abort_s == 0;
        PHASE_MARK(10);
    }
#ifdef PRISM_PHASE_TIMERS
    if (tid == 0)
        for (int k = 0; k < kPhaseSlots; ++k) atomicAdd(&prism_tc_phase_cycles[k], ph_acc_s[k]);
#endif

    // drain: after an expired wait, let every copy and MMA still in flight land (bounded by
    // one second each) before the CTA releases its shared and tensor memory
    if (tid == 0 && pending) {
        const uint64_t drain_ns = 1000000000ull;
        if (pending & 1u) (void)mbar_wait(mb_mma, ph_mma, drain_ns);
        if (pending & 2u) (void)mbar_wait(mb_qku, ph_qku, drain_ns);
        if (pending & 4u) (void)mbar_wait(mb_v[0], ph_v[0], drain_ns);
        if (pending & 8u) (void)mbar_wait(mb_v[1], ph_v[1], drain_ns);
    }
    fence_before_sync();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, 512);
}

// ---------------------------------------------------------------------------------------------
// combine: S_start[p] = S_start[p-1] M_{p-1} + N_{p-1} in fp32 from S_start[0] = S_init (or 0),
// 4 value rows per block (16 blocks a sequence: a short product per step, one block per SM), written
// out as fp16 (the fix-up's MMA operand); with S_final the map of the last segment is applied too
// and the result written out in fp32.  The maps stream through a ring of CB_STAGES shared-memory
// stages filled by bulk copies (16 KB of M and this block's 1 KB of N per segment), so the serial
// chain never waits on global memory latency.  Each step's 4x64x64 product is split over the sum
// index: thread (kq, rg, lane) accumulates rows 2 rg, 2 rg + 1, columns 2 lane, 2 lane + 1 over m
// in [16 kq, 16 kq + 16); the four partial sums meet in shared memory, thread (row, column) adding
// them.  The running rows are double-buffered, so two barriers per segment order the row exchange,
// the partial sums and the reuse of a ring stage.
constexpr int CB_ROWS = 4;
constexpr int CB_STAGES = 4;
constexpr int CB_KQ = 4;                       // parts of the sum index
constexpr int CB_THREADS = CB_KQ * 2 * 32;     // x 2 row groups (2 rows each) x 32 column pairs
static_assert(CB_THREADS == CB_ROWS * 64, "one output of the step per thread in the reduction");
constexpr int CB_STAGE_FLOATS = 64 * 64 + CB_ROWS * 64;
constexpr size_t CB_SMEM = (size_t)CB_STAGES * CB_STAGE_FLOATS * 4 + 128;
// The launch requests more shared memory than the combine uses, so that one of its blocks fits an
// SM: launched while the segment kernel drains, its blocks are placed on SMs as they free up, and
// packed three to an SM their chains ran slower (0.165 against 0.160 ms per forward at 16K tokens).
constexpr size_t CB_SMEM_LAUNCH = 120 * 1024;
static_assert(CB_SMEM <= CB_SMEM_LAUNCH && 2 * (CB_SMEM_LAUNCH + 1024) > 228 * 1024, "one combine block per SM");

__global__ void __launch_bounds__(CB_THREADS) combine_kernel(const float *__restrict__ zsum, __half *__restrict__ sstart,
                                                             int P, const float *S_init, float *S_final, int *status,
                                                             unsigned long long wait_ns)
{
    extern __shared__ __align__(128) float ring[];  // [CB_STAGES][M 64x64 | N 8x64]
    __shared__ __align__(8) uint64_t mb[CB_STAGES];
    __shared__ __align__(16) float S[2][CB_ROWS][64];
    __shared__ __align__(16) float part[CB_KQ][CB_ROWS][64];
    __shared__ int abort_s;
    const int bh = blockIdx.x, r0 = blockIdx.y * CB_ROWS, tid = threadIdx.x;
    const int kq = tid >> 6, rg = (tid >> 5) & 1, l = tid & 31, c2 = 2 * l;
    const int rr = tid >> 6, cc = tid & 63;  // the entry this thread reduces
    prism::tc::grid_dependency_wait();  // the segment maps of the segment kernel
    prism::tc::allow_dependent_launch();
    // S_init and S_final may be one buffer: each thread reads its entry here and writes the same
    // one at the end
    const float s0 = S_init ? S_init[((size_t)bh * 64 + r0 + rr) * 64 + cc] : 0.f;
    sstart[((size_t)bh * P * 64 + r0 + rr) * 64 + cc] = __float2half_rn(s0);
    S[0][rr][cc] = s0;
    const int nmaps = S_final ? P : P - 1;  // maps of segments 0..P-2 (and P-1 for S_final)
    if (nmaps == 0) return;
    auto issue = [&](int sp) {
        const int st = sp % CB_STAGES;
        const uint32_t m = prism::tc::smem_u32(&mb[st]);
        const float *z = zsum + ((size_t)bh * P + sp) * 128 * 64;
        float *dst = ring + (size_t)st * CB_STAGE_FLOATS;
        prism::tc::mbar_expect_tx(m, (64 * 64 + CB_ROWS * 64) * 4);
        prism::tc::bulk_load(prism::tc::smem_u32(dst), z + 64 * 64, 64 * 64 * 4, m);
        prism::tc::bulk_load(prism::tc::smem_u32(dst + 64 * 64), z + r0 * 64, CB_ROWS * 64 * 4, m);
    };
    if (tid == 0) {
        abort_s = 0;
        for (int st = 0; st < CB_STAGES; ++st) prism::tc::mbar_init(prism::tc::smem_u32(&mb[st]), 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        for (int sp = 0; sp < nmaps && sp < CB_STAGES; ++sp) issue(sp);
    }
    int issued = min(nmaps, CB_STAGES);
#ifdef PRISM_PHASE_TIMERS
    const bool trace = tid == 0 && blockIdx.x == 0 && blockIdx.y == 0;
    unsigned long long t_wait = 0, t_comp = 0, t_barb = 0;
    const long long t_begin = clock64();
#endif
    int k = 0;
    for (; k < nmaps; ++k) {
        const int st = k % CB_STAGES, buf = k & 1;
#ifdef PRISM_PHASE_TIMERS
        const long long tw0 = clock64();
#endif
        if (tid == 0 && !prism::tc::mbar_wait(prism::tc::smem_u32(&mb[st]), (uint32_t)((k / CB_STAGES) & 1), wait_ns)) {
            abort_s = 1;
            atomicCAS(status, 0, kDevTimeout);
        }
#ifdef PRISM_PHASE_TIMERS
        if (trace) t_wait += clock64() - tw0;
#endif
        __syncthreads();  // stage k landed; rows of step k - 1 written; stage of step k - 1 free
        if (abort_s) break;
        if (tid == 0 && k > 0 && issued < nmaps) {  // refill the stage step k - 1 read
            prism::tc::fence_async_smem();
            issue(issued++);
        }
        const float *M = ring + (size_t)st * CB_STAGE_FLOATS;
#ifdef PRISM_PHASE_TIMERS
        const long long tc0 = clock64();
#endif
        constexpr int RPT = CB_ROWS / 2;  // rows of a thread's partial sums
        float acc[RPT][2];
#pragma unroll
        for (int r = 0; r < RPT; ++r) acc[r][0] = acc[r][1] = 0.f;
#pragma unroll
        for (int m = 16 * kq; m < 16 * kq + 16; m += 4) {
            float4 sv[RPT];
#pragma unroll
            for (int r = 0; r < RPT; ++r) sv[r] = *reinterpret_cast<const float4 *>(&S[buf][RPT * rg + r][m]);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const float2 mv = *reinterpret_cast<const float2 *>(M + (m + q) * 64 + c2);
#pragma unroll
                for (int r = 0; r < RPT; ++r) {
                    const float sq = q == 0 ? sv[r].x : q == 1 ? sv[r].y : q == 2 ? sv[r].z : sv[r].w;
                    acc[r][0] = fmaf(sq, mv.x, acc[r][0]);
                    acc[r][1] = fmaf(sq, mv.y, acc[r][1]);
                }
            }
        }
#pragma unroll
        for (int r = 0; r < RPT; ++r)
            *reinterpret_cast<float2 *>(&part[kq][RPT * rg + r][c2]) = make_float2(acc[r][0], acc[r][1]);
#ifdef PRISM_PHASE_TIMERS
        const long long tc1 = clock64();
#endif
        __syncthreads();
#ifdef PRISM_PHASE_TIMERS
        if (trace) {
            t_comp += tc1 - tc0;
            t_barb += clock64() - tc1;
        }
#endif
        float o = M[64 * 64 + rr * 64 + cc];  // N_p
#pragma unroll
        for (int q = 0; q < CB_KQ; ++q) o += part[q][rr][cc];
        S[buf ^ 1][rr][cc] = o;
        if (k + 1 < P)
            sstart[(((size_t)bh * P + k + 1) * 64 + r0 + rr) * 64 + cc] = __float2half_rn(o);
        else  // k + 1 == P: the state after the last token (S_final was asked for)
            S_final[((size_t)bh * 64 + r0 + rr) * 64 + cc] = o;
    }
#ifdef PRISM_PHASE_TIMERS
    if (trace) {  // combine tracing: block (0, 0), thread 0: map waits and the whole chain
        atomicAdd(&prism_tc_phase_cycles[20], t_wait);
        atomicAdd(&prism_tc_phase_cycles[21], (unsigned long long)(clock64() - t_begin));
        atomicAdd(&prism_tc_phase_cycles[22], t_comp);
        atomicAdd(&prism_tc_phase_cycles[23], t_barb);
    }
#endif
    // after an expired wait at step k: the stages k .. issued-1 may still be in flight (each the
    // next phase of its slot; earlier ones were consumed); let them land before the block exits
    if (tid == 0 && abort_s)
        for (int j = k; j < issued; ++j)
            (void)prism::tc::mbar_wait(prism::tc::smem_u32(&mb[j % CB_STAGES]), (uint32_t)((j / CB_STAGES) & 1),
                                       1000000000ull);
}

// fixup: o = o0 + Qhat S_start^T for the chunks of tracked segments, on tcgen05: one CTA of 4 warps
// (one per tensor-memory lane quarter) per pair of consecutive chunks of a segment, several CTAs
// per SM.  A = [Qhat_c; Qhat_{c+1}] (128 token rows, K-major) and B = S_start (fp16 [c][m]) come by
// TMA; one product M = 128, N = 64, K = 64; o0 is added in the epilogue (thread = token row) and a
// bf16 result leaves by TMA stores, an fp32 one by 16-byte stores.
constexpr int FX_THREADS = 128;
constexpr uint32_t FX_PANEL = 8192;
constexpr uint32_t FX_OFF_S = 0;                      // S_start [64][64] fp16
constexpr uint32_t FX_OFF_Q = FX_PANEL;               // [Qhat_c; Qhat_{c+1}] [128][64] fp16
constexpr uint32_t FX_OFF_OUT = FX_OFF_Q + 2 * FX_PANEL;  // output tile [128][64] bf16
// [o0_c; o0_{c+1}] [128][64] fp16 (bf16 output) in the output tile's place: each thread reads its
// row's o0 there before it writes the same bytes of its row's output
constexpr uint32_t FX_OFF_O0 = FX_OFF_OUT;
constexpr uint32_t FX_SMEM = FX_OFF_OUT + 2 * FX_PANEL + 1024;

struct FixParams {
    const void *stash_o;  // [BH][NC][64][64] o0 (fp16, or fp32 with out_f32)
    void *out;
    int *status;
    int T, NC, P, out_f32, has_init;
    unsigned long long wait_ns;
};

__global__ void __launch_bounds__(FX_THREADS)
    fixup_kernel(const __grid_constant__ CUtensorMap tm_s, const __grid_constant__ CUtensorMap tm_qh,
                 const __grid_constant__ CUtensorMap tm_out, const __grid_constant__ CUtensorMap tm_o0, FixParams p)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    __shared__ uint32_t tmem_base_s;
    __shared__ __align__(8) uint64_t mbar[3];  // 0: tiles; 1: product; 2: drain
    __shared__ int abort_s;
    const int tid = threadIdx.x, warp = tid >> 5;
    const int bh = blockIdx.x / p.P, seg = blockIdx.x % p.P, k = blockIdx.y;  // pair k of the segment
    const int c_begin = (int)(((long long)seg * p.NC) / p.P), c_end = (int)(((long long)(seg + 1) * p.NC) / p.P);
    const int c0 = c_begin + 2 * k;
    if ((seg == 0 && !p.has_init) || c0 >= c_end) {  // segment 0 is written by the segment kernel
        grid_dependency_wait();
        allow_dependent_launch();
        return;
    }
    const uint32_t sbase = smem_u32(sm);
    const uint64_t dbase = sdesc(sbase, 0, 0);
    const uint32_t mb_t = smem_u32(&mbar[0]), mb_mma = smem_u32(&mbar[1]);
    if (tid == 0) {
        abort_s = 0;
        for (int i = 0; i < 3; ++i) mbar_init(smem_u32(&mbar[i]), 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 0) tmem_alloc(smem_u32(&tmem_base_s), 64);
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tmem = tmem_base_s;
    grid_dependency_wait();  // the stash of the segment kernel and S_start of the combine
    allow_dependent_launch();

    const size_t ch0 = (size_t)bh * p.NC;
    bool loads_pending = false;
    if (tid == 0) {
        mbar_expect_tx(mb_t, (p.out_f32 ? 3 : 5) * FX_PANEL);
        tma_load_2d(sbase + FX_OFF_S, &tm_s, mb_t, 0, (int)(((size_t)bh * p.P + seg) * 64));
        tma_load_2d(sbase + FX_OFF_Q, &tm_qh, mb_t, 0, (int)((ch0 + c0) * 64));
        if (!p.out_f32) tma_load_2d(sbase + FX_OFF_O0, &tm_o0, mb_t, 0, (int)((ch0 + c0) * 64));
        loads_pending = true;
    }
    // o0 of this thread's row while the tiles load
    const int r = tid, chunk = c0 + (r >> 6), i = r & 63;
    const bool valid = chunk < c_end && chunk * 64 + i < p.T;
    float o[64];  // an fp32 o0 row (fp32 output); the fp16 one comes with the tiles
    if (valid) {
        const size_t base = ((ch0 + chunk) * 64 + i) * 64;
        if (p.out_f32) {
            const float4 *src = reinterpret_cast<const float4 *>(p.stash_o) + base / 4;
#pragma unroll
            for (int e = 0; e < 16; ++e) {
                const float4 v = src[e];
                o[4 * e] = v.x;
                o[4 * e + 1] = v.y;
                o[4 * e + 2] = v.z;
                o[4 * e + 3] = v.w;
            }
        }
    }
    if (tid == 0) {
        if (mbar_wait(mb_t, 0, p.wait_ns)) {
            loads_pending = false;
            fence_after_sync();
            const uint32_t id = idesc_f16(128, 64, 0, 0);
#pragma unroll
            for (int s = 0; s < 4; ++s)
                mma_f16(tmem, dsc(dbase, FX_OFF_Q + s * 32, 16, 1024), dsc(dbase, FX_OFF_S + s * 32, 16, 1024), id, s > 0);
            mma_commit(mb_mma);
        } else {
            abort_s = 1;
            set_status(p.status, kDevTimeout);
        }
    }
    __syncthreads();
    if (abort_s == 0) {
        if (!mbar_wait(mb_mma, 0, p.wait_ns)) {
            abort_s = 1;
            set_status(p.status, kDevTimeout);
        }
        fence_after_sync();
        const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
#pragma unroll
        for (int g = 0; g < 2; ++g) {
            float v[32];
            tmem_ld(tmem + lane_off + (uint32_t)(32 * g), v);
            if (!valid) continue;
            if (p.out_f32) {
#pragma unroll
                for (int q = 0; q < 32; ++q) v[q] += o[32 * g + q];
            } else {
#pragma unroll
                for (int q = 0; q < 4; ++q) {  // o0 row r of the staged pair, 8 columns a 16-byte granule
                    const uint4 w = *reinterpret_cast<const uint4 *>(sm + FX_OFF_O0 + sw128(r, 32 * g + 8 * q));
                    const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                    for (int h2 = 0; h2 < 4; ++h2) {
                        const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&ww[h2]));
                        v[8 * q + 2 * h2] += f.x;
                        v[8 * q + 2 * h2 + 1] += f.y;
                    }
                }
            }
            if (p.out_f32) {
                float4 *dst = reinterpret_cast<float4 *>(reinterpret_cast<float *>(p.out) +
                                                         ((size_t)bh * p.T + (size_t)chunk * 64 + i) * 64 + 32 * g);
#pragma unroll
                for (int q = 0; q < 8; ++q) dst[q] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
            } else {
                uint8_t *op = sm + FX_OFF_OUT + (uint32_t)(r >> 6) * FX_PANEL;
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    uint32_t w[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const __nv_bfloat162 b2 = __floats2bfloat162_rn(v[8 * q + 2 * e], v[8 * q + 2 * e + 1]);
                        w[e] = *reinterpret_cast<const uint32_t *>(&b2);
                    }
                    *reinterpret_cast<uint4 *>(op + sw128(i, 32 * g + 8 * q)) = make_uint4(w[0], w[1], w[2], w[3]);
                }
            }
        }
        fence_async_smem();
    }
    fence_before_sync();
    __syncthreads();
    if (tid == 0) {
        if (!p.out_f32 && abort_s == 0) {  // the TMA store drops rows past T
            tma_store_3d(&tm_out, sbase + FX_OFF_OUT, 0, c0 * 64, bh);
            if (c0 + 1 < c_end) tma_store_3d(&tm_out, sbase + FX_OFF_OUT + FX_PANEL, 0, (c0 + 1) * 64, bh);
            bulk_commit();
        }
        bulk_wait_read();  // the output tile has been read (its writes complete with the grid)
        if (abort_s) {  // drain after an expired wait
            if (loads_pending) (void)mbar_wait(mb_t, 0, 1000000000ull);
            const uint32_t mb_drain = smem_u32(&mbar[2]);
            mma_commit(mb_drain);
            (void)mbar_wait(mb_drain, 0, 1000000000ull);
        }
    }
    fence_before_sync();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, 64);
}

}  // namespace tc

// ---------------------------------------------------------------------------------------------
namespace {

PFN_cuTensorMapEncodeTiled_v12000 get_encode()
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

bool encode(CUtensorMap *m, const void *base, int rank, const cuuint64_t *dims, const cuuint64_t *strides_bytes,
            const cuuint32_t *box, CUtensorMapSwizzle sw,
            CUtensorMapDataType dt = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16)
{
    auto fn = get_encode();
    if (!fn) return false;
    cuuint32_t es[5] = {1, 1, 1, 1, 1};
    return fn(m, dt, (cuuint32_t)rank, const_cast<void *>(base), dims, strides_bytes, box,
              es, CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool tc_supported(const Shape &s, prism_dtype io)
{
    return io == PRISM_BF16 && s.dk == 64 && s.dv == 64 && s.L >= 1 && s.L <= 1 + tc::RMAX;
}

int tc_segments(const Shape &s, int sm_count, long long opt)
{
    int P = opt > 0 ? (int)opt : sm_count / (s.BH > 0 ? s.BH : 1);
    if (P < 1) P = 1;
    if (P > s.NC) P = s.NC;
    return P;
}

size_t tc_workspace_bytes(const Shape &s, int P)
{
    const size_t BH = s.BH, NC = s.NC;
    return BH * P * 128 * 64 * 4 + BH * P * 64 * 64 * 2 + BH * NC * 4096 * 4 + BH * NC * 4096 * 2 + 4 * 256;
}

void tc_carve(const Shape &s, int P, void *base, TcWorkspace *w)
{
    const size_t BH = s.BH, NC = s.NC;
    uintptr_t p = ((uintptr_t)base + 255) & ~(uintptr_t)255;
    w->zsum = (float *)p;
    p += BH * P * 128 * 64 * 4;
    p = (p + 255) & ~(uintptr_t)255;
    w->sstart = (__half *)p;
    p += BH * P * 64 * 64 * 2;
    p = (p + 255) & ~(uintptr_t)255;
    w->stash_o = (float *)p;
    p += BH * NC * 4096 * 4;
    p = (p + 255) & ~(uintptr_t)255;
    w->stash_q = (__half *)p;
    w->P = P;
}

cudaError_t tc_prepare()
{
    cudaError_t e = cudaFuncSetAttribute(tc::segment_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)tc::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(tc::fixup_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)tc::FX_SMEM);
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(tc::combine_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)tc::CB_SMEM_LAUNCH);
}

cudaError_t tc_forward(const Shape &s, const ForwardArgs &a, bool out_f32, const TcWorkspace &w, int *d_status,
                       long long wait_ns, KernelTimer &tm)
{
    using namespace tc;
    CUtensorMap mq, mk, mv, mu;
    const cuuint64_t BH = s.BH, T = s.T;
    {
        cuuint64_t dims[3] = {(cuuint64_t)D, T, BH};
        cuuint64_t str[2] = {(cuuint64_t)D * 2, T * D * 2};
        cuuint32_t box[3] = {64, 64, 1};
        if (!encode(&mq, a.q, 3, dims, str, box, CU_TENSOR_MAP_SWIZZLE_128B)) return cudaErrorInvalidValue;
        if (!encode(&mk, a.k, 3, dims, str, box, CU_TENSOR_MAP_SWIZZLE_128B)) return cudaErrorInvalidValue;
        cuuint32_t vbox[3] = {64, 72, 1};
        if (!encode(&mv, a.v, 3, dims, str, vbox, CU_TENSOR_MAP_SWIZZLE_NONE)) return cudaErrorInvalidValue;
    }
    if (s.R > 0) {
        cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)s.R, T, BH};
        cuuint64_t str[3] = {(cuuint64_t)D * 2, (cuuint64_t)s.R * D * 2, T * s.R * D * 2};
        cuuint32_t box[4] = {64, 1, 64, 1};
        if (!encode(&mu, a.u, 4, dims, str, box, CU_TENSOR_MAP_SWIZZLE_128B)) return cudaErrorInvalidValue;
    } else {
        mu = mk;  // never read with L = 1
    }
    SegParams p;
    p.beta = a.beta;
    p.alpha = a.alpha;
    p.gamma = a.gamma;
    p.eta = a.eta;
    p.conv_w = (const __nv_bfloat16 *)a.conv_w;
    p.out = a.out;
    p.out_f32 = out_f32 ? 1 : 0;
    p.zsum = w.zsum;
    p.stash_o = w.stash_o;
    p.stash_q = w.stash_q;
    p.v_hist = (const __nv_bfloat16 *)a.v_hist;
    p.p_gain = (const __nv_bfloat16 *)a.p_gain;
    p.has_init = a.S_init != nullptr;
    p.status = d_status;
    p.H = s.H;
    p.T = s.T;
    p.R = s.R;
    p.NC = s.NC;
    p.P = w.P;
    p.wait_ns = wait_ns > 0 ? (unsigned long long)wait_ns : 100000000ull;
    cudaStream_t st = tm.stream;
    // programmatic stream serialization: each kernel's blocks may be scheduled while the previous
    // kernel drains; the kernels wait (griddepcontrol.wait) before touching memory it produces
    cudaLaunchAttribute pdl[1];
    pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    pdl[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.stream = st;
    cfg.attrs = pdl;
    cfg.numAttrs = 1;
    tm.begin("tc_segment");
    cfg.gridDim = dim3(s.BH * w.P);
    cfg.blockDim = dim3(NT);
    cfg.dynamicSmemBytes = SMEM_BYTES;
    cudaError_t e = cudaLaunchKernelEx(&cfg, segment_kernel, mq, mk, mv, mu, p);
    tm.end();
    if (e != cudaSuccess) return e;
    if (w.P > 1 || a.S_init || a.S_final) {
        tm.begin("tc_combine");
        cfg.gridDim = dim3(s.BH, 64 / CB_ROWS);
        cfg.blockDim = dim3(CB_THREADS);
        cfg.dynamicSmemBytes = CB_SMEM_LAUNCH;
        e = cudaLaunchKernelEx(&cfg, combine_kernel, (const float *)w.zsum, w.sstart, (int)w.P, a.S_init, a.S_final,
                               d_status, (unsigned long long)p.wait_ns);
        tm.end();
        if (e != cudaSuccess) return e;
    }
    if (w.P > 1 || a.S_init) {
        tm.begin("tc_fixup");
        CUtensorMap ms, mqh, mo, mo0;
        {
            cuuint64_t str[1] = {(cuuint64_t)D * 2};
            cuuint64_t dS[2] = {(cuuint64_t)D, (cuuint64_t)s.BH * w.P * 64}, dQ[2] = {(cuuint64_t)D, (cuuint64_t)s.BH * s.NC * 64};
            cuuint32_t b64[2] = {64, 64}, b128[2] = {64, 128};
            if (!encode(&ms, w.sstart, 2, dS, str, b64, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_DATA_TYPE_FLOAT16) ||
                !encode(&mqh, w.stash_q, 2, dQ, str, b128, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_DATA_TYPE_FLOAT16))
                return cudaErrorInvalidValue;
            if (out_f32) {
                mo = mo0 = mqh;  // not read: an fp32 output is written directly, its o0 read by the threads
            } else {
                if (!encode(&mo0, w.stash_o, 2, dQ, str, b128, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_DATA_TYPE_FLOAT16))
                    return cudaErrorInvalidValue;
                cuuint64_t dims[3] = {(cuuint64_t)D, T, BH};
                cuuint64_t ostr[2] = {(cuuint64_t)D * 2, T * D * 2};
                cuuint32_t box[3] = {64, 64, 1};
                if (!encode(&mo, a.out, 3, dims, ostr, box, CU_TENSOR_MAP_SWIZZLE_128B)) return cudaErrorInvalidValue;
            }
        }
        FixParams fp;
        fp.stash_o = w.stash_o;
        fp.out = a.out;
        fp.status = d_status;
        fp.T = s.T;
        fp.NC = s.NC;
        fp.P = w.P;
        fp.out_f32 = p.out_f32;
        fp.has_init = p.has_init;
        fp.wait_ns = p.wait_ns;
        const int max_pairs = (s.NC / w.P + 2) / 2;  // chunk pairs of the longest segment
        cfg.gridDim = dim3(s.BH * w.P, max_pairs);
        cfg.blockDim = dim3(FX_THREADS);
        cfg.dynamicSmemBytes = FX_SMEM;
        e = cudaLaunchKernelEx(&cfg, fixup_kernel, ms, mqh, mo, mo0, fp);
        tm.end();
        if (e != cudaSuccess) return e;
    }
    if (a.v_hist_out) {  // a plain launch: it runs after every kernel above has finished reading v_hist
        e = launch_history(s, PRISM_BF16, a.v_hist, a.v, a.v_hist_out, tm);
        if (e != cudaSuccess) return e;
    }
    return cudaGetLastError();
}

}  // namespace prism

#ifdef PRISM_PHASE_TIMERS
// developer tracing build only: copy out (and optionally clear) the per-phase cycle totals
extern "C" __attribute__((visibility("default"))) int prism_debug_phase_cycles(unsigned long long *out, int reset)
{
    if (cudaMemcpyFromSymbol(out, prism_tc_phase_cycles, sizeof(unsigned long long) * kPhaseSlots) != cudaSuccess)
        return -1;
    if (reset) {
        unsigned long long z[kPhaseSlots] = {0};
        if (cudaMemcpyToSymbol(prism_tc_phase_cycles, z, sizeof(z)) != cudaSuccess) return -1;
    }
    return 0;
}
#endif
