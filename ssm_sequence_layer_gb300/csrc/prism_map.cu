// Chunk-map path of the PRISM memory-recurrence forward (sm_103a: tcgen05 + TMA), for
// dk = dv = 128, 1 <= L <= 16, bf16 io.
//
// The recurrence over one 64-token chunk is an affine map of the state entering it (notes on
// PRISM, section 2.2, the A/B form S_t = S_{t-1} A_t + B_t, composed over the chunk), and the
// chunk's outputs are affine in that state too:
//   S_next = S A_c + B_c,      O = O_loc + Q~ S^T.
// Two kernels:
//   map   one CTA per SM, looping over chunks (every chunk independent of the others): the prep
//         (anchor, gain, residual chain), the Gram tiles of every level, the UT solve, the WY
//         factors, and the four map tensors A_c [dk][dk], B_c [dv][dk], Q~ [C][dk], O_loc [C][dv]
//         (fp16) written to the plan's workspace.
//   scan  one CTA per sequence: S <- S A_c + B_c and o = O_loc + Q~ S^T chunk after chunk, the
//         maps streamed through a two-stage TMA ring, both products on the tensor core.
//
// Chunk algebra (local index i, j; lambda_i = sum_{m<=i} ln alpha_m; lc = lambda_{C-1};
// D_ij = e^{lambda_i - lambda_j} (j <= i); colf_j = e^{lc - lambda_j}; Gamma_i = e^{lambda_i}),
// with the level key tiles U_{-1} = K, U_l (l < R) and x_{t,l} = gamma_{t,l} g_t (.) r_{t,l} (or, for
// the non-linear residual chain of the notes' section 2.3, x_{t,l} = gamma_{t,l} GELU(p_{t,l} r_{t,l})
// with r_{t,l+1} = r_{t,l} - GELU(p_{t,l} r_{t,l})):
//   Gram of level l:  [Q; K] U_l^T  -> rows i < 64: q_i.u_{j,l}, rows 64 + i: k_i.u_{j,l}
//   G~ = D o (Q K^T) (j <= i),  A = diag(beta) D o (K K^T) (j < i)  ->  T = (I + A)^{-1}
//   PQ_l = D o (Q U_l^T) (j <= i),  PK_l = D o (K U_l^T) (j < i)
//   [O_X ; MX] = sum_l [PQ_l ; PK_l] X_l,    B_X = sum_l X_l^T U'_l   (U'_l = diag(colf) U_l)
//   RHS = diag(beta) (V - MX),  U' = T RHS,  W = T diag(beta Gamma) K,  K' = diag(colf) K
//   B_c = B_X + U'^T K',  O_loc = O_X + G~ U',  A_c = Gamma_C I - W^T K',  Q~ = diag(Gamma) Q - G~ W
// Every decay a product needs is applied in fp32 before an operand is rounded to fp16 (the pair
// decays on the score tiles, colf on the state-side key tiles), so fp16 underflow only drops
// contributions below its range, however strong the decay.
//
// Products (tcgen05.mma kind::f16, fp32 accumulators in tensor memory): the Grams on the bf16
// input tiles; everything after them on fp16 operands (10-bit mantissa), the computed operands
// staying of order one.
#include <cuda_fp16.h>
#include <cudaTypedefs.h>

#include "prism_internal.h"
#include "tc_ptx.h"
#include "tc_util.h"

// Developer tracing: with -DPRISM_PHASE_TIMERS thread 0 of every CTA accumulates clock64() cycles
// per phase of the chunk loop (slots 0..7: map kernel, 8..15: scan kernel) into
// prism_map_phase_cycles.
#ifdef PRISM_PHASE_TIMERS
__device__ unsigned long long prism_map_phase_cycles[16];
#define MAP_MARK(k)                                            \
    do {                                                       \
        if (threadIdx.x == 0) {                                \
            const long long now_ = clock64();                  \
            ph_acc[k] += (unsigned long long)(now_ - ph_last); \
            ph_last = now_;                                    \
        }                                                      \
    } while (0)
#else
#define MAP_MARK(k) \
    do {            \
    } while (0)
#endif

namespace prism {
namespace mp {

using namespace tc;
using tcu::dsc;
using tcu::Flag;
using tcu::pack_h2;
using tcu::set_status;
using tcu::st_row_h;

constexpr int C = kChunk;
constexpr int D = 128;       // dk = dv
constexpr int RM = 15;       // levels handled (L <= 16)
constexpr int RMS = 16;      // row stride of the per-token level scalars
constexpr int NT = 512;      // threads of the map kernel: 16 warps, 4 per TMEM lane quarter
constexpr uint32_t PANEL = 8192;  // [64 rows][64 cols] 16-bit SW128

// ---- map kernel: shared memory (bytes from a 1024-aligned base) -------------------------------
// Two regions alternate between chunks: one holds the chunk's [Q_p0 | K_p0 | Q_p1 | K_p1] (bf16; K
// later K' fp16), the other its A and T (fp32) for the solve; once the solve is done the latter
// receives the next chunk's Q and K, so their loads run under the rest of the chunk.
constexpr uint32_t REGION = 34 * 1024;
constexpr uint32_t OFF_R0 = 0, OFF_R1 = REGION;
constexpr uint32_t AT_T32 = 64 * tcu::LDA * 4;       // T32 after A within the solve region
constexpr uint32_t OFF_V = 2 * REGION;               // V rows t0-8 .. t0+63, [72][128] bf16, unswizzled
constexpr uint32_t VBYTES = 72 * D * 2;
constexpr uint32_t OFF_G = OFF_V + VBYTES;           // G~ [64][64] fp16 K-major
constexpr uint32_t OFF_TF = OFF_G + PANEL;           // T  [64][64] fp16 K-major
constexpr uint32_t OFF_LV = OFF_TF + PANEL;          // two level buffers
constexpr uint32_t LVB = 3 * 2 * PANEL;              // per level buffer: U (2 panels) | [PQ; PK] | X (2 panels)
constexpr uint32_t LV_U = 0, LV_PQK = 2 * PANEL, LV_X = 4 * PANEL;
// after the level loop the level buffers hold RHS, diag(beta Gamma) K, U' and W ([64][128] fp16),
// and at the end of the chunk the map tensors on their way out (A_c, B_c [128][128], Q~, O_loc
// [64][128], fp16, SW128 panels of 64 columns)
constexpr uint32_t OFF_RHS = OFF_LV, OFF_BGK = OFF_LV + 2 * PANEL, OFF_UP = OFF_LV + 4 * PANEL,
                   OFF_W = OFF_LV + 6 * PANEL;
constexpr uint32_t OUT_A = OFF_LV, OUT_B = OFF_LV + 4 * PANEL, OUT_Q = OFF_LV + 8 * PANEL, OUT_O = OFF_LV + 10 * PANEL;
constexpr uint32_t OFF_SC = OFF_LV + 2 * LVB;        // per-token scalars
constexpr uint32_t SC_FLOATS = 6 * 64 + 2 * 64 * RMS + tcu::SOLVE_SCRATCH;
constexpr uint32_t MAP_SMEM = OFF_SC + SC_FLOATS * 4 + 1024;  // + alignment slack

static_assert(2 * AT_T32 <= REGION && 4 * PANEL <= REGION, "the alternating regions hold Q/K or A/T");
static_assert(OFF_V % 1024 == 0 && OFF_G % 1024 == 0 && OFF_TF % 1024 == 0 && OFF_LV % 1024 == 0 &&
                  LVB % 1024 == 0 && OFF_SC % 16 == 0 && REGION % 1024 == 0,
              "alignment of the tiles");
static_assert(OFF_W + 2 * PANEL <= OFF_LV + 2 * LVB && OUT_O + 2 * PANEL <= OFF_LV + 2 * LVB,
              "post-solve and output tiles fit the level buffers");
static_assert(MAP_SMEM <= 232448, "shared memory budget");

// tensor memory columns (512 allocated)
constexpr uint32_t TM_GRAM = 0;     // two 64-column Gram buffers (by level parity)
constexpr uint32_t TM_OX = 128;     // [O_X ; MX] (rows i < 64: O_loc, rows 64 + i: MX), 128 columns
constexpr uint32_t TM_BX = 256;     // B_c [c][n]
constexpr uint32_t TM_UP = 0;       // U' [i][c]       (after the level loop)
constexpr uint32_t TM_W = 384;      // W  [j][n]
constexpr uint32_t TM_AC = 0;       // W^T K' [m][n]   (after U' and W are in shared memory)
constexpr uint32_t TM_QT = 384;     // G~ W   [i][n]

struct MapParams {
    const float *beta, *alpha, *gamma, *eta;
    const __nv_bfloat16 *conv_w;
    const __nv_bfloat16 *v_hist;  // [BH][3][D] v_{-3..-1}, or null
    const __nv_bfloat16 *p_gain;  // [BH][T][R][D] gains of the non-linear residual chain, or null (linear)
    __half *mA, *mQ, *mB, *mO;    // [BH*NC][128][128], [BH*NC][64][128], [BH*NC][128][128], [BH*NC][64][128]
    int *status;
    int H, T, R, NC, nchunks;
    unsigned long long wait_ns;
};

// ---------------------------------------------------------------------------------------------
__global__ void __launch_bounds__(NT, 1)
    map_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
               const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_u,
               const __grid_constant__ CUtensorMap tm_ma, const __grid_constant__ CUtensorMap tm_mq,
               const __grid_constant__ CUtensorMap tm_mb, const __grid_constant__ CUtensorMap tm_mo, MapParams p)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    __shared__ uint32_t tmem_base_s;
    __shared__ __align__(8) uint64_t mbar[8];  // 0 Q/K/V, 1-2 U buffers, 3 Gram, 4-5 level products, 6 post products, 7 drain
    __shared__ int abort_s;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int quad = warp & 3, sub = warp >> 2;
    const int row = quad * 32 + lane;  // TMEM lane of this thread in epilogues
    const int R = p.R;

    float *sc = reinterpret_cast<float *>(sm + OFF_SC);
    float *s_beta = sc, *s_lam = sc + 64, *s_rowf = sc + 128, *s_colf = sc + 192, *s_gam = sc + 256,
          *s_bg = sc + 320;
    float *s_gm = sc + 384, *s_et = s_gm + 64 * RMS;  // [64][RMS] gamma, eta
    float *s_xtmp = s_et + 64 * RMS;

    const uint32_t sbase = smem_u32(sm);
    const uint64_t dbase = sdesc(sbase, 0, 0);
    const uint32_t mb_qkv = smem_u32(&mbar[0]), mb_gram = smem_u32(&mbar[3]), mb_post = smem_u32(&mbar[6]);
    const uint32_t mb_u[2] = {smem_u32(&mbar[1]), smem_u32(&mbar[2])};
    const uint32_t mb_lvl[2] = {smem_u32(&mbar[4]), smem_u32(&mbar[5])};

    if (tid == 0) {
        abort_s = 0;
        for (int i = 0; i < 8; ++i) mbar_init(smem_u32(&mbar[i]), 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        prefetch_tmap(&tm_q);
        prefetch_tmap(&tm_k);
        prefetch_tmap(&tm_v);
        prefetch_tmap(&tm_u);
        prefetch_tmap(&tm_ma);
        prefetch_tmap(&tm_mq);
        prefetch_tmap(&tm_mb);
        prefetch_tmap(&tm_mo);
    }
    if (warp == 0) tmem_alloc(smem_u32(&tmem_base_s), 512);
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tmem = tmem_base_s;
    const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
    // the maps this kernel writes may still be read by the previous forward's scan kernel
    grid_dependency_wait();
    allow_dependent_launch();

    // phases of the barriers (every thread tracks the ones it waits on)
    uint32_t ph_qkv = 0, ph_gram = 0, ph_post = 0, ph_u[2] = {0, 0}, ph_lvl[2] = {0, 0};
    // thread 0: the copies it has in flight and the level products it has not waited for
    bool pend_qkv = false, pend_u[2] = {false, false}, pend_lvl[2] = {false, false};
    auto expired = [&]() {
        abort_s = 1;
        set_status(p.status, kDevTimeout);
    };
    // every thread waits on an MMA barrier itself (no CTA barrier needs to follow); after an expiry
    // the chunk loop ends at the next CTA barrier and the drain waits for the products
    auto wait_all = [&](uint32_t mb, uint32_t &ph) {
        if (!mbar_wait(mb, ph, p.wait_ns)) expired();
        ph ^= 1u;
    };
    auto issue_u = [&](int chunk_bh, int t0, int l) {
        const int b = l & 1;
        const uint32_t dst = sbase + OFF_LV + b * LVB + LV_U;
        mbar_expect_tx(mb_u[b], 2 * PANEL);
        tma_load_4d(dst, &tm_u, mb_u[b], 0, l, t0, chunk_bh);
        tma_load_4d(dst + PANEL, &tm_u, mb_u[b], 64, l, t0, chunk_bh);
        pend_u[b] = true;
    };
    // Q, K (into the region `qk`) and V of the chunk with flat index `ch`
    auto issue_qkv = [&](int ch, uint32_t qk) {
        const int cbh = ch / p.NC, ct0 = (ch % p.NC) * C;
        mbar_expect_tx(mb_qkv, 4 * PANEL + VBYTES);
        tma_load_3d(sbase + qk, &tm_q, mb_qkv, 0, ct0, cbh);
        tma_load_3d(sbase + qk + PANEL, &tm_k, mb_qkv, 0, ct0, cbh);
        tma_load_3d(sbase + qk + 2 * PANEL, &tm_q, mb_qkv, 64, ct0, cbh);
        tma_load_3d(sbase + qk + 3 * PANEL, &tm_k, mb_qkv, 64, ct0, cbh);
        tma_load_3d(sbase + OFF_V, &tm_v, mb_qkv, 0, ct0 - 8, cbh);
        pend_qkv = true;
    };

    // this thread's prep elements: channels 2 cp, 2 cp + 1 of tokens tg + 8 k
    const int cp = tid & 63, tg = tid >> 6;
    // gates of one chunk in registers (loaded one chunk ahead, so their latency hides): lanes of
    // warp 0 hold beta and alpha of tokens 2 lane, 2 lane + 1; the other threads two (gamma, eta)
    // entries [i][l] each (64 R <= 2 (NT - 32) entries)
    static_assert(64 * RM <= 2 * (NT - 32), "gate entries per thread");
    float gv[4];
    auto load_gates = [&](int ch) {
        const int cbh = ch / p.NC, ct0 = (ch % p.NC) * C, cn = min(C, p.T - ct0);
        const size_t ctok = (size_t)cbh * p.T + ct0;
        if (warp == 0) {
            const int i0 = 2 * lane, i1 = i0 + 1;
            gv[0] = i0 < cn ? p.beta[ctok + i0] : 0.f;
            gv[1] = i1 < cn ? p.beta[ctok + i1] : 0.f;
            gv[2] = i0 < cn ? p.alpha[ctok + i0] : 1.f;
            gv[3] = i1 < cn ? p.alpha[ctok + i1] : 1.f;
        } else if (R > 0) {
#pragma unroll
            for (int k = 0; k < 2; ++k) {
                const int e = tid - 32 + k * (NT - 32);
                const int i = e / R, l = e % R;
                const bool valid = e < 64 * R && i < cn;
                gv[2 * k] = valid ? p.gamma[(ctok + i) * R + l] : 0.f;
                gv[2 * k + 1] = (valid && p.eta) ? p.eta[(ctok + i) * R + l] : 0.f;
            }
        }
    };
#ifdef PRISM_PHASE_TIMERS
    unsigned long long ph_acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    long long ph_last = clock64();
#endif
    if (tid == 0 && (int)blockIdx.x < p.nchunks) issue_qkv(blockIdx.x, OFF_R0);

    for (int it = 0;; ++it) {
        const int chunk = (int)blockIdx.x + it * (int)gridDim.x;
        if (chunk >= p.nchunks || abort_s) break;
        const int bh = chunk / p.NC, c = chunk % p.NC, h = bh % p.H;
        const int t0 = c * C, n = min(C, p.T - t0);
        const size_t tok0 = (size_t)bh * p.T + t0;
        const uint32_t QK = (it & 1) ? OFF_R1 : OFF_R0;  // this chunk's Q/K
        const uint32_t AT = (it & 1) ? OFF_R0 : OFF_R1;  // this chunk's A/T, then the next chunk's Q/K
        float *const sA = reinterpret_cast<float *>(sm + AT);
        float *const sT32 = reinterpret_cast<float *>(sm + AT + AT_T32);

        // ---- per-token scalars: gates (loaded during the previous chunk), log-decay prefix, decays --
        if (it == 0) load_gates(chunk);
        if (warp == 0) {  // inclusive scan of the 64 log-decays, two per lane
            const int i0 = 2 * lane, i1 = i0 + 1;
            const float b0 = gv[0], b1 = gv[1];
            const float la0 = logf(gv[2]), la1 = logf(gv[3]);
            float s = la0 + la1;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const float y = __shfl_up_sync(0xffffffffu, s, off);
                if (lane >= off) s += y;
            }
            const float l1 = s, l0 = s - la1;
            const float lcw = __shfl_sync(0xffffffffu, s, 31);
            s_beta[i0] = b0;
            s_beta[i1] = b1;
            s_lam[i0] = l0;
            s_lam[i1] = l1;
            s_rowf[i0] = __expf(l0 - lcw);  // used only while the chunk's decay is within fp32 range
            s_rowf[i1] = __expf(l1 - lcw);
            s_colf[i0] = __expf(lcw - l0);
            s_colf[i1] = __expf(lcw - l1);
            s_gam[i0] = __expf(l0);
            s_gam[i1] = __expf(l1);
            s_bg[i0] = b0 * __expf(l0);
            s_bg[i1] = b1 * __expf(l1);
        } else if (R > 0) {  // gamma, eta [i][l] of this chunk
#pragma unroll
            for (int k = 0; k < 2; ++k) {
                const int e = tid - 32 + k * (NT - 32);
                if (e < 64 * R) {
                    const int i = e / R, l = e % R;
                    s_gm[i * RMS + l] = gv[2 * k];
                    s_et[i * RMS + l] = gv[2 * k + 1];
                }
            }
        }
        // Q, K and V have landed (every thread waits; the history, if any, then replaces the halo)
        if (tid == 0) {
            if (mbar_wait(mb_qkv, ph_qkv, p.wait_ns)) pend_qkv = false;
            else expired();
        }
        ph_qkv ^= 1u;
        __syncthreads();
        if (abort_s) break;
        if (c == 0 && p.v_hist != nullptr) {
            if (tid < 48) {  // rows 5..7 of the tile (tokens -3..-1): 3 x 16 groups of 16 bytes
                const uint4 hv = reinterpret_cast<const uint4 *>(p.v_hist + (size_t)bh * 3 * D)[tid];
                *reinterpret_cast<uint4 *>(sm + OFF_V + 5 * D * 2 + tid * 16) = hv;
                fence_async_smem();  // a later TMA rewrites the tile
            }
            __syncthreads();
        }
        const float lc = s_lam[63];
        const bool factored = -lc <= 80.f;  // both decay factors in fp32 range
        MAP_MARK(0);

        // ---- level -1 (the key level): Gram [Q; K] K^T -------------------------------------------
        if (tid == 0) {
            fence_after_sync();
            const uint32_t id = idesc_bf16(128, 64, 0, 0);
#pragma unroll
            for (int s = 0; s < 8; ++s) {
                const uint32_t ko = (uint32_t)(s >> 2) * 2 * PANEL + (uint32_t)(s & 3) * 32;
                mma_f16(tmem + TM_GRAM, dsc(dbase, QK + ko, 16, 1024), dsc(dbase, QK + PANEL + ko, 16, 1024), id, s > 0);
            }
            mma_commit(mb_gram);
            // U_0, U_1 of this chunk into the level buffers, which held the previous chunk's outgoing
            // maps: requested once those stores have read them (they had the chunk's start and the
            // Gram's issue to do so; nothing before the levels touches the buffers)
            bulk_wait_read();
            if (R > 0) issue_u(bh, t0, 0);
            if (R > 1) issue_u(bh, t0, 1);
        }
        // prep, level-independent part: anchor h, gain g, residual r = v - GELU(h)
        float g_[8][2], r_[8][2];
        {
            const __nv_bfloat162 *cw2 = reinterpret_cast<const __nv_bfloat162 *>(p.conv_w) + (size_t)h * 4 * (D / 2) + cp;
            const float2 w0 = __bfloat1622float2(cw2[0]), w1 = __bfloat1622float2(cw2[D / 2]);
            const float2 w2 = __bfloat1622float2(cw2[2 * (D / 2)]), w3 = __bfloat1622float2(cw2[3 * (D / 2)]);
            const __nv_bfloat162 *vb = reinterpret_cast<const __nv_bfloat162 *>(sm + OFF_V);
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const int i = tg + 8 * k;
                const float2 v0 = __bfloat1622float2(vb[(i + 8) * (D / 2) + cp]);
                const float2 v1 = __bfloat1622float2(vb[(i + 7) * (D / 2) + cp]);
                const float2 v2 = __bfloat1622float2(vb[(i + 6) * (D / 2) + cp]);
                const float2 v3 = __bfloat1622float2(vb[(i + 5) * (D / 2) + cp]);
                const float a0 = fmaf(w0.x, v0.x, fmaf(w1.x, v1.x, fmaf(w2.x, v2.x, w3.x * v3.x)));
                const float a1 = fmaf(w0.y, v0.y, fmaf(w1.y, v1.y, fmaf(w2.y, v2.y, w3.y * v3.y)));
                float Phi0, Phi1;
                tcu::gelu_gain(a0, g_[k][0], Phi0);
                tcu::gelu_gain(a1, g_[k][1], Phi1);
                r_[k][0] = v0.x - a0 * Phi0;
                r_[k][1] = v0.y - a1 * Phi1;
            }
        }
        wait_all(mb_gram, ph_gram);
        fence_after_sync();

        // E1 of one level: the Gram buffer `gb` (64 columns) -> decayed, masked score rows.  Thread
        // (quad, sub) holds TMEM row `row` (i = row & 63; rows < 64 the query side, j <= i kept;
        // rows >= 64 the key side, j < i kept) and columns 16 sub .. 16 sub + 15.
        auto scores = [&](uint32_t gb, float (&v)[16], bool &query, int &i) {
            const int j0 = sub * 16;
            i = row & 63;
            query = row < 64;
            float dq[16];
            auto fill = [&](auto form) {
                if constexpr (decltype(form)::value) {
                    const float rf = s_rowf[i];
#pragma unroll
                    for (int g = 0; g < 4; ++g) {
                        const float4 f = reinterpret_cast<const float4 *>(s_colf + j0)[g];
                        dq[4 * g + 0] = rf * f.x;
                        dq[4 * g + 1] = rf * f.y;
                        dq[4 * g + 2] = rf * f.z;
                        dq[4 * g + 3] = rf * f.w;
                    }
                } else {
                    const float li = s_lam[i];
#pragma unroll
                    for (int q = 0; q < 16; ++q) dq[q] = __expf(fminf(li - s_lam[j0 + q], 0.f));
                }
            };
            if (factored)
                fill(Flag<true>{});
            else
                fill(Flag<false>{});
            tmem_ld(tmem + gb + lane_off + (uint32_t)j0, v);
#pragma unroll
            for (int q = 0; q < 16; ++q) {
                const int j = j0 + q;
                v[q] = (query ? j <= i : j < i) ? v[q] * dq[q] : 0.f;
            }
        };
        {
            float v[16];
            bool query;
            int i;
            scores(TM_GRAM, v, query, i);
            if (query) {
                st_row_h(sm + OFF_G, i, sub * 16, v);
            } else {  // A_ij = beta_i D_ij k_i.k_j
                float4 *A4 = reinterpret_cast<float4 *>(sA + i * tcu::LDA + sub * 16);
                const float b = s_beta[i];
#pragma unroll
                for (int g = 0; g < 4; ++g) A4[g] = make_float4(b * v[4 * g], b * v[4 * g + 1], b * v[4 * g + 2], b * v[4 * g + 3]);
            }
        }
        fence_before_sync();
        __syncthreads();
        MAP_MARK(1);

        // ---- levels 0 .. R-1 -------------------------------------------------------------------------
        for (int l = 0; l < R; ++l) {
            const int b = l & 1;
            const uint32_t lvb = OFF_LV + b * LVB;
            // the non-linear chain's gains of this level (read early: their latency hides behind the Gram)
            uint32_t pz[8];
            if (p.p_gain) {
                const uint32_t *pg = reinterpret_cast<const uint32_t *>(p.p_gain) + ((tok0 * R + l) * D) / 2 + cp;
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const int i = tg + 8 * k;
                    pz[k] = i < n ? pg[(size_t)i * R * (D / 2)] : 0u;
                }
            }
            if (tid == 0) {
                // the Gram first (it queues behind level l - 1's products), then the prefetch of U_{l+1}
                // into the other buffer once level l - 1's products have completed
                if (mbar_wait(mb_u[b], ph_u[b], p.wait_ns)) {
                    ph_u[b] ^= 1u;
                    pend_u[b] = false;
                    fence_after_sync();
                    const uint32_t id = idesc_bf16(128, 64, 0, 0);
#pragma unroll
                    for (int s = 0; s < 8; ++s) {
                        const uint32_t ko = (uint32_t)(s >> 2) * 2 * PANEL + (uint32_t)(s & 3) * 32;
                        const uint32_t uo = lvb + LV_U + (uint32_t)(s >> 2) * PANEL + (uint32_t)(s & 3) * 32;
                        mma_f16(tmem + TM_GRAM + 64 * b, dsc(dbase, QK + ko, 16, 1024), dsc(dbase, uo, 16, 1024), id,
                                s > 0);
                    }
                    mma_commit(mb_gram);
                    if (l >= 1 && l + 1 < R) {
                        if (mbar_wait(mb_lvl[b ^ 1], ph_lvl[b ^ 1], p.wait_ns)) {
                            ph_lvl[b ^ 1] ^= 1u;
                            pend_lvl[b ^ 1] = false;
                            issue_u(bh, t0, l + 1);
                        } else {
                            expired();
                        }
                    }
                } else {
                    expired();
                }
            }
            __syncthreads();  // an expiry above is seen by every thread before it waits on the Gram
            if (abort_s) break;
            wait_all(mb_gram, ph_gram);
            fence_after_sync();
            {  // [PQ_l ; PK_l] rows
                float v[16];
                bool query;
                int i;
                scores(TM_GRAM + 64 * b, v, query, i);
                st_row_h(sm + lvb + LV_PQK, row, sub * 16, v);
            }
            // U_l -> U'_l = diag(colf) U_l (fp16, in place; the Gram has read it)
#pragma unroll
            for (int e2 = 0; e2 < 2; ++e2) {
                const int e = tid + NT * e2;  // 16-byte group: panel e >> 9, row (e & 511) >> 3
                uint4 w = reinterpret_cast<const uint4 *>(sm + lvb + LV_U)[e];
                const float sc_j = s_colf[(e & 511) >> 3];
                uint32_t *pw = &w.x;
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&pw[q]));
                    pw[q] = pack_h2(sc_j * f.x, sc_j * f.y);
                }
                reinterpret_cast<uint4 *>(sm + lvb + LV_U)[e] = w;
            }
            // X_l = gamma_l g r, then r <- r (1 - eta_l g); or, with gains p, the non-linear chain
            // delta = GELU(p r), X_l = gamma_l delta, r <- r - delta
            {
                uint8_t *xp = sm + lvb + LV_X + (uint32_t)((2 * cp) >> 6) * PANEL;
                const int col = (2 * cp) & 63;
                if (p.p_gain) {
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        const int i = tg + 8 * k;
                        const float gm = s_gm[i * RMS + l];
                        const float2 pf = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&pz[k]));
                        const float d0 = tcu::gelu_value(pf.x * r_[k][0]), d1 = tcu::gelu_value(pf.y * r_[k][1]);
                        *reinterpret_cast<uint32_t *>(xp + sw128(i, col)) = pack_h2(gm * d0, gm * d1);
                        r_[k][0] -= d0;
                        r_[k][1] -= d1;
                    }
                } else {
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        const int i = tg + 8 * k;
                        const float gm = s_gm[i * RMS + l], et = s_et[i * RMS + l];
                        *reinterpret_cast<uint32_t *>(xp + sw128(i, col)) =
                            pack_h2(gm * g_[k][0] * r_[k][0], gm * g_[k][1] * r_[k][1]);
                        r_[k][0] *= 1.f - et * g_[k][0];
                        r_[k][1] *= 1.f - et * g_[k][1];
                    }
                }
            }
            fence_async_smem();
            fence_before_sync();
            __syncthreads();
            if (tid == 0) {
                fence_after_sync();
                // [O_X ; MX] += [PQ_l ; PK_l] X_l   (A K-major, B = X_l [j][c] MN-major)
                const uint32_t id1 = idesc_f16(128, 128, 0, 1);
#pragma unroll
                for (int s = 0; s < 4; ++s)
                    mma_f16(tmem + TM_OX, dsc(dbase, lvb + LV_PQK + s * 32, 16, 1024),
                            dsc(dbase, lvb + LV_X + s * 2048, PANEL, 1024), id1, (l | s) != 0);
                // B_X += X_l^T U'_l   (A = X_l [j][c] MN-major, B = U'_l [j][n] MN-major)
                const uint32_t id2 = idesc_f16(128, 128, 1, 1);
#pragma unroll
                for (int s = 0; s < 4; ++s)
                    mma_f16(tmem + TM_BX, dsc(dbase, lvb + LV_X + s * 2048, PANEL, 1024),
                            dsc(dbase, lvb + LV_U + s * 2048, PANEL, 1024), id2, (l | s) != 0);
                mma_commit(mb_lvl[b]);
                pend_lvl[b] = true;
            }
        }
        if (abort_s) break;
        MAP_MARK(2);

        // ---- after the levels: the products of the last ones complete, then the solve (warps 8-15)
        // beside the RHS, diag(beta Gamma) K and K' (warps 0-7) ---------------------------------------
        if (tid == 0) {
            for (int b = 0; b < 2; ++b)
                if (pend_lvl[b]) {
                    if (mbar_wait(mb_lvl[b], ph_lvl[b], p.wait_ns)) {
                        ph_lvl[b] ^= 1u;
                        pend_lvl[b] = false;
                    } else {
                        expired();
                    }
                }
        }
        fence_before_sync();
        __syncthreads();
        if (abort_s) break;
        fence_after_sync();
        if (warp >= 8) {
            tcu::ut_solve(sA, sT32, s_xtmp, sm + OFF_TF, tid - 256, 1);
        } else if (quad >= 2) {  // RHS = diag(beta) (V - MX): TMEM rows 64 + i, 64 columns per thread
            const int i = row - 64, c0 = (warp >> 2) * 64;
            const __nv_bfloat16 *vb = reinterpret_cast<const __nv_bfloat16 *>(sm + OFF_V) + (size_t)(i + 8) * D;
            const float bi = s_beta[i];
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                float mx[32];
                if (R > 0) {
                    tmem_ld(tmem + TM_OX + lane_off + (uint32_t)(c0 + 32 * half), mx);
                } else {
#pragma unroll
                    for (int q = 0; q < 32; ++q) mx[q] = 0.f;  // no levels: MX = 0 (never written)
                }
                float rv[32];
#pragma unroll
                for (int q = 0; q < 32; ++q) rv[q] = bi * (__bfloat162float(vb[c0 + 32 * half + q]) - mx[q]);
                st_row_h(sm + OFF_RHS + (uint32_t)(c0 >> 6) * PANEL, i, 32 * half, rv);
            }
        } else {  // diag(beta Gamma) K and K' = diag(colf) K from the bf16 K panels (warps 0, 1, 4, 5)
            const int t = (warp >> 2) * 64 + (warp & 1) * 32 + lane;  // 0..127
            for (int e = t; e < 1024; e += 128) {
                const int pnl = e >> 9, j = (e & 511) >> 3;
                uint8_t *kp = sm + QK + PANEL + (uint32_t)pnl * 2 * PANEL;
                uint4 w = reinterpret_cast<const uint4 *>(kp)[e & 511];
                uint4 wb = w;
                const float bg = s_bg[j], cf = s_colf[j];
                uint32_t *pw = &w.x, *pb = &wb.x;
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&pw[q]));
                    pb[q] = pack_h2(bg * f.x, bg * f.y);
                    pw[q] = pack_h2(cf * f.x, cf * f.y);
                }
                reinterpret_cast<uint4 *>(sm + OFF_BGK + (uint32_t)pnl * PANEL)[e & 511] = wb;
                reinterpret_cast<uint4 *>(kp)[e & 511] = w;
            }
        }
        fence_async_smem();
        fence_before_sync();
        __syncthreads();
        MAP_MARK(3);

        // ---- U' = T RHS, W = T diag(beta Gamma) K; the next chunk's Q, K, V load under the rest ------
        if (tid == 0) {
            fence_after_sync();
            const uint32_t id = idesc_f16(128, 128, 0, 1);  // A = T [i][j] K-major (rows 64.. unused)
#pragma unroll
            for (int s = 0; s < 4; ++s) {
                mma_f16(tmem + TM_UP, dsc(dbase, OFF_TF + s * 32, 16, 1024), dsc(dbase, OFF_RHS + s * 2048, PANEL, 1024), id,
                        s > 0);
                mma_f16(tmem + TM_W, dsc(dbase, OFF_TF + s * 32, 16, 1024), dsc(dbase, OFF_BGK + s * 2048, PANEL, 1024), id,
                        s > 0);
            }
            mma_commit(mb_post);
            // the solve region (A, T) is free and V has been read: prefetch the next chunk's inputs
            const int next = chunk + (int)gridDim.x;
            if (next < p.nchunks) issue_qkv(next, AT);
        }
        {  // the next chunk's gates, while the products run
            const int next = chunk + (int)gridDim.x;
            if (next < p.nchunks) load_gates(next);
        }
        wait_all(mb_post, ph_post);
        fence_after_sync();
        if (quad < 2) {  // rows i < 64: sub 0, 1 -> U' columns, sub 2, 3 -> W columns (64 per thread)
            const bool isw = sub >= 2;
            const int c0 = (sub & 1) * 64;
            const uint32_t src = tmem + (isw ? TM_W : TM_UP) + lane_off + (uint32_t)c0;
            uint8_t *dst = sm + (isw ? OFF_W : OFF_UP) + (uint32_t)(c0 >> 6) * PANEL;
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                float v[32];
                tmem_ld(src + 32 * half, v);
                st_row_h(dst, row, 32 * half, v);
            }
        }
        fence_async_smem();
        fence_before_sync();
        __syncthreads();
        if (abort_s) break;
        MAP_MARK(4);

        // ---- B_c += U'^T K', O_loc += G~ U', W^T K', G~ W ----------------------------------------------
        if (tid == 0) {
            fence_after_sync();
            const uint32_t idmm = idesc_f16(128, 128, 1, 1), idkm = idesc_f16(128, 128, 0, 1);
            const uint32_t kq = QK + PANEL;  // K' panels at 16 KB stride
#pragma unroll
            for (int s = 0; s < 4; ++s) {
                const uint32_t ks = s * 2048;
                mma_f16(tmem + TM_BX, dsc(dbase, OFF_UP + ks, PANEL, 1024), dsc(dbase, kq + ks, 2 * PANEL, 1024), idmm,
                        (R > 0 || s > 0) ? 1u : 0u);
                mma_f16(tmem + TM_OX, dsc(dbase, OFF_G + s * 32, 16, 1024), dsc(dbase, OFF_UP + ks, PANEL, 1024), idkm,
                        (R > 0 || s > 0) ? 1u : 0u);
                mma_f16(tmem + TM_AC, dsc(dbase, OFF_W + ks, PANEL, 1024), dsc(dbase, kq + ks, 2 * PANEL, 1024), idmm, s > 0);
                mma_f16(tmem + TM_QT, dsc(dbase, OFF_G + s * 32, 16, 1024), dsc(dbase, OFF_W + ks, PANEL, 1024), idkm, s > 0);
            }
            mma_commit(mb_post);
        }
        wait_all(mb_post, ph_post);
        fence_after_sync();
        MAP_MARK(5);

        // ---- the map tensors: thread row = TMEM lane, 32 columns per thread, into SW128 panels of
        // the level buffers (free now), then out by TMA stores --------------------------------------
        {
            const int n0 = sub * 32;
            const float gC = __expf(lc);
            const uint32_t pnl = (uint32_t)(n0 >> 6) * 2 * PANEL;  // [128][64] panels of A_c, B_c
            float v[32];
            // A_c [m][n] = Gamma_C [m == n] - (W^T K')[m][n]
            tmem_ld(tmem + TM_AC + lane_off + (uint32_t)n0, v);
#pragma unroll
            for (int q = 0; q < 32; ++q) v[q] = (n0 + q == row ? gC : 0.f) - v[q];
            st_row_h(sm + OUT_A + pnl, row, n0 & 63, v);
            // B_c [c][n]
            tmem_ld(tmem + TM_BX + lane_off + (uint32_t)n0, v);
            st_row_h(sm + OUT_B + pnl, row, n0 & 63, v);
            if (quad < 2) {
                const uint32_t pq = (uint32_t)(n0 >> 6) * PANEL;  // [64][64] panels of Q~, O_loc
                // Q~ [i][n] = Gamma_i Q[i][n] - (G~ W)[i][n]
                tmem_ld(tmem + TM_QT + lane_off + (uint32_t)n0, v);
                const float gi = s_gam[row];
                const uint8_t *qp = sm + QK + (uint32_t)(n0 >> 6) * 2 * PANEL;
#pragma unroll
                for (int e = 0; e < 4; ++e) {  // 16-byte groups of 8 bf16 of the swizzled Q row
                    const uint4 w = *reinterpret_cast<const uint4 *>(qp + sw128(row, (n0 & 63) + 8 * e));
                    const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                    for (int h2 = 0; h2 < 4; ++h2) {
                        const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&ww[h2]));
                        v[8 * e + 2 * h2] = gi * f.x - v[8 * e + 2 * h2];
                        v[8 * e + 2 * h2 + 1] = gi * f.y - v[8 * e + 2 * h2 + 1];
                    }
                }
                st_row_h(sm + OUT_Q + pq, row, n0 & 63, v);
                // O_loc [i][c]
                tmem_ld(tmem + TM_OX + lane_off + (uint32_t)n0, v);
                st_row_h(sm + OUT_O + pq, row, n0 & 63, v);
            }
        }
        fence_async_smem();
        fence_before_sync();
        __syncthreads();  // every read of this chunk's tiles and tensor memory is done
        if (tid == 0) {
            const int ra = chunk * 128, rq = chunk * 64;
            tma_store_2d(&tm_ma, sbase + OUT_A, 0, ra);
            tma_store_2d(&tm_ma, sbase + OUT_A + 2 * PANEL, 64, ra);
            tma_store_2d(&tm_mb, sbase + OUT_B, 0, ra);
            tma_store_2d(&tm_mb, sbase + OUT_B + 2 * PANEL, 64, ra);
            tma_store_2d(&tm_mq, sbase + OUT_Q, 0, rq);
            tma_store_2d(&tm_mq, sbase + OUT_Q + PANEL, 64, rq);
            tma_store_2d(&tm_mo, sbase + OUT_O, 0, rq);
            tma_store_2d(&tm_mo, sbase + OUT_O + PANEL, 64, rq);
            bulk_commit();
        }
        MAP_MARK(6);
    }
#ifdef PRISM_PHASE_TIMERS
    if (tid == 0)
        for (int k = 0; k < 8; ++k) atomicAdd(&prism_map_phase_cycles[k], ph_acc[k]);
#endif

    // drain: after an expired wait, let every copy and product still in flight land (bounded by one
    // second each) before the CTA releases its shared and tensor memory.  One more commit arrives
    // once every product this thread issued has completed.
    if (tid == 0) {
        bulk_wait_all();  // the outgoing maps have been written
        if (abort_s) {
            const uint64_t drain_ns = 1000000000ull;
            if (pend_qkv) (void)mbar_wait(mb_qkv, ph_qkv, drain_ns);
            for (int b = 0; b < 2; ++b)
                if (pend_u[b]) (void)mbar_wait(mb_u[b], ph_u[b], drain_ns);
            const uint32_t mb_drain = smem_u32(&mbar[7]);
            mma_commit(mb_drain);
            (void)mbar_wait(mb_drain, 0, drain_ns);
        }
    }
    fence_before_sync();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, 512);
}

// ---------------------------------------------------------------------------------------------
// scan: two CTAs per sequence, one per half of the value rows (the rows of S evolve independently),
// 8 warps each.  Per chunk: D1 = S_h A_c and D2 = Q~ S_h^T (S_h, this CTA's 64 state rows, fp16 in
// shared memory, K-major [c][m]), then S_h <- D1 + B_c (rows c < 64: warps of lane quarters 0-1,
// 64 columns per thread) and o = D2 + O_loc for the chunk's tokens and this half's 64 channels.
// A_c, Q~ and this half of B_c stream through a three-stage ring of TMA copies; a stage is refilled
// as soon as the products have read it and B_c has been taken into registers.  O_loc is read from
// global memory into registers at the start of the step; a bf16 output leaves through a
// shared-memory tile and a TMA store.
// v[o .. o + 7] += the 8 halves of w
template <int N>
__device__ __forceinline__ void add_h8(float (&v)[N], int o, const uint4 w)
{
    const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int h2 = 0; h2 < 4; ++h2) {
        const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&ww[h2]));
        v[o + 2 * h2] += f.x;
        v[o + 2 * h2 + 1] += f.y;
    }
}

__device__ __forceinline__ uint32_t pack_b2(float a, float b)
{
    const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<const uint32_t *>(&h);
}

constexpr int ST = 256;
constexpr int SC_STAGES = 3;
constexpr uint32_t SC_OFF_S = 0;  // S_h: 2 panels [64 rows][64] fp16 (8 KB each)
constexpr uint32_t STAGE = 4 * PANEL + 2 * PANEL + 2 * PANEL;  // A_c | Q~ | B_c rows of this half
constexpr uint32_t SG_A = 0, SG_Q = 4 * PANEL, SG_B = 6 * PANEL;
constexpr uint32_t SC_OFF_ST = 2 * PANEL;
constexpr uint32_t SC_OFF_OUT = SC_OFF_ST + SC_STAGES * STAGE;  // bf16 output tile: [64 tokens][64 channels]
constexpr uint32_t SCAN_SMEM = SC_OFF_OUT + PANEL + 1024;
static_assert(SCAN_SMEM <= 232448, "shared memory budget");
constexpr uint32_t TM_D1 = 0, TM_D2 = 128;

struct ScanParams {
    const float *S_init;  // [BH][D][D] or null
    float *S_final;       // [BH][D][D] or null
    float *S_seg;         // with G > 1: the state entering each segment, [BH][G][D][D]
    float *seg_maps;      // the compose pass's output: [BH][G][2][D][D] (B_seg, A_seg)
    int G;                // segments a sequence (the chunks of segment g: g NC / G .. (g + 1) NC / G - 1)
    const __half *mO;     // [BH*NC][64][128] O_loc
    void *out;            // [BH][T][D] bf16, or fp32 with out_f32
    int *status;
    int T, NC, out_f32;
    unsigned long long wait_ns;
};

__global__ void __launch_bounds__(ST, 1)
    scan_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_qt,
                const __grid_constant__ CUtensorMap tm_b, const __grid_constant__ CUtensorMap tm_out, ScanParams p)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    __shared__ uint32_t tmem_base_s;
    __shared__ __align__(8) uint64_t mbar[SC_STAGES + 2];  // ring stages; products; drain
    __shared__ int abort_s;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int quad = warp & 3, half = warp >> 2;  // TMEM lane quarter; column half of the epilogues
    const int row = quad * 32 + lane;             // state row / token within this half (< 64: live)
    const bool live = quad < 2;
    // block (sequence bh, segment seg, half vh of the value rows)
    const int vh = blockIdx.x & 1, seg = (int)(blockIdx.x >> 1) % p.G, bh = (int)(blockIdx.x >> 1) / p.G;
    const int r0 = 64 * vh;  // first state row / channel of this half
    const int cb = (int)((long long)seg * p.NC / p.G), ce = (int)((long long)(seg + 1) * p.NC / p.G);
    const float *s_in = p.G > 1 ? p.S_seg + ((size_t)bh * p.G + seg) * D * D
                                : (p.S_init ? p.S_init + (size_t)bh * D * D : nullptr);
    const uint32_t sbase = smem_u32(sm);
    const uint64_t dbase = sdesc(sbase, 0, 0);
    const uint32_t mb_mma = smem_u32(&mbar[SC_STAGES]);

    if (tid == 0) {
        abort_s = 0;
        for (int i = 0; i < SC_STAGES + 2; ++i) mbar_init(smem_u32(&mbar[i]), 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        prefetch_tmap(&tm_a);
        prefetch_tmap(&tm_qt);
        prefetch_tmap(&tm_b);
        prefetch_tmap(&tm_out);
    }
    if (p.G > 1) grid_dependency_wait();  // the segments' start states (the carry pass)
    if (warp == 0) tmem_alloc(smem_u32(&tmem_base_s), 256);
    // the initial state (fp16 operand copy): row `row`, 64 columns of this thread's half
    if (live) {
        uint8_t *sp = sm + SC_OFF_S + (uint32_t)half * PANEL;
#pragma unroll
        for (int g = 0; g < 2; ++g) {
            float w[32];
#pragma unroll
            for (int q = 0; q < 32; ++q)
                w[q] = s_in ? s_in[(size_t)(r0 + row) * D + 64 * half + 32 * g + q] : 0.f;
            st_row_h(sp, row, 32 * g, w);
        }
    }
    fence_async_smem();
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tmem = tmem_base_s;
    const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
    grid_dependency_wait();  // the maps of the map kernel
    allow_dependent_launch();

    const int NC = p.NC, nk = ce - cb;
    const size_t ch0 = (size_t)bh * NC;
    auto issue = [&](int k) {  // chunk cb + k's A_c, Q~ and this half of B_c into stage k % SC_STAGES
        const int c = cb + k, st = k % SC_STAGES;
        const uint32_t base = sbase + SC_OFF_ST + st * STAGE, mb = smem_u32(&mbar[st]);
        const int ra = (int)((ch0 + c) * 128), rq = (int)((ch0 + c) * 64);
        mbar_expect_tx(mb, STAGE);
        tma_load_2d(base + SG_A, &tm_a, mb, 0, ra);
        tma_load_2d(base + SG_A + 2 * PANEL, &tm_a, mb, 64, ra);
        tma_load_2d(base + SG_Q, &tm_qt, mb, 0, rq);
        tma_load_2d(base + SG_Q + PANEL, &tm_qt, mb, 64, rq);
        tma_load_2d(base + SG_B, &tm_b, mb, 0, ra + r0);
        tma_load_2d(base + SG_B + PANEL, &tm_b, mb, 64, ra + r0);
    };
    uint32_t ph_mma = 0;
    int issued = 0, consumed = 0;  // thread 0: chunks whose maps were requested / have landed
    if (tid == 0) {
        for (; issued < SC_STAGES && issued < nk; ++issued) issue(issued);
    }
    bool finite = true;
#ifdef PRISM_PHASE_TIMERS
    unsigned long long ph_acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    long long ph_last = clock64();
#endif
    for (int k = 0; k < nk && abort_s == 0; ++k) {
        const int c = cb + k, st = k % SC_STAGES;
        const uint32_t sb = SC_OFF_ST + st * STAGE;
        if (tid == 0) {
            if (mbar_wait(smem_u32(&mbar[st]), (uint32_t)((k / SC_STAGES) & 1), p.wait_ns)) {
                ++consumed;
                fence_after_sync();
                // D1 = S_h A_c (A = S_h [c][m] K-major, rows 64.. unused; B = A_c [m][n] MN-major);
                // D2 = Q~ S_h^T (A = Q~ [i][n] K-major, rows 64.. unused; B = S_h [c][m] as N x K)
                const uint32_t id1 = idesc_f16(128, 128, 0, 1), id2 = idesc_f16(128, 64, 0, 0);
#pragma unroll
                for (int s = 0; s < 8; ++s) {
                    const uint32_t so = SC_OFF_S + (uint32_t)(s >> 2) * PANEL + (uint32_t)(s & 3) * 32;
                    mma_f16(tmem + TM_D1, dsc(dbase, so, 16, 1024), dsc(dbase, sb + SG_A + s * 2048, 2 * PANEL, 1024), id1,
                            s > 0);
                }
#pragma unroll
                for (int s = 0; s < 8; ++s) {
                    const uint32_t so = SC_OFF_S + (uint32_t)(s >> 2) * PANEL + (uint32_t)(s & 3) * 32;
                    const uint32_t qo = sb + SG_Q + (uint32_t)(s >> 2) * PANEL + (uint32_t)(s & 3) * 32;
                    mma_f16(tmem + TM_D2, dsc(dbase, qo, 16, 1024), dsc(dbase, so, 16, 1024), id2, s > 0);
                }
                mma_commit(mb_mma);
            } else {
                abort_s = 1;
                set_status(p.status, kDevTimeout);
            }
        }
        // O_loc of this thread's token row and 32 channels, from global memory while the products run
        uint4 ol[4];
        if (live) {
            const uint4 *src = reinterpret_cast<const uint4 *>(p.mO + ((ch0 + c) * 64 + row) * D + r0 + 32 * half);
#pragma unroll
            for (int e = 0; e < 4; ++e) ol[e] = src[e];
        }
        __syncthreads();
        if (abort_s) break;
        MAP_MARK(0);
        // B_c of this thread's state row (64 columns) into registers, so that the stage can be refilled
        uint4 bc[8];
        if (live) {
            const uint8_t *bp = sm + sb + SG_B + (uint32_t)half * PANEL;
#pragma unroll
            for (int e = 0; e < 8; ++e) bc[e] = *reinterpret_cast<const uint4 *>(bp + sw128(row, 8 * e));
        }
        if (!mbar_wait(mb_mma, ph_mma, p.wait_ns)) {
            abort_s = 1;
            set_status(p.status, kDevTimeout);
        }
        ph_mma ^= 1u;
        if (tid == 0) bulk_wait_read();  // the previous chunk's output tile has been read out
        fence_before_sync();
        __syncthreads();  // stage st is consumed: refill it with chunk c + SC_STAGES
        fence_after_sync();
        if (tid == 0 && issued < nk && abort_s == 0) issue(issued++);
        MAP_MARK(1);
        if (live) {
            // S_h <- S_h A_c + B_c (row `row`, columns 64 half .. 64 half + 63)
            uint8_t *sp = sm + SC_OFF_S + (uint32_t)half * PANEL;
#pragma unroll
            for (int g = 0; g < 2; ++g) {
                float v[32];
                tmem_ld(tmem + TM_D1 + lane_off + (uint32_t)(64 * half + 32 * g), v);
#pragma unroll
                for (int e = 0; e < 4; ++e) add_h8(v, 8 * e, bc[4 * g + e]);
                if (c + 1 == NC && p.S_final) {
                    float4 *sf = reinterpret_cast<float4 *>(p.S_final + ((size_t)bh * D + r0 + row) * D + 64 * half + 32 * g);
#pragma unroll
                    for (int q = 0; q < 8; ++q) sf[q] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
                }
                st_row_h(sp, row, 32 * g, v);
            }
        }
        MAP_MARK(2);
        if (live) {
            // o = Q~ S_h^T + O_loc: token `row`, this half's channels 32 half .. 32 half + 31
            const int n = min(C, p.T - c * C);
            float v[32];
            tmem_ld(tmem + TM_D2 + lane_off + (uint32_t)(32 * half), v);
#pragma unroll
            for (int e = 0; e < 4; ++e) add_h8(v, 8 * e, ol[e]);
#pragma unroll
            for (int q = 0; q < 32; ++q) finite = finite && isfinite(v[q]);
            if (!p.out_f32) {  // into the output tile (the TMA store drops rows past T)
                uint8_t *op = sm + SC_OFF_OUT;
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    *reinterpret_cast<uint4 *>(op + sw128(row, 32 * half + 8 * q)) =
                        make_uint4(pack_b2(v[8 * q], v[8 * q + 1]), pack_b2(v[8 * q + 2], v[8 * q + 3]),
                                   pack_b2(v[8 * q + 4], v[8 * q + 5]), pack_b2(v[8 * q + 6], v[8 * q + 7]));
            } else if (row < n) {
                const size_t o = ((size_t)bh * p.T + (size_t)c * C + row) * D + r0 + 32 * half;
                float4 *dst = reinterpret_cast<float4 *>(reinterpret_cast<float *>(p.out) + o);
#pragma unroll
                for (int q = 0; q < 8; ++q) dst[q] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
            }
        }
        MAP_MARK(3);
        fence_async_smem();  // S_h is the next chunk's MMA operand; the output tile goes out by TMA
        fence_before_sync();
        __syncthreads();
        fence_after_sync();
        if (tid == 0 && !p.out_f32) {
            tma_store_3d(&tm_out, sbase + SC_OFF_OUT, r0, c * C, bh);
            bulk_commit();
        }
        MAP_MARK(4);
    }
#ifdef PRISM_PHASE_TIMERS
    if (tid == 0)
        for (int k = 0; k < 5; ++k) atomicAdd(&prism_map_phase_cycles[8 + k], ph_acc[k]);
#endif
    if (!finite) set_status(p.status, kDevBounds);  // outside the fp16 operand range
    // drain: the output stores complete; after an expired wait, copies and products still in flight
    // land before the CTA exits
    if (tid == 0) {
        bulk_wait_all();
        if (abort_s) {
            for (int k = consumed; k < issued; ++k)
                (void)mbar_wait(smem_u32(&mbar[k % SC_STAGES]), (uint32_t)((k / SC_STAGES) & 1), 1000000000ull);
            const uint32_t mb_drain = smem_u32(&mbar[SC_STAGES + 1]);
            mma_commit(mb_drain);
            (void)mbar_wait(mb_drain, 0, 1000000000ull);
        }
    }
    fence_before_sync();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, 256);
}

// ---------------------------------------------------------------------------------------------
// Segment maps of the chunk scan, for sequences of many chunks and few sequences.  The compose pass
// runs the scan's step over one segment of G for the block rows [S_h; P_h] of the product's A
// operand: S_h (rows 0-63) starts at zero and takes B_c, P_h (rows 64-127) starts at the identity
// rows r0 .. r0 + 63, so that one product per chunk carries both the segment's offset
// B_seg = (... (B_cb A_cb+1 + B_cb+1) ...) and the rows of its transition A_seg = A_cb ... A_ce-1;
// S_out = S_in A_seg + B_seg.  Shared memory: the two K blocks of [S_h; P_h] (128 rows each, fp16,
// 128B-swizzled), then a ring of A_c and this half's rows of B_c.
constexpr uint32_t CP_STAGE = 4 * PANEL + 2 * PANEL;  // A_c | B_c rows of this half
constexpr uint32_t CP_OFF_ST = 4 * PANEL;
constexpr uint32_t CP_SMEM = CP_OFF_ST + SC_STAGES * CP_STAGE + 1024;
static_assert(CP_SMEM <= 232448, "shared memory budget");

__global__ void __launch_bounds__(ST, 1)
    compose_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b, ScanParams p)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    __shared__ uint32_t tmem_base_s;
    __shared__ __align__(8) uint64_t mbar[SC_STAGES + 2];  // ring stages; products; drain
    __shared__ int abort_s;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int quad = warp & 3, half = warp >> 2;  // TMEM lane quarter; column half (= K block)
    const int row = quad * 32 + lane;             // 0-63: a row of S_h, 64-127: a row of P_h
    const int vh = blockIdx.x & 1, seg = (int)(blockIdx.x >> 1) % p.G, bh = (int)(blockIdx.x >> 1) / p.G;
    const int r0 = 64 * vh;
    const int cb = (int)((long long)seg * p.NC / p.G), ce = (int)((long long)(seg + 1) * p.NC / p.G), nk = ce - cb;
    const uint32_t sbase = smem_u32(sm);
    const uint64_t dbase = sdesc(sbase, 0, 0);
    const uint32_t mb_mma = smem_u32(&mbar[SC_STAGES]);
    if (tid == 0) {
        abort_s = 0;
        for (int i = 0; i < SC_STAGES + 2; ++i) mbar_init(smem_u32(&mbar[i]), 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        prefetch_tmap(&tm_a);
        prefetch_tmap(&tm_b);
    }
    if (warp == 0) tmem_alloc(smem_u32(&tmem_base_s), 128);
    {  // S_h = 0, P_h = the identity rows of this half: row `row`, the 64 columns of K block `half`
        uint8_t *sp = sm + (uint32_t)half * 2 * PANEL;
#pragma unroll
        for (int g = 0; g < 2; ++g) {
            float w[32];
#pragma unroll
            for (int q = 0; q < 32; ++q) w[q] = (row >= 64 && 64 * half + 32 * g + q == r0 + row - 64) ? 1.f : 0.f;
            st_row_h(sp, row, 32 * g, w);
        }
    }
    fence_async_smem();
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tmem = tmem_base_s;
    const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
    grid_dependency_wait();  // the maps of the map kernel
    allow_dependent_launch();
    const size_t ch0 = (size_t)bh * p.NC;
    auto issue = [&](int k) {  // chunk cb + k's A_c and this half of B_c into stage k % SC_STAGES
        const int st = k % SC_STAGES;
        const uint32_t base = sbase + CP_OFF_ST + st * CP_STAGE, mb = smem_u32(&mbar[st]);
        const int ra = (int)((ch0 + cb + k) * 128);
        mbar_expect_tx(mb, CP_STAGE);
        tma_load_2d(base, &tm_a, mb, 0, ra);
        tma_load_2d(base + 2 * PANEL, &tm_a, mb, 64, ra);
        tma_load_2d(base + 4 * PANEL, &tm_b, mb, 0, ra + r0);
        tma_load_2d(base + 5 * PANEL, &tm_b, mb, 64, ra + r0);
    };
    uint32_t ph_mma = 0;
    int issued = 0, consumed = 0;
    if (tid == 0)
        for (; issued < SC_STAGES && issued < nk; ++issued) issue(issued);
    for (int k = 0; k < nk && abort_s == 0; ++k) {
        const int st = k % SC_STAGES;
        const uint32_t sb = CP_OFF_ST + st * CP_STAGE;
        if (tid == 0) {
            if (mbar_wait(smem_u32(&mbar[st]), (uint32_t)((k / SC_STAGES) & 1), p.wait_ns)) {
                ++consumed;
                fence_after_sync();
                // D1 = [S_h; P_h] A_c (A = [S_h; P_h] [r][m] K-major, 128 rows a K block; B = A_c MN-major)
                const uint32_t id1 = idesc_f16(128, 128, 0, 1);
#pragma unroll
                for (int s2 = 0; s2 < 8; ++s2) {
                    const uint32_t so = (uint32_t)(s2 >> 2) * 2 * PANEL + (uint32_t)(s2 & 3) * 32;
                    mma_f16(tmem, dsc(dbase, so, 16, 1024), dsc(dbase, sb + s2 * 2048, 2 * PANEL, 1024), id1, s2 > 0);
                }
                mma_commit(mb_mma);
            } else {
                abort_s = 1;
                set_status(p.status, kDevTimeout);
            }
        }
        __syncthreads();
        if (abort_s) break;
        uint4 bc[8];  // B_c of this thread's S row (rows < 64), read before the stage is refilled
        if (row < 64) {
            const uint8_t *bp = sm + sb + 4 * PANEL + (uint32_t)half * PANEL;
#pragma unroll
            for (int e = 0; e < 8; ++e) bc[e] = *reinterpret_cast<const uint4 *>(bp + sw128(row, 8 * e));
        }
        if (!mbar_wait(mb_mma, ph_mma, p.wait_ns)) {
            abort_s = 1;
            set_status(p.status, kDevTimeout);
        }
        ph_mma ^= 1u;
        fence_before_sync();
        __syncthreads();  // stage st and the operand rows are consumed
        fence_after_sync();
        if (tid == 0 && issued < nk && abort_s == 0) issue(issued++);
        uint8_t *sp = sm + (uint32_t)half * 2 * PANEL;
        const bool last = k + 1 == nk;
#pragma unroll
        for (int g = 0; g < 2; ++g) {
            float v[32];
            tmem_ld(tmem + lane_off + (uint32_t)(64 * half + 32 * g), v);
            if (row < 64) {
#pragma unroll
                for (int e = 0; e < 4; ++e) add_h8(v, 8 * e, bc[4 * g + e]);
            }
            if (last) {  // the segment's map: B_seg row r0 + row (row < 64), A_seg row r0 + row - 64
                float *dst = p.seg_maps + ((((size_t)bh * p.G + seg) * 2 + (row >= 64)) * D + r0 + (row & 63)) * D +
                             64 * half + 32 * g;
#pragma unroll
                for (int q = 0; q < 8; ++q)
                    reinterpret_cast<float4 *>(dst)[q] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
            } else {
                st_row_h(sp, row, 32 * g, v);
            }
        }
        fence_async_smem();  // [S_h; P_h] is the next chunk's MMA operand
        fence_before_sync();
        __syncthreads();
        fence_after_sync();
    }
    if (tid == 0 && abort_s) {  // drain after an expired wait
        for (int k = consumed; k < issued; ++k)
            (void)mbar_wait(smem_u32(&mbar[k % SC_STAGES]), (uint32_t)((k / SC_STAGES) & 1), 1000000000ull);
        const uint32_t mb_drain = smem_u32(&mbar[SC_STAGES + 1]);
        mma_commit(mb_drain);
        (void)mbar_wait(mb_drain, 0, 1000000000ull);
    }
    fence_before_sync();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, 128);
}

// The segments' start states: S_0 = S_init (or 0), S_{g+1} = S_g A_seg(g) + B_seg(g), fp32.  Block
// (bh, rb) takes 8 state rows; warp w row 8 rb + w, lane the columns 4 lane .. 4 lane + 3.
__global__ void __launch_bounds__(256) carry_kernel(ScanParams p)
{
    __shared__ float s[8][D];
    const int bh = blockIdx.x, rb = blockIdx.y, w = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int r = 8 * rb + w, c4 = 4 * lane;
    grid_dependency_wait();  // the segment maps of the compose pass
    allow_dependent_launch();
    float4 cur = p.S_init ? *reinterpret_cast<const float4 *>(p.S_init + ((size_t)bh * D + r) * D + c4)
                          : make_float4(0.f, 0.f, 0.f, 0.f);
    for (int g = 0; g < p.G; ++g) {
        *reinterpret_cast<float4 *>(p.S_seg + (((size_t)bh * p.G + g) * D + r) * D + c4) = cur;
        if (g + 1 == p.G) break;
        *reinterpret_cast<float4 *>(&s[w][c4]) = cur;
        __syncwarp();
        const float *Bm = p.seg_maps + (((size_t)bh * p.G + g) * 2 + 0) * D * D;
        const float *Am = p.seg_maps + (((size_t)bh * p.G + g) * 2 + 1) * D * D;
        float4 acc = *reinterpret_cast<const float4 *>(Bm + (size_t)r * D + c4);
#pragma unroll 8
        for (int m = 0; m < D; ++m) {
            const float sm_ = s[w][m];
            const float4 a = *reinterpret_cast<const float4 *>(Am + (size_t)m * D + c4);
            acc.x = fmaf(sm_, a.x, acc.x);
            acc.y = fmaf(sm_, a.y, acc.y);
            acc.z = fmaf(sm_, a.z, acc.z);
            acc.w = fmaf(sm_, a.w, acc.w);
        }
        __syncwarp();
        cur = acc;
    }
}

}  // namespace mp

// ---------------------------------------------------------------------------------------------
namespace {

PFN_cuTensorMapEncodeTiled_v12000 map_encoder()
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

bool encode_map(CUtensorMap *m, CUtensorMapDataType dt, const void *base, int rank, const cuuint64_t *dims,
                const cuuint64_t *strides_bytes, const cuuint32_t *box, CUtensorMapSwizzle sw)
{
    auto fn = map_encoder();
    if (!fn) return false;
    cuuint32_t es[5] = {1, 1, 1, 1, 1};
    return fn(m, dt, (cuuint32_t)rank, const_cast<void *>(base), dims, strides_bytes, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool map_supported(const Shape &s, prism_dtype io)
{
    return io == PRISM_BF16 && s.dk == mp::D && s.dv == mp::D && s.L >= 1 && s.L <= 1 + mp::RM;
}

// Segments of the chunk scan: long sequences (256 chunks or more) of few heads run the scan as G
// segments (compose, carry, then the scan of each segment from its start state) so that the
// scan's blocks fill more of the SMs; G <= kMaxScanSegments.  The segment maps and start states
// follow the other map buffers in the workspace.
constexpr int kMaxScanSegments = 8;
bool scan_segments_eligible(const Shape &s) { return s.NC >= 256 && 4 * s.BH <= 152; }
int scan_segments(const Shape &s, int sm_count)
{
    if (!scan_segments_eligible(s)) return 1;
    int g = sm_count / (2 * s.BH);
    g = g < kMaxScanSegments ? g : kMaxScanSegments;
    g = g < s.NC / 64 ? g : s.NC / 64;
    return g > 1 ? g : 1;
}
size_t scan_segment_bytes(const Shape &s)
{
    return scan_segments_eligible(s) ? (size_t)s.BH * kMaxScanSegments * 3 * mp::D * mp::D * 4 + 256 : 0;
}

size_t map_workspace_bytes(const Shape &s)
{
    const size_t chunks = (size_t)s.BH * s.NC;
    return chunks * (2 * 128 + 2 * 64) * mp::D * 2 + 4 * 256 + scan_segment_bytes(s);
}

void map_carve(const Shape &s, void *base, MapWorkspace *w)
{
    const size_t chunks = (size_t)s.BH * s.NC;
    uintptr_t p = ((uintptr_t)base + 255) & ~(uintptr_t)255;
    w->A = (__half *)p;
    p += chunks * 128 * mp::D * 2;
    w->Q = (__half *)p;
    p += chunks * 64 * mp::D * 2;
    w->B = (__half *)p;
    p += chunks * 128 * mp::D * 2;
    w->O = (__half *)p;
}

cudaError_t map_prepare()
{
    cudaError_t e = cudaFuncSetAttribute(mp::map_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)mp::MAP_SMEM);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(mp::compose_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)mp::CP_SMEM);
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(mp::scan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)mp::SCAN_SMEM);
}

cudaError_t map_forward(const Shape &s, const ForwardArgs &a, bool out_f32, const MapWorkspace &w, int sm_count,
                        int *d_status, long long wait_ns, KernelTimer &tm)
{
    using namespace mp;
    const cuuint64_t BH = s.BH, T = s.T;
    CUtensorMap mq, mk, mv, mu, ma, mqt, mb, mo, mbh;
    const CUtensorMapDataType BF = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, F16 = CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    {
        cuuint64_t dims[3] = {(cuuint64_t)D, T, BH};
        cuuint64_t str[2] = {(cuuint64_t)D * 2, T * D * 2};
        cuuint32_t box[3] = {64, 64, 1};
        if (!encode_map(&mq, BF, a.q, 3, dims, str, box, CU_TENSOR_MAP_SWIZZLE_128B)) return cudaErrorInvalidValue;
        if (!encode_map(&mk, BF, a.k, 3, dims, str, box, CU_TENSOR_MAP_SWIZZLE_128B)) return cudaErrorInvalidValue;
        cuuint32_t vbox[3] = {(cuuint32_t)D, 72, 1};
        if (!encode_map(&mv, BF, a.v, 3, dims, str, vbox, CU_TENSOR_MAP_SWIZZLE_NONE)) return cudaErrorInvalidValue;
    }
    if (s.R > 0) {
        cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)s.R, T, BH};
        cuuint64_t str[3] = {(cuuint64_t)D * 2, (cuuint64_t)s.R * D * 2, T * s.R * D * 2};
        cuuint32_t box[4] = {64, 1, 64, 1};
        if (!encode_map(&mu, BF, a.u, 4, dims, str, box, CU_TENSOR_MAP_SWIZZLE_128B)) return cudaErrorInvalidValue;
    } else {
        mu = mk;  // never read with L = 1
    }
    const cuuint64_t chunks = (cuuint64_t)s.BH * s.NC;
    {
        cuuint64_t str[1] = {(cuuint64_t)D * 2};
        cuuint64_t d128[2] = {(cuuint64_t)D, chunks * 128}, d64[2] = {(cuuint64_t)D, chunks * 64};
        cuuint32_t b128[2] = {64, 128}, b64[2] = {64, 64};
        if (!encode_map(&ma, F16, w.A, 2, d128, str, b128, CU_TENSOR_MAP_SWIZZLE_128B)) return cudaErrorInvalidValue;
        if (!encode_map(&mqt, F16, w.Q, 2, d64, str, b64, CU_TENSOR_MAP_SWIZZLE_128B)) return cudaErrorInvalidValue;
        if (!encode_map(&mb, F16, w.B, 2, d128, str, b128, CU_TENSOR_MAP_SWIZZLE_128B)) return cudaErrorInvalidValue;
        if (!encode_map(&mbh, F16, w.B, 2, d128, str, b64, CU_TENSOR_MAP_SWIZZLE_128B)) return cudaErrorInvalidValue;
        if (!encode_map(&mo, F16, w.O, 2, d64, str, b64, CU_TENSOR_MAP_SWIZZLE_128B)) return cudaErrorInvalidValue;
    }
    const unsigned long long wns = wait_ns > 0 ? (unsigned long long)wait_ns : 100000000ull;
    MapParams mp_;
    mp_.beta = a.beta;
    mp_.alpha = a.alpha;
    mp_.gamma = a.gamma;
    mp_.eta = a.eta;
    mp_.conv_w = (const __nv_bfloat16 *)a.conv_w;
    mp_.v_hist = (const __nv_bfloat16 *)a.v_hist;
    mp_.p_gain = (const __nv_bfloat16 *)a.p_gain;
    mp_.mA = w.A;
    mp_.mQ = w.Q;
    mp_.mB = w.B;
    mp_.mO = w.O;
    mp_.status = d_status;
    mp_.H = s.H;
    mp_.T = s.T;
    mp_.R = s.R;
    mp_.NC = s.NC;
    mp_.nchunks = (int)chunks;
    mp_.wait_ns = wns;
    CUtensorMap mout;
    if (out_f32) {
        mout = ma;  // not read: an fp32 output is written directly
    } else {
        cuuint64_t dims[3] = {(cuuint64_t)D, T, BH};
        cuuint64_t str[2] = {(cuuint64_t)D * 2, T * D * 2};
        cuuint32_t box[3] = {64, 64, 1};
        if (!encode_map(&mout, BF, a.out, 3, dims, str, box, CU_TENSOR_MAP_SWIZZLE_128B)) return cudaErrorInvalidValue;
    }
    ScanParams sp;
    sp.mO = w.O;
    sp.S_init = a.S_init;
    sp.S_final = a.S_final;
    sp.out = a.out;
    sp.status = d_status;
    sp.T = s.T;
    sp.NC = s.NC;
    sp.out_f32 = out_f32 ? 1 : 0;
    sp.wait_ns = wns;
    const int G = scan_segments(s, sm_count);
    sp.G = G;
    sp.S_seg = nullptr;
    sp.seg_maps = nullptr;
    if (G > 1) {  // after the O_loc maps (map_workspace_bytes counted the room)
        const size_t chunks = (size_t)s.BH * s.NC;
        const uintptr_t q = ((uintptr_t)(w.O + chunks * 64 * D) + 255) & ~(uintptr_t)255;
        sp.seg_maps = reinterpret_cast<float *>(q);
        sp.S_seg = sp.seg_maps + (size_t)s.BH * G * 2 * D * D;
    }

    cudaLaunchAttribute pdl[1];
    pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    pdl[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.stream = tm.stream;
    cfg.attrs = pdl;
    cfg.numAttrs = 1;
    tm.begin("map_chunks");
    cfg.gridDim = dim3((unsigned)((int)chunks < sm_count ? (int)chunks : sm_count));
    cfg.blockDim = dim3(NT);
    cfg.dynamicSmemBytes = MAP_SMEM;
    cudaError_t e = cudaLaunchKernelEx(&cfg, map_kernel, mq, mk, mv, mu, ma, mqt, mb, mo, mp_);
    tm.end();
    if (e != cudaSuccess) return e;
    if (G > 1) {
        tm.begin("map_compose");
        cfg.gridDim = dim3((unsigned)(2 * s.BH * G));
        cfg.blockDim = dim3(ST);
        cfg.dynamicSmemBytes = CP_SMEM;
        e = cudaLaunchKernelEx(&cfg, compose_kernel, ma, mbh, sp);
        tm.end();
        if (e != cudaSuccess) return e;
        tm.begin("map_carry");
        cfg.gridDim = dim3((unsigned)s.BH, (unsigned)(D / 8));
        cfg.blockDim = dim3(256);
        cfg.dynamicSmemBytes = 0;
        e = cudaLaunchKernelEx(&cfg, carry_kernel, sp);
        tm.end();
        if (e != cudaSuccess) return e;
    }
    tm.begin("map_scan");
    cfg.gridDim = dim3((unsigned)(2 * s.BH * G));
    cfg.blockDim = dim3(ST);
    cfg.dynamicSmemBytes = SCAN_SMEM;
    e = cudaLaunchKernelEx(&cfg, scan_kernel, ma, mqt, mbh, mout, sp);
    tm.end();
    if (e != cudaSuccess) return e;
    if (a.v_hist_out) {  // a plain launch: it runs after the kernels above have read v_hist
        e = launch_history(s, PRISM_BF16, a.v_hist, a.v, a.v_hist_out, tm);
        if (e != cudaSuccess) return e;
    }
    return cudaGetLastError();
}

}  // namespace prism

#ifdef PRISM_PHASE_TIMERS
// developer tracing build only: copy out (and optionally clear) the per-phase cycle totals
extern "C" __attribute__((visibility("default"))) int prism_debug_map_phase_cycles(unsigned long long *out, int reset)
{
    if (cudaMemcpyFromSymbol(out, prism_map_phase_cycles, sizeof(unsigned long long) * 16) != cudaSuccess) return -1;
    if (reset) {
        unsigned long long z[16] = {0};
        if (cudaMemcpyToSymbol(prism_map_phase_cycles, z, sizeof(z)) != cudaSuccess) return -1;
    }
    return 0;
}
#endif
