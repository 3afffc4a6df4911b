// Device helpers shared by the tensor-core kernels of the chunk-map path: fp16 packing into
// 128B-swizzled tiles, shared-memory descriptors relative to a 1024-aligned base, the exact-erf
// GELU gain, warp-level fp16 MMA fragments and the UT solve of one 64-token chunk.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "tc_ptx.h"

namespace prism {
namespace tcu {

using tc::sw128;

__device__ __forceinline__ void set_status(int *st, int code) { atomicCAS(st, 0, code); }

// compile-time flag for code paths chosen by a uniform runtime branch
template <bool B>
struct Flag {
    static constexpr bool value = B;
};

__device__ __forceinline__ uint32_t pack_h2(float a, float b)
{
    const __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<const uint32_t *>(&h);
}

// write N consecutive fp32 values (columns col0..col0+N-1 of row `row`, col0 a multiple of 8)
// as fp16 into a [rows][64] SW128 panel
template <int N>
__device__ __forceinline__ void st_row_h(uint8_t *panel, int row, int col0, const float (&v)[N])
{
#pragma unroll
    for (int g = 0; g < N / 8; ++g) {
        uint4 w;
        w.x = pack_h2(v[8 * g + 0], v[8 * g + 1]);
        w.y = pack_h2(v[8 * g + 2], v[8 * g + 3]);
        w.z = pack_h2(v[8 * g + 4], v[8 * g + 5]);
        w.w = pack_h2(v[8 * g + 6], v[8 * g + 7]);
        *reinterpret_cast<uint4 *>(panel + sw128(row, col0 + 8 * g)) = w;
    }
}

// Descriptor of the operand at byte offset `off` of the CTA's 1024-aligned shared-memory base
// (a descriptor of the base plus the offset fields; every field stays in range).
__device__ __forceinline__ uint64_t dsc(uint64_t base, uint32_t off, uint32_t lbo, uint32_t sbo)
{
    return base + (uint64_t)(off >> 4) + ((uint64_t)(lbo >> 4) << 16) + ((uint64_t)(sbo >> 4) << 32);
}

// The normal cdf Phi(a) and density phi(a) = e^{-a^2/2} / sqrt(2 pi).  Phi uses the rational
// approximation of erf from Abramowitz & Stegun, Handbook of Mathematical Functions, formula
// 7.1.26 (|error| <= 1.5e-7), which shares the Gaussian factor e^{-a^2/2} with phi.
__device__ __forceinline__ void gauss_parts(float a, float &Phi, float &phi)
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
    phi = 0.39894228040143268f * E;
}

// Gain g = GELU'(a) = Phi(a) + a phi(a) and Phi(a), for the exact-erf GELU.
__device__ __forceinline__ void gelu_gain(float a, float &g, float &Phi)
{
    float phi;
    gauss_parts(a, Phi, phi);
    g = fmaf(a, phi, Phi);
}

// GELU(z) = z Phi(z) (exact-erf form).
__device__ __forceinline__ float gelu_value(float z)
{
    float Phi, phi;
    gauss_parts(z, Phi, phi);
    return z * Phi;
}

// barrier over `n` threads (whole warps) of the CTA; ids 1.. (0 is __syncthreads')
__device__ __forceinline__ void named_bar(int id, int n) { asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory"); }

// ---- warp-level fp16 MMA (the 64x64 triangular solve's block products) ----------------------
// m16n8k16 fragments of fp32 matrices in shared memory (row-major, row stride ld; A: 16 rows from
// r0, 16 columns from k0; B: 16 rows (k) from k0, 8 columns (n) from n0), rounded to fp16 (T
// enters the tensor-core products as fp16 anyway, and fp16 keeps tf32's 10 mantissa bits); the
// C fragment: rows gq and gq + 8, columns 2 tq, 2 tq + 1 of a 16 x 8 tile.
struct Frag {
    int gq, tq;  // lane / 4, lane % 4
};
__device__ __forceinline__ void frag_a(const Frag &f, const float *M, int ld, int r0, int k0, uint32_t (&a)[4])
{
    const float *p = M + (r0 + f.gq) * ld + k0 + 2 * f.tq;
    a[0] = pack_h2(p[0], p[1]);
    a[1] = pack_h2(p[8 * ld], p[8 * ld + 1]);
    a[2] = pack_h2(p[8], p[9]);
    a[3] = pack_h2(p[8 * ld + 8], p[8 * ld + 9]);
}
__device__ __forceinline__ void frag_b(const Frag &f, const float *M, int ld, int k0, int n0, uint32_t &b0, uint32_t &b1)
{
    const float *p = M + (k0 + 2 * f.tq) * ld + n0 + f.gq;
    b0 = pack_h2(p[0], p[ld]);
    b1 = pack_h2(p[8 * ld], p[9 * ld]);
}
// D += A B for one m16n8k16 tile (fp16 in, fp32 accumulate)
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

constexpr int LDA = 68;             // row stride (floats) of A and T32 (float4 rows, conflict-free fragments)
constexpr int SOLVE_THREADS = 256;  // 8 warps
constexpr int SOLVE_SCRATCH = 4 * 256;

// T = (I + A)^{-1} for a strictly lower-triangular 64x64 A (fp32, row stride LDA), by 16x16
// blocks: the diagonal blocks by forward substitution, then the blocks below them,
// T[bi][bj] = -T[bi][bi] sum_k A[bi][k] T[k][bj], in two merge levels (16 -> 32 -> 64) on warp
// fp16 MMAs (m16n8k16, fp32 accumulation).  Writes T (fp32, T32) and its fp16 copy into the [64][64] SW128 panel `tf` ([i][j],
// zero above the diagonal).  Run by SOLVE_THREADS threads (whole warps, st = 0..255) that sync on
// named barrier `bar`; `x` is SOLVE_SCRATCH floats of scratch.  Blocks (0,1) and (2,3) of T32 stay
// unwritten and are never read.
__device__ __forceinline__ void ut_solve(const float *A, float *T32, float *x, uint8_t *tf, int st, int bar)
{
    const int sw = st >> 5, lane = st & 31;
    const Frag fr{lane >> 2, lane & 3};
    if (st < 64) {  // diagonal 16x16 blocks, one column per thread
        const int o = 16 * (st >> 4), cc = st & 15;
        float t[16];
        // the block's row r of A as four 16-byte loads, the next row's in flight while a row is
        // summed; T's column is stored after the whole column (a store between the rows would keep
        // every later row's loads of A, which it may alias, behind it)
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
    named_bar(bar, SOLVE_THREADS);
    if (sw < 4) {
        // 16 -> 32: T[1][0] = -T[1][1] A[1][0] T[0][0], T[3][2] likewise; warp sw owns one 8-column
        // tile of one block
        const int pb = sw >> 1, nt = sw & 1;
        const int ri = 16 + 32 * pb, cj = 32 * pb;
        float xa[4] = {0.f, 0.f, 0.f, 0.f};
        {
            uint32_t a[4], b0, b1;
            frag_a(fr, A, LDA, ri, cj, a);
            frag_b(fr, T32, LDA, cj, cj + 8 * nt, b0, b1);
            mma_h16(xa, a, b0, b1);
        }
        float *X = x + sw * 128;  // 16 x 8
        X[fr.gq * 8 + 2 * fr.tq] = xa[0];
        X[fr.gq * 8 + 2 * fr.tq + 1] = xa[1];
        X[(fr.gq + 8) * 8 + 2 * fr.tq] = xa[2];
        X[(fr.gq + 8) * 8 + 2 * fr.tq + 1] = xa[3];
        __syncwarp();
        float y[4] = {0.f, 0.f, 0.f, 0.f};
        {
            uint32_t a[4], b0, b1;
            frag_a(fr, T32, LDA, ri, ri, a);
            frag_b(fr, X, 8, 0, 0, b0, b1);
            mma_h16(y, a, b0, b1);
        }
        frag_c_store(fr, T32, LDA, ri, cj + 8 * nt, y, -1.f);
    }
    named_bar(bar, SOLVE_THREADS);
    {
        // 32 -> 64: T[32:64][0:32] = -T[32:64][32:64] A[32:64][0:32] T[0:32][0:32]; warp sw owns the
        // 16-row half mt = sw / 4 of the 8-column tile nt = sw % 4 (n0 = 8 nt): its rows of
        // X = A_lo T_lo, then (once all of X is in) its rows of -T_hi X
        const int nt = sw & 3, mt = sw >> 2, n0 = 8 * nt;
        float xa[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int ks = 0; ks < 2; ++ks) {
            if (n0 >= 16 && ks == 0) continue;  // T_lo[k][n] = 0 for k < 16 <= n
            uint32_t a[4], b0, b1;
            frag_b(fr, T32, LDA, 16 * ks, n0, b0, b1);
            frag_a(fr, A, LDA, 32 + 16 * mt, 16 * ks, a);
            mma_h16(xa, a, b0, b1);
        }
        float *X = x + nt * 256;  // 32 x 8
        X[(16 * mt + fr.gq) * 8 + 2 * fr.tq] = xa[0];
        X[(16 * mt + fr.gq) * 8 + 2 * fr.tq + 1] = xa[1];
        X[(16 * mt + fr.gq + 8) * 8 + 2 * fr.tq] = xa[2];
        X[(16 * mt + fr.gq + 8) * 8 + 2 * fr.tq + 1] = xa[3];
        named_bar(bar, SOLVE_THREADS);  // both halves of every X tile are in
        float y[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int ks = 0; ks < 2; ++ks) {
            if (mt == 0 && ks == 1) continue;  // T_hi[0:16][16:32] = 0
            uint32_t a[4], b0, b1;
            frag_b(fr, X, 8, 16 * ks, 0, b0, b1);
            frag_a(fr, T32, LDA, 32 + 16 * mt, 32 + 16 * ks, a);
            mma_h16(y, a, b0, b1);
        }
        frag_c_store(fr, T32, LDA, 32 + 16 * mt, n0, y, -1.f);
    }
    named_bar(bar, SOLVE_THREADS);
    for (int e = st; e < 64 * 8; e += SOLVE_THREADS) {  // fp16 copy, zero above the diagonal
        const int i = e >> 3, g = e & 7;
        const float4 lo = *reinterpret_cast<const float4 *>(T32 + i * LDA + 8 * g);
        const float4 hi = *reinterpret_cast<const float4 *>(T32 + i * LDA + 8 * g + 4);
        const float v[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
        float m[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) m[q] = (8 * g + q <= i) ? v[q] : 0.f;
        uint4 w;
        w.x = pack_h2(m[0], m[1]);
        w.y = pack_h2(m[2], m[3]);
        w.z = pack_h2(m[4], m[5]);
        w.w = pack_h2(m[6], m[7]);
        *reinterpret_cast<uint4 *>(tf + sw128(i, 8 * g)) = w;
    }
}

}  // namespace tcu
}  // namespace prism
