// kda_chunk.cuh -- warp-level pieces of the intra-chunk algebra shared by the
// KDA kernels: the decay-scaled chunk products A = Kl Kr^T and P = Ql Kr^T
// from bf16 hi/lo operand pairs, and the unit-lower inverse (I + A)^-1 from
// the nilpotent product form (I - A)(I + A^2)(I + A^4)(I + A^8), all on
// m16n8k16 warp MMA with register-resident fragments.
//
// "How FlashKDA's CHUNK Size of 16 Improves Numerical Stability Over CHUNK
// 64" -- "Efficient 16x16 Matrix Inversion": 16-token chunks, the unit-lower
// chunk matrix is inverted by a Neumann series (exact here: A^16 = 0).
#pragma once
#include "kda_common.cuh"

namespace kda {

// 8x8 16-bit matrix transpose within a warp (standard fragment layout).
__device__ __forceinline__ uint32_t movm_t(uint32_t a)
{
    uint32_t d;
    asm("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(d) : "r"(a));
    return d;
}

// Accumulator fragments of a 16x16 fp32 matrix as two m16n8 tiles: c[nt][i] holds
// (row g + 8 (i >> 1), col 8 nt + 2 t + (i & 1)), g = lane / 4, t = lane % 4.
struct Frag16 {
    float c[2][4];
};

__device__ __forceinline__ void frag_zero(Frag16 &f)
{
#pragma unroll
    for (int i = 0; i < 2; ++i) f.c[i][0] = f.c[i][1] = f.c[i][2] = f.c[i][3] = 0.f;
}

// A-operand (m16 x k16, f16) of an accumulator matrix.
__device__ __forceinline__ void frag_as_a(const Frag16 &f, uint32_t (&a)[4])
{
    a[0] = pack_f16(f.c[0][0], f.c[0][1]);
    a[1] = pack_f16(f.c[0][2], f.c[0][3]);
    a[2] = pack_f16(f.c[1][0], f.c[1][1]);
    a[3] = pack_f16(f.c[1][2], f.c[1][3]);
}

// B-operand (k16 x n8 tiles, f16) of an accumulator matrix X, i.e. B[k][n] = X[k][n]:
// b[nt][kb] is the transpose of the 8x8 block (rows 8 kb.., cols 8 nt..).
__device__ __forceinline__ void frag_as_b(const Frag16 &f, uint32_t (&b)[2][2])
{
    b[0][0] = movm_t(pack_f16(f.c[0][0], f.c[0][1]));
    b[0][1] = movm_t(pack_f16(f.c[0][2], f.c[0][3]));
    b[1][0] = movm_t(pack_f16(f.c[1][0], f.c[1][1]));
    b[1][1] = movm_t(pack_f16(f.c[1][2], f.c[1][3]));
}

// x + s I (in place), for accumulator fragments
__device__ __forceinline__ void frag_add_diag(Frag16 &f, float s, int g, int t)
{
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int i = 0; i < 4; ++i)
            if (nt == (i >> 1) && g == 2 * t + (i & 1)) f.c[nt][i] += s;
}

// c = a * b for 16x16x16 (fp32 accumulate into zeroed c)
__device__ __forceinline__ void frag_mul(Frag16 &c, const uint32_t (&a)[4], const uint32_t (&b)[2][2])
{
    frag_zero(c);
    mma_f16(c.c[0], a, b[0][0], b[0][1]);
    mma_f16(c.c[1], a, b[1][0], b[1][1]);
}

// T = (I + A)^-1 for strictly lower A (fp32 fragments in, fp32 fragments out),
// as (I - A)(I + A^2)(I + A^4)(I + A^8) with f16 operands.
__device__ __forceinline__ void unit_lower_inverse(const Frag16 &A, Frag16 &T, int g, int t)
{
    uint32_t a[4], b[2][2], ax[4], bx[2][2];
    Frag16 p2, p4, p8, m, x;
    frag_as_a(A, a);
    frag_as_b(A, b);
    frag_mul(p2, a, b);            // A^2
    Frag16 ia = A;                 // I - A
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int i = 0; i < 4; ++i) ia.c[nt][i] = -ia.c[nt][i];
    frag_add_diag(ia, 1.f, g, t);
    frag_as_a(p2, a);
    frag_as_b(p2, b);
    frag_mul(p4, a, b);            // A^4
    frag_add_diag(p2, 1.f, g, t);
    frag_as_a(ia, ax);
    frag_as_b(p2, bx);
    frag_mul(m, ax, bx);           // (I - A)(I + A^2), independent of A^4
    frag_as_a(p4, a);
    frag_as_b(p4, b);
    frag_mul(p8, a, b);            // A^8
    frag_add_diag(p4, 1.f, g, t);
    frag_as_a(m, ax);
    frag_as_b(p4, bx);
    frag_mul(x, ax, bx);           // ... (I + A^4), independent of A^8
    frag_add_diag(p8, 1.f, g, t);
    frag_as_a(x, a);
    frag_as_b(p8, b);
    frag_mul(T, a, b);             // ... (I + A^8)
}

// Split two floats into bf16 hi and lo parts (x ~= hi + lo to ~16 mantissa bits).
__device__ __forceinline__ void split_bf16(float x0, float x1, uint32_t &hi, uint32_t &lo)
{
    hi = pack_bf16(x0, x1);
    lo = pack_bf16(x0 - bf16_lo(hi), x1 - bf16_hi(hi));
}

// Split two floats into a truncated bf16 hi part and a rounded bf16 lo part
// (x ~= hi + lo to ~16 mantissa bits); hi is a byte permute, x - hi is exact.
__device__ __forceinline__ void split_bf16_trunc(float x0, float x1, uint32_t &hi, uint32_t &lo)
{
    const uint32_t b0 = __float_as_uint(x0), b1 = __float_as_uint(x1);
    hi = __byte_perm(b0, b1, 0x7632);
    lo = pack_bf16(x0 - __uint_as_float(b0 & 0xffff0000u), x1 - __uint_as_float(b1 & 0xffff0000u));
}

// acc[nt] (16 rows r x 16 cols j) = sum_c X[r][c] R[j][c] over the channels c in
// [16 kbase, 16 (kbase + NK)), from 16-bit tiles stored row-major [16][136] (272-byte rows):
// X rounded to bf16 once and R as bf16 hi + lo, two bf16 products X Rh + X Rl per entry
// (R keeps ~16-bit precision, X 8 bits; the bf16 exponent range holds 2^{+-58}).
template <int NK>
__device__ __forceinline__ void chunk_gram_x2(uint32_t x, uint32_t rh, uint32_t rl, Frag16 &acc, int lane, int kbase)
{
    const int mi = lane >> 3, ri = lane & 7;
    const uint32_t aoff = (ri + 8 * (mi & 1)) * 272 + 16 * (mi >> 1) + 32 * kbase;
    const uint32_t boff = (ri + 8 * (mi >> 1)) * 272 + 16 * (mi & 1) + 32 * kbase;
    Frag16 cross;
    frag_zero(acc);
    frag_zero(cross);
#pragma unroll
    for (int kk = 0; kk < NK; ++kk) {
        uint32_t a[4], bh[4], bl[4];
        ldsm_x4(x + aoff + 32 * kk, a[0], a[1], a[2], a[3]);
        ldsm_x4(rh + boff + 32 * kk, bh[0], bh[1], bh[2], bh[3]);
        ldsm_x4(rl + boff + 32 * kk, bl[0], bl[1], bl[2], bl[3]);
        mma_bf16(acc.c[0], a, bh[0], bh[1]);
        mma_bf16(acc.c[1], a, bh[2], bh[3]);
        mma_bf16(cross.c[0], a, bl[0], bl[1]);
        mma_bf16(cross.c[1], a, bl[2], bl[3]);
    }
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int i = 0; i < 4; ++i) acc.c[nt][i] += cross.c[nt][i];
}

}  // namespace kda
