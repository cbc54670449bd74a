// kda_fwd_tc.cuh -- KDA forward pass with the state products on the 5th-gen
// tensor core (tcgen05) and the fp32 state held in tensor memory. One CTA
// per (sequence, head) state, all 128 V rows.
//
// Chunk algebra. For chunk n (16 tokens) with state S_n (V x K) at its start,
//   Z_n = [K*Gamma ; Q*Gamma] (32 x K),  Phi_n = [[-T', 0], [-s M, s I]] (32 x 32),
//   TM_n = [T' ; s M] (32 x 16),  Kbar_n (16 x K),  gamma_n (K),  V_n,
// with T' = (I + A)^-1 diag(beta), M = P T', s = scale, so that one product
// gives both the rows written into the state and the outputs:
//   [E_n | O_n] = D_n = V_n^T TM_n^T + S_n (Phi_n Z_n)^T,
//   S_{n+1} = S_n Diag(gamma_n) + E_n Kbar_n.
// (W_n = Phi_n Z_n = [-w ; s q^] with w = T' (K*Gamma), q^ = Q*Gamma - M (K*Gamma).)
// The state product is formed two chunks ahead from the decayed state two
// chunks back and corrected by the two rank-16 updates in between (exact in
// real arithmetic):
//   S_n W_n^T = Sb_{n-2} W'_n^T + E_{n-2} (Kbar_{n-2} W'_n^T) + E_{n-1} (Kbar_{n-1} W_n^T),
//   Sb_{n-2} = f16(S_{n-2} Diag(gamma_{n-2})),  W'_n = W_n Diag(gamma_{n-1}).
// Every term is a 16-bit tcgen05 MMA into the one accumulator D_n, so the
// tensor core orders them (same accumulator and shape) and no MMA reads
// another MMA's result. Only the last term depends on the previous chunk, so
// each chunk's critical path is one 16-deep MMA plus one commit.
//
// Warp roles (448 + 64 NFIN threads):
//   warp 0      TMA producer (lane 0); allocates / frees tensor memory.
//   warp 1      MMA issuer: the whole warp runs the issue loop with warp-uniform
//               operands and one elected lane issues each MMA and commit.
//   warps 2-5   state warps, one V row per thread (tensor-memory lane):
//               read [E|O], hand E to the tensor core, decay the state
//               (S <- S Diag(gamma)) and keep its f16 copy, store outputs.
//   warps 6-13  two prep lanes of four warps, alternate chunks: gate, scaled
//               key / query tiles, chunk-product partial sums.
//   warps 14..  NFIN finishers per lane (with two, one per 16-row half of W):
//               T', M, TM, W = Phi Z (written over Z as W'), Kbar_{n-1} W^T
//               and Kbar_{n-2} W'^T; they hand the slot to the tensor core.
// Tensor memory (512 columns): state fp32 [0,128), D x3 [128,224),
// E x2 (f16 pairs) [224,240), f16 state copies x2 [256,384).
//
// Page references: base-2 gate with the LOG2E-folded scale and the tanh form
// of the sigmoid ("FlashKDA lower_bound Parameter ..." -- "Conversion to the
// Gate Scale Factor"; "Base-2 Exponent Optimization in FlashKDA ..." --
// "Re-basing the Gate Activation"), CHUNK = 16 and the unit-lower chunk
// inverse ("How FlashKDA's CHUNK Size of 16 ..." -- "Efficient 16x16 Matrix
// Inversion"), tensor contract ("FlashKDA Input Tensor Shapes and DTypes ...").
#pragma once
#include "kda_common.cuh"
#include "kda_chunk.cuh"
#include "tcgen05.cuh"

namespace kda {
namespace tcs {

constexpr int NR = 3;  // raw chunk ring
// prep slot ring: slot n is last read by the finisher of chunk n + 2 (Kbar_n); with five slots a
// prep lane refilling a slot waits on the other lane's finisher, never on its own
constexpr int NP = 5;
// finisher warps per prep lane (1 or 2)
constexpr int NFIN = 1;
constexpr int NTHREADS = 32 * (14 + 2 * NFIN);
constexpr int W_UNROLL = 1;  // unroll of the finisher's 16-channel loop (code size against overlap)

constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t T_S = 0;     // fp32 state, 128 columns
constexpr uint32_t T_D = 128;   // D[3], 32 columns each
constexpr uint32_t T_E = 224;   // E[2], 8 columns each (16 f16)
constexpr uint32_t T_SB = 256;  // f16 state copies [2], 64 columns each

// prep slot (bytes)
constexpr int L_Z = 0;         // f16 Z, then W' in place: K-major 128B swizzle, 2 K-blocks x [32 rows][128 B]
constexpr int L_V16 = 8192;    // f16 V, MN-major 128B swizzle: 2 boxes x [16 rows][128 B]
constexpr int L_KB = 12288;    // f16 Kbar [16 j][128 c], MN-major 128B swizzle (the raw-tile layout)
constexpr int L_TM = 16384;    // f16 TM [32 n][16 k]
constexpr int L_CC = 17408;    // f16 (Kbar_{n-1} W^T)^T [32 n][16 k]
constexpr int L_HP = 18432;    // f16 (Kbar_{n-2} W'^T)^T [32 n][16 k]
constexpr int L_GAM = 19456;   // fp32 gamma [128]
constexpr int SLOT = 20480;

// prep scratch (per lane); fp32 tiles are [16][132] (528-byte rows: ldmatrix rows fall in distinct banks)
constexpr int F_LD = 528;
constexpr int S_KL = 0;                  // fp32 K * 2^(G - G_mid)
constexpr int S_QL = S_KL + 16 * F_LD;   // fp32 Q * 2^(G - G_mid)
constexpr int S_KR = S_QL + 16 * F_LD;   // fp32 K * 2^(G_mid - G)
// handed to the lane's finisher warp, two buffers (alternate chunks of the lane)
constexpr int S_BETA = S_KR + 16 * F_LD; // fp32 [2][16] beta
constexpr int S_GP = S_BETA + 128;        // fp32 [2][4 warps][2 tiles][32 lanes][4]: A (warps 0, 2) and P (1, 3) partial
                                          // sums; before them the chunk's gate sums [4 row quarters][32 lanes][4]
constexpr int SCR = S_GP + 2 * 4096;

constexpr int OFF_RAW = 0;
constexpr int OFF_SLOT = OFF_RAW + NR * RAW_STAGE;
constexpr int OFF_SCR = OFF_SLOT + NP * SLOT;
constexpr int OFF_BAR = OFF_SCR + 2 * SCR;
// barrier indices
constexpr int B_RAW_FULL = 0, B_RAW_EMPTY = B_RAW_FULL + NR, B_PREP_FULL = B_RAW_EMPTY + NR,
              B_PREP_EMPTY = B_PREP_FULL + NP, B_P2 = B_PREP_EMPTY + NP, B_D = B_P2 + NP, B_E = B_D + 2, B_G = B_E + 2,
              B_S = B_G + 2, B_I = B_S + 2, B_F = B_I + 1, B_GRAM = B_F + 1, B_FDONE = B_GRAM + 4, B_ZREAD = B_FDONE + 4,
              NBARS = B_ZREAD + 4;
constexpr int OFF_TMEMPTR = OFF_BAR + NBARS * 8;
constexpr int OFF_FLAGS = OFF_TMEMPTR + 16;
constexpr int SMEM_USED = OFF_FLAGS + 16;
constexpr int SMEM_ALLOC = SMEM_USED + 1024;

static_assert(SLOT % 1024 == 0 && OFF_SLOT % 1024 == 0 && RAW_STAGE % 1024 == 0, "swizzled operands need 1024-byte alignment");
static_assert(S_BETA % 16 == 0 && S_GP % 16 == 0 && SCR % 16 == 0, "alignment");
static_assert(OFF_BAR % 8 == 0, "mbarrier alignment");
static_assert(SMEM_ALLOC <= 227 * 1024, "shared memory budget");

// byte offset of (row n, col k) in a K-major, non-swizzled f16 operand with
// 16 K elements per row: 8x8 core matrices, LBO = 128 (K), SBO = 256 (N)
__device__ __forceinline__ uint32_t cm16(int n, int k)
{
    return (n >> 3) * 256 + (k >> 3) * 128 + (n & 7) * 16 + (k & 7) * 2;
}
// byte offset of (row, col) in a 16-bit K-major 128B-swizzled operand, K = 128
// as two 64-column blocks of 32 rows
__device__ __forceinline__ uint32_t sw128_32rows(int row, int c)
{
    return (c >> 6) * 4096 + row * 128 + ((((c & 63) >> 3) ^ (row & 7)) << 4) + (c & 7) * 2;
}
__device__ __forceinline__ float h_lo(uint32_t w) { return __low2float(*reinterpret_cast<const __half2 *>(&w)); }
__device__ __forceinline__ float h_hi(uint32_t w) { return __high2float(*reinterpret_cast<const __half2 *>(&w)); }

// D_n = V_n^T TM_n^T + Sb[b] W'_n^T [+ E[e] (Kbar_{n-2} W'_n^T)] for the prep slot at `sl`.
// Executed by the whole issuing warp; one elected lane issues.
__device__ __forceinline__ void issue_d(uint32_t tmem, uint32_t sl, int dbuf, int b, int e)
{
    const uint32_t id_u = tc::idesc(tc::F16, 128, 32, 1, 0);
    const uint32_t id_c = tc::idesc(tc::F16, 128, 32, 0, 0);
    const uint32_t dn = tmem + T_D + 32 * dbuf;
    // descriptor of W', advanced by adding (byte offset >> 4) to the address field
    const uint64_t dz = tc::sdesc(sl + L_Z, 16, 1024, tc::SWZ_128B);
    tc::mma_ss_w(dn, tc::sdesc(sl + L_V16, 2048, 1024, tc::SWZ_128B), tc::sdesc(sl + L_TM, 128, 256, tc::SWZ_NONE), id_u, 0);
#pragma unroll
    for (int i = 0; i < 8; ++i)
        tc::mma_ts_w(dn, tmem + T_SB + 64 * b + 8 * i, dz + (((i >> 2) * 4096 + (i & 3) * 32) >> 4), id_c, 1);
    if (e >= 0) tc::mma_ts_w(dn, tmem + T_E + 8 * e, tc::sdesc(sl + L_HP, 128, 256, tc::SWZ_NONE), id_c, 1);
}

// L2 scale factors 1 / sqrt(sum x^2 + 1e-6) of the four k rows and four q rows held by this
// warp (a thread holds 4 channels of each row, the warp all 128). The eight sums of squares
// are reduced in a reduce-scatter butterfly (each exchange halves the values a lane keeps),
// so lane l ends with the full sum of value (l >> 2): k rows 0..3, then q rows 0..3.
__device__ __forceinline__ void qk_row_scales(const uint2 (&kw)[4], const uint2 (&qw)[4], int lane, float (&sk)[4],
                                              float (&sq)[4])
{
    float v[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float k0 = bf16_lo(kw[i].x), k1 = bf16_hi(kw[i].x), k2 = bf16_lo(kw[i].y), k3 = bf16_hi(kw[i].y);
        const float q0 = bf16_lo(qw[i].x), q1 = bf16_hi(qw[i].x), q2 = bf16_lo(qw[i].y), q3 = bf16_hi(qw[i].y);
        v[i] = fmaf(k0, k0, fmaf(k1, k1, fmaf(k2, k2, k3 * k3)));
        v[4 + i] = fmaf(q0, q0, fmaf(q1, q1, fmaf(q2, q2, q3 * q3)));
    }
#pragma unroll
    for (int w = 16, n = 4; w >= 4; w >>= 1, n >>= 1) {
        const bool up = lane & w;
#pragma unroll
        for (int i = 0; i < n; ++i) {
            const float keep = up ? v[i + n] : v[i], send = up ? v[i] : v[i + n];
            v[i] = keep + __shfl_xor_sync(0xffffffffu, send, w);
        }
    }
    v[0] += __shfl_xor_sync(0xffffffffu, v[0], 2);
    v[0] += __shfl_xor_sync(0xffffffffu, v[0], 1);
    const float f = rsqrtf(v[0] + 1e-6f);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        sk[i] = __shfl_sync(0xffffffffu, f, 4 * i);
        sq[i] = __shfl_sync(0xffffffffu, f, 16 + 4 * i);
    }
}

// acc[nt] (16 rows r x 16 columns j) = sum_c X[r][c] R[j][c] over the 64 channels c in [cbase, cbase + 64),
// from fp32 tiles [16][132] (528-byte rows), on m16n8k8 tf32 warp MMA. ldmatrix on 32-bit data hands
// thread 4 g + t the word (row g, column t) of each 8 x 4 block: the tf32 A and B fragment layouts.
__device__ __forceinline__ void chunk_gram_tf32(uint32_t x, uint32_t r, Frag16 &acc, int lane, int cbase)
{
    const int mi = lane >> 3, ri = lane & 7;
    const uint32_t aoff = (ri + 8 * (mi & 1)) * F_LD + 16 * (mi >> 1) + 4 * cbase;  // A: rows r, k = c
    const uint32_t boff = (ri + 8 * (mi >> 1)) * F_LD + 16 * (mi & 1) + 4 * cbase;  // B: rows j, k = c
    frag_zero(acc);
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
        uint32_t a[4], b[4];
        ldsm_x4(x + aoff + 32 * kk, a[0], a[1], a[2], a[3]);
        ldsm_x4(r + boff + 32 * kk, b[0], b[1], b[2], b[3]);
        mma_tf32(acc.c[0], a, b[0], b[1]);
        mma_tf32(acc.c[1], a, b[2], b[3]);
    }
}

// QKN: L2-normalise the q and k rows in the element-wise pass (KDA_FLAG_QK_L2NORM).
template <bool QKN>
__global__ void __launch_bounds__(NTHREADS, 1)
    kda_fwd_tc_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                      const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap tg, const Params p)
{
    extern __shared__ uint8_t smem_dyn[];
    // align to 1024 B by pointer arithmetic on the shared array, so that accesses
    // through `smem` stay in the shared address space
    uint8_t *smem = smem_dyn + ((1024u - (smem_u32(smem_dyn) & 1023u)) & 1023u);
    const uint32_t sb = smem_u32(smem);
// plain C++ shared-memory access at a 32-bit shared address (lets the compiler schedule it)
#define SM_AT(T, a) (*reinterpret_cast<T *>(smem + ((a) - sb)))
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int h = blockIdx.x % p.H;
    const int seq = (p.cu && p.nseq <= LPT_MAX_SEQS) ? lpt_sequence(p, blockIdx.x / p.H) : blockIdx.x / p.H;
    const Span sp = seq_span(p, seq);
    if (threadIdx.x == 0) {
        if (p.cu && blockIdx.x == 0 && (p.cu[0] != 0 || p.cu[p.nseq] != p.total)) atomicOr(&g_dev_error, DEVERR_SEQLENS);
        if (!sp.ok && h == 0) atomicOr(&g_dev_error, DEVERR_SEQLENS);
    }
    if (!sp.ok) return;  // CTA-uniform, before any tensor memory is taken
    const int nch = (sp.len + CHUNK - 1) / CHUNK;

    volatile int *flags = reinterpret_cast<volatile int *>(smem + OFF_FLAGS);
    auto bar = [&](int i) { return sb + OFF_BAR + 8 * i; };
    auto slot = [&](int n) { return sb + OFF_SLOT + (n % NP) * SLOT; };

    if (warp == 0) {
        tc::alloc(sb + OFF_TMEMPTR, TMEM_COLS);
        tc::relinquish();
    }
    if (threadIdx.x == 32) {
        for (int i = 0; i < NR; ++i) {
            mbar_init(bar(B_RAW_FULL + i), 1);
            mbar_init(bar(B_RAW_EMPTY + i), 1);
        }
        for (int i = 0; i < NP; ++i) {
            mbar_init(bar(B_PREP_FULL + i), NFIN);           // the chunk's finisher warps
            mbar_init(bar(B_PREP_EMPTY + i), 1 + 2 * NFIN);  // the state update's commit + the finishers of the next two chunks
            mbar_init(bar(B_P2 + i), 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(bar(B_D + i), 1);
            mbar_init(bar(B_E + i), 4);
            mbar_init(bar(B_G + i), 4);
            mbar_init(bar(B_S + i), 1);
        }
        mbar_init(bar(B_I), 4);
        mbar_init(bar(B_F), 1);
        for (int i = 0; i < 4; ++i) {
            mbar_init(bar(B_GRAM + i), 4);
            mbar_init(bar(B_FDONE + i), NFIN);
            mbar_init(bar(B_ZREAD + i), 1);
        }
        flags[0] = 0;
        fence_mbar_init();
    }
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(smem + OFF_TMEMPTR);

    if (warp == 0) {
        // ---------------------------------------------------------------- producer
        if (lane == 0) {
            tma_prefetch_desc(&tq);
            tma_prefetch_desc(&tk);
            tma_prefetch_desc(&tv);
            tma_prefetch_desc(&tg);
            int n = 0;
            for (; n < nch; ++n) {
                const int s = n % NR;
                if (!wait_bar(bar(B_RAW_EMPTY + s), ((n / NR) & 1) ^ 1, flags)) break;
                const uint32_t fb = bar(B_RAW_FULL + s);
                mbar_arrive_expect_tx(fb, RAW_STAGE);
                const int tok = sp.bos + n * CHUNK;
                const uint32_t dst = sb + OFF_RAW + s * RAW_STAGE;
#pragma unroll
                for (int b = 0; b < 2; ++b) {
                    tma_load_3d(dst + OFF_Q + b * RAW_BOX, &tq, 64 * b, h, tok, fb);
                    tma_load_3d(dst + OFF_K + b * RAW_BOX, &tk, 64 * b, h, tok, fb);
                    tma_load_3d(dst + OFF_V + b * RAW_BOX, &tv, 64 * b, h, tok, fb);
                    tma_load_3d(dst + OFF_G + b * RAW_BOX, &tg, 64 * b, h, tok, fb);
                }
            }
            for (int m = (n > NR ? n - NR : 0); m < n; ++m) drain_bar(bar(B_RAW_FULL + m % NR), (m / NR) & 1);
        }
    } else if (warp == 1) {
        // ---------------------------------------------------------------- MMA issuer (whole warp)
        if (nch > 0) {
            const uint32_t id_c = tc::idesc(tc::F16, 128, 32, 0, 0);
            const uint32_t id_s = tc::idesc(tc::F16, 128, 128, 0, 1);  // Kbar MN-major
            // every lane waits; the warp goes on only when all lanes saw the phase (or all give up)
            auto wait_all = [&](int b, uint32_t par) {
                const bool ok = __all_sync(0xffffffffu, wait_bar(bar(b), par, flags));
                __syncwarp();
                return ok;
            };
            bool ok = wait_all(B_I, 0);
            for (int n = 0; ok && n < (nch < 2 ? nch : 2); ++n) {
                ok = wait_all(B_PREP_FULL + n % NP, (n / NP) & 1);
                if (!ok) break;
                tc::fence_after();
                issue_d(tmem, slot(n), n % 3, n & 1, -1);
                if (n == 0) tc::commit_w(bar(B_D + 0));
            }
            for (int k = 0; ok && k < nch; ++k) {
                ok = wait_all(B_E + (k & 1), (k >> 1) & 1);
                if (!ok) break;
                tc::fence_after();
                const uint32_t e = tmem + T_E + 8 * (k & 1);
                if (k + 1 < nch) {  // D_{k+1} += E_k (Kbar_k W_{k+1}^T)
                    tc::mma_ts_w(tmem + T_D + 32 * ((k + 1) % 3), e, tc::sdesc(slot(k + 1) + L_CC, 128, 256, tc::SWZ_NONE),
                                 id_c, 1);
                    tc::commit_w(bar(B_D + ((k + 1) & 1)));
                }
                ok = wait_all(B_G + (k & 1), (k >> 1) & 1);
                if (!ok) break;
                tc::fence_after();
                // S += E_k Kbar_k (the state was decayed in place by the state warps)
                tc::mma_ts_w(tmem + T_S, e, tc::sdesc(slot(k) + L_KB, 2048, 1024, tc::SWZ_128B), id_s, 1);
                tc::commit_w(bar(B_S + (k & 1)));
                tc::commit_w(bar(B_PREP_EMPTY + k % NP));
                if (k + 2 < nch) {
                    const int n = k + 2;
                    ok = wait_all(B_PREP_FULL + n % NP, (n / NP) & 1);
                    if (!ok) break;
                    tc::fence_after();
                    issue_d(tmem, slot(n), n % 3, k & 1, k & 1);
                }
            }
            tc::commit_w(bar(B_F));
            if (lane == 0) drain_bar(bar(B_F), 0);
            __syncwarp();
        }
    } else if (warp < 6) {
        // ---------------------------------------------------------------- state warps
        const int q4 = warp & 3;
        const int row = 32 * q4 + lane;
        const uint32_t lb = tmem + (static_cast<uint32_t>(32 * q4) << 16);
        const size_t st_row = (static_cast<size_t>(seq) * p.H + h) * (DH * DH) + static_cast<size_t>(row) * DH;
        // S_0, and f16(S_0) for the products of chunks 0 and 1 (chunk 1's W' carries gamma_0)
        bool ok = true;
#pragma unroll 1
        for (int g4 = 0; g4 < 4; ++g4) {
            uint32_t r32[32], r16[16];
            if (!p.init) {
#pragma unroll
                for (int i = 0; i < 32; ++i) r32[i] = 0u;
            } else if (p.init_dtype == KDA_DTYPE_FP32) {
                const uint4 *src = reinterpret_cast<const uint4 *>(static_cast<const float *>(p.init) + st_row + 32 * g4);
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const uint4 w = src[i];
                    r32[4 * i] = w.x;
                    r32[4 * i + 1] = w.y;
                    r32[4 * i + 2] = w.z;
                    r32[4 * i + 3] = w.w;
                }
            } else {
                const uint4 *src = reinterpret_cast<const uint4 *>(static_cast<const uint16_t *>(p.init) + st_row + 32 * g4);
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const uint4 w = src[i];
                    r32[8 * i] = w.x << 16;
                    r32[8 * i + 1] = w.x & 0xffff0000u;
                    r32[8 * i + 2] = w.y << 16;
                    r32[8 * i + 3] = w.y & 0xffff0000u;
                    r32[8 * i + 4] = w.z << 16;
                    r32[8 * i + 5] = w.z & 0xffff0000u;
                    r32[8 * i + 6] = w.w << 16;
                    r32[8 * i + 7] = w.w & 0xffff0000u;
                }
            }
#pragma unroll
            for (int i = 0; i < 32; i += 2) r16[i / 2] = pack_f16(__uint_as_float(r32[i]), __uint_as_float(r32[i + 1]));
            tc::st32(lb + T_S + 32 * g4, r32);
            tc::st16(lb + T_SB + 16 * g4, r16);
            tc::st16(lb + T_SB + 64 + 16 * g4, r16);
        }
        tc::wait_st();
        tc::fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(B_I));

        uint16_t *op = p.out + (static_cast<size_t>(sp.bos) * p.H + h) * DH + row;
        const size_t ostride = static_cast<size_t>(p.H) * DH;
        for (int k = 0; ok && k < nch; ++k) {
            ok = wait_bar(bar(B_D + (k & 1)), (k >> 1) & 1, flags);
            if (!__all_sync(0xffffffffu, ok)) {
                ok = false;
                break;
            }
            tc::fence_after();
            uint32_t o8[8];  // outputs as bf16 pairs, stored after the decay pass
            {  // E_k (f16) -> tensor memory, then release the chain
                uint32_t d[32], e8[8];
                tc::ld32(lb + T_D + 32 * (k % 3), d);
                tc::wait_ld();
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    e8[i] = pack_f16(__uint_as_float(d[2 * i]), __uint_as_float(d[2 * i + 1]));
                    o8[i] = pack_bf16(__uint_as_float(d[16 + 2 * i]), __uint_as_float(d[17 + 2 * i]));
                }
                tc::st8(lb + T_E + 8 * (k & 1), e8);
                tc::wait_st();
                tc::fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(B_E + (k & 1)));
            }
            // decay the state for this chunk, S <- S Diag(gamma_k), and keep f16 of it for
            // chunk k + 2's product (whose W' carries gamma_{k+1})
            ok = (k == 0) || wait_bar(bar(B_S + ((k - 1) & 1)), ((k - 1) >> 1) & 1, flags);
            ok = ok && wait_bar(bar(B_PREP_FULL + k % NP), (k / NP) & 1, flags);
            if (!__all_sync(0xffffffffu, ok)) {
                ok = false;
                break;
            }
            tc::fence_after();
            const uint32_t gam = slot(k) + L_GAM;
#pragma unroll 1
            for (int g4 = 0; g4 < 4; ++g4) {
                uint32_t r32[32], r16[16];
                tc::ld32(lb + T_S + 32 * g4, r32);
                tc::wait_ld();
#pragma unroll
                for (int i = 0; i < 32; i += 4) {
                    const float4 gv = SM_AT(const float4, gam + (32 * g4 + i) * 4);
                    const float2 a01 = fmul2(make_float2(__uint_as_float(r32[i]), __uint_as_float(r32[i + 1])), make_float2(gv.x, gv.y));
                    const float2 a23 = fmul2(make_float2(__uint_as_float(r32[i + 2]), __uint_as_float(r32[i + 3])), make_float2(gv.z, gv.w));
                    r32[i] = __float_as_uint(a01.x);
                    r32[i + 1] = __float_as_uint(a01.y);
                    r32[i + 2] = __float_as_uint(a23.x);
                    r32[i + 3] = __float_as_uint(a23.y);
                    r16[i / 2] = pack_f16(a01.x, a01.y);
                    r16[i / 2 + 1] = pack_f16(a23.x, a23.y);
                }
                tc::st32(lb + T_S + 32 * g4, r32);
                tc::st16(lb + T_SB + 64 * (k & 1) + 16 * g4, r16);
            }
            tc::wait_st();
            tc::fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(B_G + (k & 1)));
            // outputs (already scaled), straight from registers: one 2-byte store per token,
            // 64 contiguous bytes per warp; rows past the sequence end are not written
            const int Lv = min(CHUNK, sp.len - k * CHUNK);
            if (Lv == CHUNK) {
#pragma unroll
                for (int r = 0; r < CHUNK; ++r) op[r * ostride] = static_cast<uint16_t>(o8[r >> 1] >> (16 * (r & 1)));
            } else {
#pragma unroll
                for (int r = 0; r < CHUNK; ++r)
                    if (r < Lv) op[r * ostride] = static_cast<uint16_t>(o8[r >> 1] >> (16 * (r & 1)));
            }
            op += CHUNK * ostride;
        }
        if (p.fin) {
            if (ok && nch > 0) ok = wait_bar(bar(B_S + ((nch - 1) & 1)), ((nch - 1) >> 1) & 1, flags);
            ok = __all_sync(0xffffffffu, ok);
            tc::fence_after();
#pragma unroll 1
            for (int g4 = 0; g4 < 4; ++g4) {
                uint32_t r32[32];
                tc::ld32(lb + T_S + 32 * g4, r32);
                tc::wait_ld();
                if (p.fin_dtype == KDA_DTYPE_FP32) {
                    float4 *dst = reinterpret_cast<float4 *>(static_cast<float *>(p.fin) + st_row + 32 * g4);
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        dst[i] = make_float4(__uint_as_float(r32[4 * i]), __uint_as_float(r32[4 * i + 1]),
                                             __uint_as_float(r32[4 * i + 2]), __uint_as_float(r32[4 * i + 3]));
                } else {
                    uint4 *dst = reinterpret_cast<uint4 *>(static_cast<uint16_t *>(p.fin) + st_row + 32 * g4);
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        dst[i] = make_uint4(pack_bf16(__uint_as_float(r32[8 * i]), __uint_as_float(r32[8 * i + 1])),
                                            pack_bf16(__uint_as_float(r32[8 * i + 2]), __uint_as_float(r32[8 * i + 3])),
                                            pack_bf16(__uint_as_float(r32[8 * i + 4]), __uint_as_float(r32[8 * i + 5])),
                                            pack_bf16(__uint_as_float(r32[8 * i + 6]), __uint_as_float(r32[8 * i + 7])));
                }
            }
        }
        tc::fence_before();
    } else if (warp < 14) {
        // ---------------------------------------------------------------- prep lanes
        // lane = 4 warps = 128 threads, alternate chunks. Element-wise passes: thread ->
        // channels [c0, c0 + 4) (c0 = 4 lane), rows [4 rq, 4 rq + 4) (row quarter rq = warp
        // in lane). The lane forms the gate, the scaled key / query tiles and the
        // chunk-product partial sums; its finisher warp does the rest.
        const int ln = (warp - 6) >> 2;
        const int lt = threadIdx.x - 192 - 128 * ln;  // 0..127
        const int lw = lt >> 5;
        const uint32_t bar_id = 1 + ln;
        const uint32_t scr = sb + OFF_SCR + ln * SCR;
        const int rq = lw;
        const int c0 = 4 * lane, r0 = 4 * rq;
        // x / 2 = ah2 * g + bb, with x = exp(A_log) (g + dt_bias)
        float ah2 = 0.5f, bb[4] = {0.f, 0.f, 0.f, 0.f};
        if (p.A_log) ah2 = 0.5f * ex2_approx(__ldg(p.A_log + h) * LOG2E);
        if (p.dt_bias) {
#pragma unroll
            for (int j = 0; j < 4; ++j) bb[j] = ah2 * __ldg(p.dt_bias + h * DH + c0 + j);
        }
        const float hs = p.half_gs;

        // bf16 bits of the beta logit of row lt of chunk n, loaded one lane-chunk ahead and
        // left untouched until used (rows past the sequence end read its last row and are
        // masked where they are used)
        auto beta_bits = [&](int n) -> uint32_t {
            if (lt >= CHUNK) return 0u;
            const int r = min(n * CHUNK + lt, sp.len - 1);
            return __ldg(p.beta + static_cast<size_t>(sp.bos + r) * p.H + h);
        };
        uint32_t bnext = ln < nch ? beta_bits(ln) : 0u;
        bool failed = false;  // sticky: a wait gave up; OR-reduced at the lane barriers
        for (int n = ln; n < nch; n += 2) {
            const int rs = n % NR;
            const uint32_t sl = slot(n);
            const int Lv = min(CHUNK, sp.len - n * CHUNK);
            const uint32_t bbits = bnext;
            if (n + 2 < nch) bnext = beta_bits(n + 2);
            const int xb = (n >> 1) & 1;                        // finisher buffer of this chunk
            const uint32_t xpar = static_cast<uint32_t>(n >> 2) & 1;
            if (!wait_bar(bar(B_RAW_FULL + rs), (n / NR) & 1, flags)) failed = true;
            const uint32_t raw = sb + OFF_RAW + rs * RAW_STAGE;

            // gate (log2 units) over this thread's 4 rows x 4 channels, local inclusive cumsum;
            // rows past the chunk's end add nothing
            float G[4][4];
            {
                float a[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int r = r0 + i;
                    const uint2 gw = SM_AT(const uint2, raw + OFF_G + raw_off(r, c0));
                    const float gx[4] = {bf16_lo(gw.x), bf16_hi(gw.x), bf16_lo(gw.y), bf16_hi(gw.y)};
                    const bool live = r < Lv;
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const float tj = tanh_approx(fmaf(ah2, gx[j], bb[j]));
                        a[j] += live ? fmaf(hs, tj, hs) : 0.f;
                        G[i][j] = a[j];
                    }
                }
            }
            if (!wait_bar(bar(B_PREP_EMPTY + n % NP), ((n / NP) & 1) ^ 1, flags)) failed = true;
            // the finisher is done with this buffer's previous chunk
            if (!wait_bar(bar(B_FDONE + 2 * ln + xb), xpar ^ 1, flags)) failed = true;
            // gate sums of the row quarters, in this chunk's partial-sum buffer (free until the products)
            const uint32_t gsum = scr + S_GP + xb * 4096;
            SM_AT(float4, gsum + rq * 512 + lane * 16) = make_float4(G[3][0], G[3][1], G[3][2], G[3][3]);
            if (lt < CHUNK)
                SM_AT(float, scr + S_BETA + xb * 64 + lt * 4) =
                    lt < Lv ? fmaf(0.5f, tanh_approx(0.5f * __uint_as_float(bbits << 16)), 0.5f) : 0.f;
            if (named_bar_or(bar_id, 128, failed)) break;
            // quarter sums -> prefix before this quarter; Gm = G at row 7 (reference: halves the
            // exponent range), Ge = G at row 15; d = G_r - Gm = G_local - (Gm - prefix)
            float off[4], gr[4], se[4];
            {
                const float4 s0 = SM_AT(const float4, gsum + 0 * 512 + lane * 16);
                const float4 s1 = SM_AT(const float4, gsum + 1 * 512 + lane * 16);
                const float4 s2 = SM_AT(const float4, gsum + 2 * 512 + lane * 16);
                const float4 s3 = SM_AT(const float4, gsum + 3 * 512 + lane * 16);
                const float q0[4] = {s0.x, s0.y, s0.z, s0.w}, q1[4] = {s1.x, s1.y, s1.z, s1.w};
                const float q2[4] = {s2.x, s2.y, s2.z, s2.w}, q3[4] = {s3.x, s3.y, s3.z, s3.w};
                float ge[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const float pre = rq == 0 ? 0.f : rq == 1 ? q0[j] : rq == 2 ? q0[j] + q1[j] : q0[j] + q1[j] + q2[j];
                    const float gm = q0[j] + q1[j];
                    ge[j] = gm + q2[j] + q3[j];
                    off[j] = gm - pre;
                    gr[j] = ex2_approx(gm);            // 2^Gm
                    se[j] = ex2_approx(ge[j] - gm);    // 2^(Ge - Gm)
                }
                if (rq == 3)
                    SM_AT(float4, sl + L_GAM + c0 * 4) =
                        make_float4(ex2_approx(ge[0]), ex2_approx(ge[1]), ex2_approx(ge[2]), ex2_approx(ge[3]));
            }
            // all raw loads first: stores below may alias them as far as the compiler knows
            uint2 kwv[4], qwv[4], vwv[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int r = r0 + i;
                const uint2 kraw = SM_AT(const uint2, raw + OFF_K + raw_off(r, c0));
                kwv[i] = r < Lv ? kraw : make_uint2(0u, 0u);  // keys past the chunk's end are zero
                qwv[i] = SM_AT(const uint2, raw + OFF_Q + raw_off(r, c0));
                vwv[i] = SM_AT(const uint2, raw + OFF_V + raw_off(r, c0));
            }
            float sk[4], sq[4];
            if constexpr (QKN) qk_row_scales(kwv, qwv, lane, sk, sq);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int r = r0 + i;
                float k[4] = {bf16_lo(kwv[i].x), bf16_hi(kwv[i].x), bf16_lo(kwv[i].y), bf16_hi(kwv[i].y)};
                float q[4] = {bf16_lo(qwv[i].x), bf16_hi(qwv[i].x), bf16_lo(qwv[i].y), bf16_hi(qwv[i].y)};
                if constexpr (QKN) {
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        k[j] *= sk[i];
                        q[j] *= sq[i];
                    }
                }
                float kl[4], ql[4], kr[4], kg[4], qg[4], kb[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const float d = G[i][j] - off[j];
                    const float u = ex2_approx(d), f = ex2_approx(-d);  // 2^(G_r - Gm), 2^(Gm - G_r)
                    kl[j] = k[j] * u;
                    ql[j] = q[j] * u;
                    kr[j] = k[j] * f;
                    kg[j] = kl[j] * gr[j];  // K * Gamma
                    qg[j] = ql[j] * gr[j];  // Q * Gamma
                    kb[j] = kr[j] * se[j];  // Kbar = K * 2^(Ge - G_r)
                }
                const uint32_t o = r * F_LD + c0 * 4;
                SM_AT(uint2, sl + L_Z + sw128_32rows(r, c0)) = make_uint2(pack_f16(kg[0], kg[1]), pack_f16(kg[2], kg[3]));
                SM_AT(uint2, sl + L_Z + sw128_32rows(16 + r, c0)) = make_uint2(pack_f16(qg[0], qg[1]), pack_f16(qg[2], qg[3]));
                const uint2 vw = vwv[i];
                SM_AT(uint2, sl + L_V16 + raw_off(r, c0)) = make_uint2(pack_f16(bf16_lo(vw.x), bf16_hi(vw.x)),
                                                                       pack_f16(bf16_lo(vw.y), bf16_hi(vw.y)));
                SM_AT(uint2, sl + L_KB + raw_off(r, c0)) = make_uint2(pack_f16(kb[0], kb[1]), pack_f16(kb[2], kb[3]));
                SM_AT(float4, scr + S_KL + o) = make_float4(kl[0], kl[1], kl[2], kl[3]);
                SM_AT(float4, scr + S_QL + o) = make_float4(ql[0], ql[1], ql[2], ql[3]);
                SM_AT(float4, scr + S_KR + o) = make_float4(kr[0], kr[1], kr[2], kr[3]);
            }
            tc::fence_async_smem();  // V and Kbar are read by the tensor core
            named_bar_sync(bar_id, 128);
            if (lt == 0) {
                mbar_arrive(bar(B_RAW_EMPTY + rs));
                mbar_arrive(bar(B_P2 + n % NP));  // Kbar_n and gamma_n are in the slot
            }

            // A (warps 0, 2) and P (warps 1, 3) partial sums over one channel half each, on tf32 warp MMA
            {
                Frag16 acc;
                chunk_gram_tf32(scr + ((lw & 1) ? S_QL : S_KL), scr + S_KR, acc, lane, 64 * (lw >> 1));
                const uint32_t gp = scr + S_GP + xb * 4096 + lw * 1024 + lane * 16;
                SM_AT(float4, gp) = make_float4(acc.c[0][0], acc.c[0][1], acc.c[0][2], acc.c[0][3]);
                SM_AT(float4, gp + 512) = make_float4(acc.c[1][0], acc.c[1][1], acc.c[1][2], acc.c[1][3]);
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(B_GRAM + 2 * ln + xb));
            }
        }
    } else {
        // ---------------------------------------------------------------- finishers
        // NFIN warps per prep lane. A and P from the lane's partial sums, T' = (I + A)^-1 diag(beta)
        // and M = P T'; then, 16 channels at a time, the 16-row halves of W = Phi Z (half 0:
        // -T' (K Gamma); half 1: s (Q Gamma) - s M (K Gamma)) are written over Z as
        // W' = W Diag(gamma_{n-1}), and their columns of Kbar_{n-1} W^T and Kbar_{n-2} W'^T are
        // accumulated; then the slot is handed on. Half 0 writes over the K Gamma rows that half 1
        // reads: with two warps it stores only once half 1 is done, with one warp it runs second.
        const int fw = warp - (NTHREADS / 32 - 2 * NFIN);
        const int ln = fw / NFIN, myhalf = fw % NFIN;
        const uint32_t scr = sb + OFF_SCR + ln * SCR;
        const float sc = p.scale;
        const int g = lane >> 2, t = lane & 3;
        const int mi = lane >> 3, ri = lane & 7;
        const uint32_t stsm_row = (mi >> 1) * 256 + (mi & 1) * 128 + ri * 16;
        constexpr uint32_t NEG2 = 0x80008000u;  // negates both halves of an f16 pair
        for (int n = ln; n < nch; n += 2) {
            const int xb = (n >> 1) & 1;
            const uint32_t xpar = static_cast<uint32_t>(n >> 2) & 1;
            const uint32_t sl = slot(n);
            const uint32_t gp = scr + S_GP + xb * 4096 + lane * 16;
            const uint32_t bet = scr + S_BETA + xb * 64;
            if (!__all_sync(0xffffffffu, wait_bar(bar(B_GRAM + 2 * ln + xb), xpar, flags))) break;
            // A = strictly-lower part with rows scaled by beta; P = lower part (diagonal included)
            Frag16 A, P;
            {
                float4 x[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) x[i] = SM_AT(const float4, gp + 512 * i);  // [warp][tile]
                const float4 a0 = make_float4(x[0].x + x[4].x, x[0].y + x[4].y, x[0].z + x[4].z, x[0].w + x[4].w);
                const float4 a1 = make_float4(x[1].x + x[5].x, x[1].y + x[5].y, x[1].z + x[5].z, x[1].w + x[5].w);
                const float4 p0 = make_float4(x[2].x + x[6].x, x[2].y + x[6].y, x[2].z + x[6].z, x[2].w + x[6].w);
                const float4 p1 = make_float4(x[3].x + x[7].x, x[3].y + x[7].y, x[3].z + x[7].z, x[3].w + x[7].w);
                const float av[2][4] = {{a0.x, a0.y, a0.z, a0.w}, {a1.x, a1.y, a1.z, a1.w}};
                const float pv[2][4] = {{p0.x, p0.y, p0.z, p0.w}, {p1.x, p1.y, p1.z, p1.w}};
                const float bg = SM_AT(const float, bet + g * 4), bg8 = SM_AT(const float, bet + (g + 8) * 4);
#pragma unroll
                for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int r = g + 8 * (i >> 1), j = 8 * nt + 2 * t + (i & 1);
                        A.c[nt][i] = j < r ? av[nt][i] * ((i >> 1) ? bg8 : bg) : 0.f;
                        P.c[nt][i] = j <= r ? pv[nt][i] : 0.f;
                    }
            }
            Frag16 T;
            unit_lower_inverse(A, T, g, t);
            // T' = T diag(beta) rounded to f16 once: tw[col block][row block] in fragment layout;
            // TM rows 0..15 = T'
            uint32_t tw[2][2];
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
                const int col = 8 * nt + 2 * t;
                const float2 bc = SM_AT(const float2, bet + col * 4);
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    const uint32_t w = pack_f16(T.c[nt][2 * hh] * bc.x, T.c[nt][2 * hh + 1] * bc.y);
                    tw[nt][hh] = w;
                    if (myhalf == 0) SM_AT(uint32_t, sl + L_TM + cm16(g + 8 * hh, col)) = w;
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(B_FDONE + 2 * ln + xb));  // partial sums and beta are read
            // A fragments of the rows of Phi in the K Gamma columns: -T' (half 0) and -s M (half 1),
            // M = P T' with s M rounded to f16 once (TM rows 16..31)
            const uint32_t aT[4] = {tw[0][0] ^ NEG2, tw[0][1] ^ NEG2, tw[1][0] ^ NEG2, tw[1][1] ^ NEG2};
            uint32_t aM[4] = {0u, 0u, 0u, 0u};
            if (NFIN == 1 || myhalf == 1) {
                uint32_t aP[4];
                frag_as_a(P, aP);
                float m[2][4];
#pragma unroll
                for (int nb = 0; nb < 2; ++nb) {
                    m[nb][0] = m[nb][1] = m[nb][2] = m[nb][3] = 0.f;
                    mma_f16(m[nb], aP, movm_t(tw[nb][0]), movm_t(tw[nb][1]));
                }
                uint32_t sm16[2][2];
#pragma unroll
                for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                    for (int hh = 0; hh < 2; ++hh) {
                        const uint32_t w = pack_f16(sc * m[nt][2 * hh], sc * m[nt][2 * hh + 1]);
                        sm16[nt][hh] = w;
                        SM_AT(uint32_t, sl + L_TM + cm16(16 + g + 8 * hh, 8 * nt + 2 * t)) = w;
                    }
                aM[0] = sm16[0][0] ^ NEG2;
                aM[1] = sm16[0][1] ^ NEG2;
                aM[2] = sm16[1][0] ^ NEG2;
                aM[3] = sm16[1][1] ^ NEG2;
            }
            // Kbar_{n-1} and gamma_{n-1} (the other lane's previous chunk) are in their slot
            if (n >= 1 && !__all_sync(0xffffffffu, wait_bar(bar(B_P2 + (n - 1) % NP), ((n - 1) / NP) & 1, flags))) break;
            const uint32_t prev = slot(n + NP - 1), prev2 = slot(n + NP - 2);
            uint32_t keep[8][4];  // with two finisher warps, half 0's W' fragments (stored once half 1 read K Gamma)
            // this warp's 16-row halves of W: both with one finisher warp per lane, else its own
            constexpr int NH = NFIN == 1 ? 2 : 1;
            const int h0 = NFIN == 1 ? 0 : myhalf;
            const bool defer = NFIN == 2 && myhalf == 0;  // store W' only once the other warp has read K Gamma
            float hc[NH][2][4], hp[NH][2][4];  // this warp's columns of Kbar_{n-1} W^T and Kbar_{n-2} W'^T
#pragma unroll
            for (int a = 0; a < NH; ++a)
#pragma unroll
                for (int i = 0; i < 2; ++i)
#pragma unroll
                    for (int j = 0; j < 4; ++j) hc[a][i][j] = hp[a][i][j] = 0.f;
#pragma unroll (W_UNROLL)
            for (int kk = 0; kk < 8; ++kk) {
                // this lane's matrix row for ldmatrix / stmatrix: W (or Z) row ri + 8 (mi & 1) [+ 16],
                // channels 16 kk + 8 (mi >> 1) ..
                const uint32_t za = sl + L_Z + sw128_32rows(ri + 8 * (mi & 1), 16 * kk + 8 * (mi >> 1));
                uint32_t bz[4];
                ldsm_x4_t(za, bz[0], bz[1], bz[2], bz[3]);  // B fragments of the K Gamma rows (k = row, n = channel)
                // W' = W Diag(gamma_{n-1}) over channels 16 kk + 8 nt + 2 t + {0, 1}
                float2 gv[2] = {make_float2(1.f, 1.f), make_float2(1.f, 1.f)};
                if (n >= 1) {
                    gv[0] = SM_AT(const float2, prev + L_GAM + (16 * kk + 2 * t) * 4);
                    gv[1] = SM_AT(const float2, prev + L_GAM + (16 * kk + 8 + 2 * t) * 4);
                }
                uint32_t wq[NH][2][2], wpq[NH][2][2];  // f16 pairs of W and W' as B fragments: [half][row block][k half]
#pragma unroll
                for (int a = 0; a < NH; ++a) {
                    const int half = h0 + a;
                    float w[2][4];
                    if (half == 0) {
#pragma unroll
                        for (int nt = 0; nt < 2; ++nt) w[nt][0] = w[nt][1] = w[nt][2] = w[nt][3] = 0.f;
                    } else {
                        uint32_t zq[4];
                        ldsm_x4(za + 2048, zq[0], zq[1], zq[2], zq[3]);  // Q Gamma rows (16 on) in the accumulator layout
#pragma unroll
                        for (int nt = 0; nt < 2; ++nt) {
                            w[nt][0] = sc * h_lo(zq[2 * nt]);
                            w[nt][1] = sc * h_hi(zq[2 * nt]);
                            w[nt][2] = sc * h_lo(zq[2 * nt + 1]);
                            w[nt][3] = sc * h_hi(zq[2 * nt + 1]);
                        }
                    }
                    const uint32_t aPhi[4] = {half ? aM[0] : aT[0], half ? aM[1] : aT[1], half ? aM[2] : aT[2],
                                              half ? aM[3] : aT[3]};
#pragma unroll
                    for (int nt = 0; nt < 2; ++nt) {
                        mma_f16(w[nt], aPhi, bz[2 * nt], bz[2 * nt + 1]);
                        wq[a][0][nt] = pack_f16(w[nt][0], w[nt][1]);
                        wq[a][1][nt] = pack_f16(w[nt][2], w[nt][3]);
                        wpq[a][0][nt] = pack_f16(w[nt][0] * gv[nt].x, w[nt][1] * gv[nt].y);
                        wpq[a][1][nt] = pack_f16(w[nt][2] * gv[nt].x, w[nt][3] * gv[nt].y);
                    }
                }
                if (defer) {
                    keep[kk][0] = wpq[0][0][0];
                    keep[kk][1] = wpq[0][1][0];
                    keep[kk][2] = wpq[0][0][1];
                    keep[kk][3] = wpq[0][1][1];
                } else {
                    __syncwarp();  // every lane's read of these rows is done before they are overwritten
#pragma unroll
                    for (int a = 0; a < NH; ++a)
                        stsm_x4(za + 2048 * (h0 + a), wpq[a][0][0], wpq[a][1][0], wpq[a][0][1], wpq[a][1][1]);
                }
                if (n >= 1) {
                    const uint32_t koff = raw_off(ri + 8 * (mi & 1), 16 * kk + 8 * (mi >> 1));  // A rows j, k = c
                    uint32_t aK[4];
                    ldsm_x4(prev + L_KB + koff, aK[0], aK[1], aK[2], aK[3]);
#pragma unroll
                    for (int a = 0; a < NH; ++a)
#pragma unroll
                        for (int rb = 0; rb < 2; ++rb) mma_f16(hc[a][rb], aK, wq[a][rb][0], wq[a][rb][1]);
                    if (n >= 2) {
                        ldsm_x4(prev2 + L_KB + koff, aK[0], aK[1], aK[2], aK[3]);
#pragma unroll
                        for (int a = 0; a < NH; ++a)
#pragma unroll
                            for (int rb = 0; rb < 2; ++rb) mma_f16(hp[a][rb], aK, wpq[a][rb][0], wpq[a][rb][1]);
                    }
                }
            }
            bool ok = true;
            if (NFIN == 2) {
                if (myhalf == 1) {
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bar(B_ZREAD + 2 * ln + xb));  // the K Gamma rows are read
                } else {
                    ok = __all_sync(0xffffffffu, wait_bar(bar(B_ZREAD + 2 * ln + xb), xpar, flags));
                    if (ok) {
#pragma unroll
                        for (int kk = 0; kk < 8; ++kk)
                            stsm_x4(sl + L_Z + sw128_32rows(ri + 8 * (mi & 1), 16 * kk + 8 * (mi >> 1)), keep[kk][0],
                                    keep[kk][1], keep[kk][2], keep[kk][3]);
                    }
                }
            }
            // (Kbar W^T)^T as [32 n][16 k] core matrices: column n of the 16 x 32 product is row n;
            // each half's 16 columns
#pragma unroll
            for (int a = 0; a < NH; ++a) {
                const int half = h0 + a;
                stsm_x4_t(sl + L_CC + half * 512 + stsm_row, pack_f16(hc[a][0][0], hc[a][0][1]),
                          pack_f16(hc[a][0][2], hc[a][0][3]), pack_f16(hc[a][1][0], hc[a][1][1]),
                          pack_f16(hc[a][1][2], hc[a][1][3]));
                stsm_x4_t(sl + L_HP + half * 512 + stsm_row, pack_f16(hp[a][0][0], hp[a][0][1]),
                          pack_f16(hp[a][0][2], hp[a][0][3]), pack_f16(hp[a][1][0], hp[a][1][1]),
                          pack_f16(hp[a][1][2], hp[a][1][3]));
            }
            if (!ok) break;
            tc::fence_async_smem();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(bar(B_PREP_FULL + n % NP));
                if (n >= 1) mbar_arrive(bar(B_PREP_EMPTY + (n - 1) % NP));  // last read of Kbar_{n-1}, gamma_{n-1}
                if (n >= 2) mbar_arrive(bar(B_PREP_EMPTY + (n - 2) % NP));  // last read of Kbar_{n-2}
            }
        }
    }

    tc::fence_before();
    __syncthreads();
    if (warp == 0) {
        tc::fence_after();
        tc::dealloc(tmem, TMEM_COLS);
    }
#undef SM_AT
}

}  // namespace tcs
}  // namespace kda
