// kda_fwd_tc.cuh -- KDA forward pass with the state products on the 5th-gen
// tensor core (tcgen05) and the fp32 state held in tensor memory. One CTA
// per (sequence, head) state, all 128 V rows.
//
// Chunk algebra. For chunk n (16 tokens) with state S_n (V x K) at its start,
// the prep lanes reduce the chunk to
//   Z_n = [K*Gamma ; Q*Gamma] (32 x K),  Phi_n = [[-T', 0], [-s M, s I]] (32 x 32),
//   TM_n = [T' ; s M] (32 x 16),  Kbar_n (16 x K),  gamma_n (K),  V_n,
// with T' = (I + A)^-1 diag(beta), M = P T', s = scale, so that one product
// gives both the rows written into the state and the outputs:
//   [E_n | O_n] = D_n = V_n^T TM_n^T + S_n Z_n^T Phi_n^T,
//   S_{n+1} = S_n Diag(gamma_n) + E_n Kbar_n.
// (Phi_n Z_n = [-w ; s q^] with w = T' (K*Gamma), q^ = Q*Gamma - M (K*Gamma).)
// The state product is formed two chunks ahead from the decayed state two
// chunks back and corrected by the two rank-16 updates in between (exact in
// real arithmetic):
//   S_n Z_n^T = Sb_{n-2} Z'_n^T + E_{n-2} H''_n + E_{n-1} H_n,
//   Sb_{n-2} = bf16(S_{n-2} Diag(gamma_{n-2})),  Z'_n = Z_n Diag(gamma_{n-1}),
//   H_n = Kbar_{n-1} Z_n^T,  H''_n = Kbar_{n-2} Diag(gamma_{n-1}) Z_n^T,
// so D_n = V_n^T TM_n^T + X_n Phi_n^T + E_{n-1} (H_n Phi_n^T), where
// X_n = Sb_{n-2} Z'_n^T + E_{n-2} H''_n is accumulated in tensor memory and
// read back as the (tf32) A operand of the Phi product. Only the last term
// depends on the previous chunk's result, so each chunk's critical path is one
// 16-deep MMA plus one commit, and the prep lanes never form the 32 x K rows
// of w and q^ themselves. The slot stores Z' (the prep of chunk n reads
// gamma_{n-1} from the other lane's slot), so the state warps scale the state
// by their own chunk's gate only.
//
// Warp roles (512 threads):
//   warp 0      TMA producer (lane 0); allocates / frees tensor memory.
//   warp 1      MMA issuer: the whole warp runs the issue loop with warp-uniform
//               operands and one elected lane issues each MMA and commit.
//   warps 2-5   state warps, one V row per thread (tensor-memory lane):
//               read [E|O], hand E to the tensor core, decay the state
//               (S <- S Diag(gamma)) and keep its bf16 copy, store outputs.
//   warps 6-13  two prep lanes of four warps, alternate chunks: gate, scaled
//               key / query tiles, chunk-product partial sums, H and H''.
//   warps 14-15 one finisher per lane: T', M, TM, Phi, (H Phi^T)^T; hands
//               the slot to the tensor core.
// Tensor memory (512 columns): state fp32 [0,128), D x3 [128,224),
// E x2 (f16 pairs) [224,240), bf16 state copies x2 [256,384), X x2 [384,448).
// X_n is written by MMAs and then read as the A operand of the tf32 Phi MMAs
// into a different accumulator; the tensor core orders only MMAs into the same
// accumulator, so X_n is committed and waited on before it is read, and the two
// X buffers alternate between chunks.
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
constexpr int NP = 4;  // prep slot ring
constexpr int NTHREADS = 512;

constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t T_S = 0;     // fp32 state, 128 columns
constexpr uint32_t T_D = 128;   // D[3], 32 columns each
constexpr uint32_t T_E = 224;   // E[2], 8 columns each (16 f16)
constexpr uint32_t T_SB = 256;  // bf16 state copies [2], 64 columns each
constexpr uint32_t T_X = 384;   // X[2], 32 fp32 columns each

// prep slot (bytes)
constexpr int L_Z = 0;         // bf16 Z, K-major 128B swizzle: 2 K-blocks x [32 rows][128 B]
constexpr int L_V16 = 8192;    // f16 V, MN-major 128B swizzle: 2 boxes x [16 rows][128 B]
constexpr int L_KB = 12288;    // f16 Kbar [16 j][128 c], MN-major 128B swizzle (the raw-tile layout)
constexpr int L_PHI = 16384;   // fp32 Phi [32 n][32 k], K-major core matrices (LBO 128, SBO 1024)
constexpr int L_TM = 20480;    // f16 TM [32 n][16 k]
constexpr int L_CC = 21504;    // f16 (H Phi^T)^T [32 n][16 k]
constexpr int L_HP = 22528;    // f16 H''^T [32 n][16 k]
constexpr int L_GAM = 23552;   // fp32 gamma [128]
constexpr int SLOT = 24576;

// prep scratch (per lane); 16-bit tiles are [16][136] (272-byte rows)
constexpr int H_LD = 272;
constexpr int S_KLH = 0;                 // bf16 K * 2^(G - G_mid)
constexpr int S_QLH = S_KLH + 16 * H_LD; // bf16 Q * 2^(G - G_mid)
constexpr int S_KRH = S_QLH + 16 * H_LD; // bf16 hi / lo of K * 2^(G_mid - G)
constexpr int S_KRL = S_KRH + 16 * H_LD;
constexpr int S_KG = S_KRL + 16 * H_LD;  // f16 K * Gamma
constexpr int S_QG = S_KG + 16 * H_LD;   // f16 Q * Gamma
// handed to the lane's finisher warp, two buffers (alternate chunks of the lane)
constexpr int S_BETA = S_QG + 16 * H_LD; // fp32 [2][16] beta
constexpr int S_GP = S_BETA + 128;       // fp32 [2][4 warps][2 tiles][32 lanes][4]: A (warps 0, 2) and P (1, 3) partial
                                         // sums; before them the chunk's gate sums [4 row quarters][32 lanes][4]
constexpr int S_HX = S_GP + 2 * 4096;    // [2][H^w as an f16 A fragment (32 lanes x 16 B) | H^q fragments (2 x 32 lanes x 16 B)]
constexpr int SCR = S_HX + 2 * 1536;

constexpr int OFF_RAW = 0;
constexpr int OFF_SLOT = OFF_RAW + NR * RAW_STAGE;
constexpr int OFF_SCR = OFF_SLOT + NP * SLOT;
constexpr int OFF_BAR = OFF_SCR + 2 * SCR;
// barrier indices
constexpr int B_RAW_FULL = 0, B_RAW_EMPTY = 4, B_PREP_FULL = 8, B_PREP_EMPTY = 12, B_D = 16, B_E = 18, B_G = 20,
              B_S = 22, B_I = 24, B_F = 25, B_P2 = 26, B_GRAM = 30, B_HRDY = 34, B_FDONE = 38, B_GAM = 42, B_X = 46,
              NBARS = 48;
constexpr int OFF_TMEMPTR = OFF_BAR + NBARS * 8;
constexpr int OFF_FLAGS = OFF_TMEMPTR + 16;
constexpr int SMEM_USED = OFF_FLAGS + 16;
constexpr int SMEM_ALLOC = SMEM_USED + 1024;

static_assert(NR <= 4 && NP == 4, "barrier index ranges");
static_assert(SLOT % 1024 == 0 && OFF_SLOT % 1024 == 0 && RAW_STAGE % 1024 == 0, "swizzled operands need 1024-byte alignment");
static_assert(S_KG % 16 == 0 && S_GP % 16 == 0 && S_HX % 16 == 0 && SCR % 16 == 0, "alignment");
static_assert(OFF_BAR % 8 == 0, "mbarrier alignment");
static_assert(SMEM_ALLOC <= 227 * 1024, "shared memory budget");

// byte offset of (row n, col k) in a K-major, non-swizzled f16 operand with
// 16 K elements per row: 8x8 core matrices, LBO = 128 (K), SBO = 256 (N)
__device__ __forceinline__ uint32_t cm16(int n, int k)
{
    return (n >> 3) * 256 + (k >> 3) * 128 + (n & 7) * 16 + (k & 7) * 2;
}
// byte offset of (row n, col k) in a K-major, non-swizzled fp32 (tf32) operand
// with 32 K elements per row: 8 x 4 core matrices, LBO = 128 (K), SBO = 1024 (N)
__device__ __forceinline__ uint32_t cm32(int n, int k)
{
    return (n >> 3) * 1024 + (k >> 2) * 128 + (n & 7) * 16 + (k & 3) * 4;
}
// byte offset of (row, col) in a bf16 K-major 128B-swizzled operand, K = 128
// as two 64-column blocks of 32 rows
__device__ __forceinline__ uint32_t sw128_32rows(int row, int c)
{
    return (c >> 6) * 4096 + row * 128 + ((((c & 63) >> 3) ^ (row & 7)) << 4) + (c & 7) * 2;
}
__device__ __forceinline__ float h_lo(uint32_t w) { return __low2float(*reinterpret_cast<const __half2 *>(&w)); }
__device__ __forceinline__ float h_hi(uint32_t w) { return __high2float(*reinterpret_cast<const __half2 *>(&w)); }
__device__ __forceinline__ uint32_t hmul2(uint32_t a, uint32_t b)
{
    const __half2 r = __hmul2(*reinterpret_cast<const __half2 *>(&a), *reinterpret_cast<const __half2 *>(&b));
    return *reinterpret_cast<const uint32_t *>(&r);
}

// First half of D_n for the prep slot at `sl`: D_n = V_n^T TM_n^T, and X[xb] = Sb[b] Z'_n^T
// [+ E[e] H''_n]. Executed by the whole issuing warp; one elected lane issues.
__device__ __forceinline__ void issue_x(uint32_t tmem, uint32_t sl, int dbuf, int b, int e, int xb)
{
    const uint32_t id_u = tc::idesc(tc::F16, 128, 32, 1, 0);
    const uint32_t id_c = tc::idesc(tc::F16, 128, 32, 0, 0);
    const uint32_t id_y = tc::idesc(tc::BF16, 128, 32, 0, 0);
    const uint32_t dn = tmem + T_D + 32 * dbuf, x = tmem + T_X + 32 * xb;
    // descriptors of the slot's operands, advanced by adding (byte offset >> 4) to the address field
    const uint64_t dz = tc::sdesc(sl + L_Z, 16, 1024, tc::SWZ_128B);
    tc::mma_ss_w(dn, tc::sdesc(sl + L_V16, 2048, 1024, tc::SWZ_128B), tc::sdesc(sl + L_TM, 128, 256, tc::SWZ_NONE), id_u, 0);
#pragma unroll
    for (int i = 0; i < 8; ++i)
        tc::mma_ts_w(x, tmem + T_SB + 64 * b + 8 * i, dz + (((i >> 2) * 4096 + (i & 3) * 32) >> 4), id_y, i > 0);
    if (e >= 0) tc::mma_ts_w(x, tmem + T_E + 8 * e, tc::sdesc(sl + L_HP, 128, 256, tc::SWZ_NONE), id_c, 1);
}

// Second half, once X[xb] is complete: D_n += X[xb] Phi_n^T (tf32, X as the A operand).
__device__ __forceinline__ void issue_phi(uint32_t tmem, uint32_t sl, int dbuf, int xb)
{
    const uint32_t id_p = tc::idesc(tc::TF32, 128, 32, 0, 0);
    const uint32_t dn = tmem + T_D + 32 * dbuf, x = tmem + T_X + 32 * xb;
    const uint64_t dp = tc::sdesc(sl + L_PHI, 128, 1024, tc::SWZ_NONE);
#pragma unroll
    for (int i = 0; i < 4; ++i) tc::mma_ts_tf32_w(dn, x + 8 * i, dp + ((256 * i) >> 4), id_p, 1);
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

// QKN: L2-normalise the q and k rows in the element-wise pass (KDA_FLAG_QK_L2NORM).
// DUMP: also copy each finished prep slot of CTA 0 (chunks below p.dump_chunks) to p.dump, byte
// for byte, when it is handed to the tensor core (the per-step probe; the product never sets it).
template <bool QKN, bool DUMP = false>
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
#define SM_AT(T, a) (*reinterpret_cast<T *>(smem + (smem_checked((a), sizeof(T), sb) - sb)))
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
            mbar_init(bar(B_PREP_FULL + i), 1);
            mbar_init(bar(B_PREP_EMPTY + i), 1 + 4);  // the state update's commit + the lane's warps reading it two chunks later
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(bar(B_D + i), 1);
            mbar_init(bar(B_E + i), 4);
            mbar_init(bar(B_G + i), 4);
            mbar_init(bar(B_S + i), 1);
        }
        mbar_init(bar(B_I), 4);
        mbar_init(bar(B_F), 1);
        mbar_init(bar(B_X + 0), 1);
        mbar_init(bar(B_X + 1), 1);
        for (int i = 0; i < 4; ++i) {
            mbar_init(bar(B_P2 + i), 1);
            mbar_init(bar(B_GAM + i), 1);
            mbar_init(bar(B_GRAM + i), 4);
            mbar_init(bar(B_HRDY + i), 4);
            mbar_init(bar(B_FDONE + i), 1);
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
            // D_n for slot n, from the state copy b and (e >= 0) the correction E[e] H''_n: X_n is
            // committed and waited on before the Phi MMAs read it
            auto issue_d = [&](int n, int b, int e) {
                const int xb = n & 1;
                issue_x(tmem, slot(n), n % 3, b, e, xb);
                tc::commit_w(bar(B_X + xb));
                if (!wait_all(B_X + xb, (n >> 1) & 1)) return false;
                tc::fence_after();
                issue_phi(tmem, slot(n), n % 3, xb);
                return true;
            };
            bool ok = wait_all(B_I, 0);
            for (int n = 0; ok && n < (nch < 2 ? nch : 2); ++n) {
                ok = wait_all(B_PREP_FULL + n % NP, (n / NP) & 1);
                if (!ok) break;
                tc::fence_after();
                ok = issue_d(n, n & 1, -1);
                if (ok && n == 0) tc::commit_w(bar(B_D + 0));
            }
            for (int k = 0; ok && k < nch; ++k) {
                ok = wait_all(B_E + (k & 1), (k >> 1) & 1);
                if (!ok) break;
                tc::fence_after();
                const uint32_t e = tmem + T_E + 8 * (k & 1);
                if (k + 1 < nch) {  // D_{k+1} += E_k (H_{k+1} Phi_{k+1}^T)
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
                    ok = issue_d(n, k & 1, k & 1);
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
        // S_0, and bf16(S_0) for the products of chunks 0 and 1 (chunk 1's Z carries gamma_0)
        bool ok = true;
#pragma unroll 1
        for (int g4 = 0; g4 < 4; ++g4) {
            uint32_t r32[32], r16[16];
            if (!p.init || !gmem_ok(st_row + 32 * g4, 32, state_elems(p))) {
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
            for (int i = 0; i < 32; i += 2) r16[i / 2] = pack_bf16(__uint_as_float(r32[i]), __uint_as_float(r32[i + 1]));
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
            // decay the state for this chunk, S <- S Diag(gamma_k), and keep bf16 of it for
            // chunk k + 2's product (whose Z carries gamma_{k+1})
            ok = (k == 0) || wait_bar(bar(B_S + ((k - 1) & 1)), ((k - 1) >> 1) & 1, flags);
            ok = ok && wait_bar(bar(B_PREP_FULL + k % NP), (k / NP) & 1, flags);
            if (!__all_sync(0xffffffffu, ok)) {
                ok = false;
                break;
            }
            tc::fence_after();
            const uint32_t gam = slot(k) + L_GAM;
            auto decay_block = [&](int g4, uint32_t(&r32)[32]) {
                uint32_t r16[16];
#pragma unroll
                for (int i = 0; i < 32; i += 4) {
                    const float4 gv = SM_AT(const float4, gam + (32 * g4 + i) * 4);
                    const float2 a01 = fmul2(make_float2(__uint_as_float(r32[i]), __uint_as_float(r32[i + 1])), make_float2(gv.x, gv.y));
                    const float2 a23 = fmul2(make_float2(__uint_as_float(r32[i + 2]), __uint_as_float(r32[i + 3])), make_float2(gv.z, gv.w));
                    r32[i] = __float_as_uint(a01.x);
                    r32[i + 1] = __float_as_uint(a01.y);
                    r32[i + 2] = __float_as_uint(a23.x);
                    r32[i + 3] = __float_as_uint(a23.y);
                    r16[i / 2] = pack_bf16(a01.x, a01.y);
                    r16[i / 2 + 1] = pack_bf16(a23.x, a23.y);
                }
                tc::st32(lb + T_S + 32 * g4, r32);
                tc::st16(lb + T_SB + 64 * (k & 1) + 16 * g4, r16);
            };
#pragma unroll 1
            for (int g4 = 0; g4 < 4; ++g4) {
                uint32_t ra[32];
                tc::ld32(lb + T_S + 32 * g4, ra);
                tc::wait_ld();
                decay_block(g4, ra);
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
                for (int r = 0; r < CHUNK; ++r)
                    if (gmem_ok(static_cast<size_t>(op - p.out) + r * ostride, 1, out_elems(p)))
                        op[r * ostride] = static_cast<uint16_t>(o8[r >> 1] >> (16 * (r & 1)));
            } else {
#pragma unroll
                for (int r = 0; r < CHUNK; ++r)
                    if (r < Lv && gmem_ok(static_cast<size_t>(op - p.out) + r * ostride, 1, out_elems(p)))
                        op[r * ostride] = static_cast<uint16_t>(o8[r >> 1] >> (16 * (r & 1)));
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
                if (!gmem_ok(st_row + 32 * g4, 32, state_elems(p))) {
                } else if (p.fin_dtype == KDA_DTYPE_FP32) {
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
        // in lane). The lane forms the gate, the scaled key / query tiles, the chunk-product
        // partial sums and the cross-chunk products; its finisher warp does the rest.
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
        const int t = lane & 3;
        const int mi = lane >> 3, ri = lane & 7;
        // B operand (n = tile row, k = tile column) of a row-major [16][136] 16-bit tile
        const uint32_t b_row = (ri + 8 * (mi >> 1)) * H_LD + 16 * (mi & 1);
        // transposed fragment stores into a [32 n][16 k] K-major core-matrix tile: lane 8 mi + ri
        // addresses row ri of the core matrix (n block mi >> 1, k block mi & 1)
        const uint32_t stsm_row = (mi >> 1) * 256 + (mi & 1) * 128 + ri * 16;

        // bf16 bits of the beta logit of row lt of chunk n, loaded one lane-chunk ahead and
        // left untouched until used (rows past the sequence end read its last row and are
        // masked where they are used)
        auto beta_bits = [&](int n) -> uint32_t {
            if (lt >= CHUNK) return 0u;
            const int r = min(n * CHUNK + lt, sp.len - 1);
            const size_t idx = static_cast<size_t>(sp.bos + r) * p.H + h;
            return gmem_ok(idx, 1, tokhead_elems(p)) ? __ldg(p.beta + idx) : 0u;
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
            // with in-kernel q/k normalisation the row scales come from the raw tile alone: they are
            // formed here, while the lane would otherwise wait for its slot
            float sk[4], sq[4];
            if constexpr (QKN) {
                uint2 kn[4], qn[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int r = r0 + i;
                    const uint2 kraw = SM_AT(const uint2, raw + OFF_K + raw_off(r, c0));
                    kn[i] = r < Lv ? kraw : make_uint2(0u, 0u);
                    qn[i] = SM_AT(const uint2, raw + OFF_Q + raw_off(r, c0));
                }
                qk_row_scales(kn, qn, lane, sk, sq);
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
                if (rq == 3) {
                    SM_AT(float4, sl + L_GAM + c0 * 4) =
                        make_float4(ex2_approx(ge[0]), ex2_approx(ge[1]), ex2_approx(ge[2]), ex2_approx(ge[3]));
                    __syncwarp();  // the warp's stores happen before its one arrival
                    if (lane == 0) mbar_arrive(bar(B_GAM + n % NP));
                }
            }
            // gamma_{n-1} of this thread's channels (the previous chunk, the other lane): the state
            // product of chunk n reads Z_n Diag(gamma_{n-1}) against the state decayed to the start
            // of chunk n-1, so Z is stored pre-scaled (gamma_{-1} = 1)
            float gp[4] = {1.f, 1.f, 1.f, 1.f};
            if (n >= 1) {
                if (!wait_bar(bar(B_GAM + (n - 1) % NP), ((n - 1) / NP) & 1, flags)) failed = true;
                const float4 gv = SM_AT(const float4, slot(n + NP - 1) + L_GAM + c0 * 4);
                gp[0] = gv.x; gp[1] = gv.y; gp[2] = gv.z; gp[3] = gv.w;
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
                const uint32_t o = r * H_LD + c0 * 2;
                SM_AT(uint2, scr + S_KG + o) = make_uint2(pack_f16(kg[0], kg[1]), pack_f16(kg[2], kg[3]));
                SM_AT(uint2, scr + S_QG + o) = make_uint2(pack_f16(qg[0], qg[1]), pack_f16(qg[2], qg[3]));
                SM_AT(uint2, sl + L_Z + sw128_32rows(r, c0)) =
                    make_uint2(pack_bf16(kg[0] * gp[0], kg[1] * gp[1]), pack_bf16(kg[2] * gp[2], kg[3] * gp[3]));
                SM_AT(uint2, sl + L_Z + sw128_32rows(16 + r, c0)) =
                    make_uint2(pack_bf16(qg[0] * gp[0], qg[1] * gp[1]), pack_bf16(qg[2] * gp[2], qg[3] * gp[3]));
                const uint2 vw = vwv[i];
                SM_AT(uint2, sl + L_V16 + raw_off(r, c0)) = make_uint2(pack_f16(bf16_lo(vw.x), bf16_hi(vw.x)),
                                                                       pack_f16(bf16_lo(vw.y), bf16_hi(vw.y)));
                SM_AT(uint2, sl + L_KB + raw_off(r, c0)) = make_uint2(pack_f16(kb[0], kb[1]), pack_f16(kb[2], kb[3]));
                SM_AT(uint2, scr + S_KLH + o) = make_uint2(pack_bf16(kl[0], kl[1]), pack_bf16(kl[2], kl[3]));
                SM_AT(uint2, scr + S_QLH + o) = make_uint2(pack_bf16(ql[0], ql[1]), pack_bf16(ql[2], ql[3]));
                uint32_t h0, l0, h1, l1;
                split_bf16_trunc(kr[0], kr[1], h0, l0);
                split_bf16_trunc(kr[2], kr[3], h1, l1);
                SM_AT(uint2, scr + S_KRH + o) = make_uint2(h0, h1);
                SM_AT(uint2, scr + S_KRL + o) = make_uint2(l0, l1);
            }
            tc::fence_async_smem();  // Z', V and Kbar are read by the tensor core
            named_bar_sync(bar_id, 128);
            if (lt == 0) {
                mbar_arrive(bar(B_RAW_EMPTY + rs));
                mbar_arrive(bar(B_P2 + n % NP));  // Kbar_n and gamma_n are in the slot
            }

            // A (warps 0, 2) and P (warps 1, 3) partial sums over one channel half each;
            // two bf16 products per entry: Kl, Ql rounded once, Kr as hi + lo
            {
                Frag16 acc;
                chunk_gram_x2<4>(scr + ((lw & 1) ? S_QLH : S_KLH), scr + S_KRH, scr + S_KRL, acc, lane, 4 * (lw >> 1));
                const uint32_t gp = scr + S_GP + xb * 4096 + lw * 1024 + lane * 16;
                SM_AT(float4, gp) = make_float4(acc.c[0][0], acc.c[0][1], acc.c[0][2], acc.c[0][3]);
                SM_AT(float4, gp + 512) = make_float4(acc.c[1][0], acc.c[1][1], acc.c[1][2], acc.c[1][3]);
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(B_GRAM + 2 * ln + xb));
            }

            // cross-chunk products, one per warp (slots n-1, n-2; for n < 2 they read stale
            // slots and are stored but never used):
            //   warp 0: H^w = Kbar_{n-1} (K Gamma)^T,   warp 1: H^q = Kbar_{n-1} (Q Gamma)^T,
            //   warps 2, 3: H'' = Kbar_{n-2} Diag(gamma_{n-1}) [K Gamma ; Q Gamma]^T, one half each
            if (n >= 1 && !wait_bar(bar(B_P2 + (n - 1) % NP), ((n - 1) / NP) & 1, flags)) failed = true;
            {
                const uint32_t prev = slot(n + NP - 1), prev2 = slot(n + NP - 2);
                const uint32_t zt = scr + ((lw & 1) ? S_QG : S_KG) + b_row;
                const uint32_t hx = scr + S_HX + xb * 1536;
                float hc[2][4];
#pragma unroll
                for (int i = 0; i < 2; ++i) hc[i][0] = hc[i][1] = hc[i][2] = hc[i][3] = 0.f;
                if (lw < 2) {
#pragma unroll
                    for (int kb = 0; kb < 8; ++kb) {
                        const uint32_t koff = raw_off(ri + 8 * (mi & 1), 16 * kb + 8 * (mi >> 1));  // A rows j, k = c
                        uint32_t aK[4], bz[4];
                        ldsm_x4(prev + L_KB + koff, aK[0], aK[1], aK[2], aK[3]);
                        ldsm_x4(zt + 32 * kb, bz[0], bz[1], bz[2], bz[3]);
                        mma_f16(hc[0], aK, bz[0], bz[1]);
                        mma_f16(hc[1], aK, bz[2], bz[3]);
                    }
                    if (lw == 0) {
                        SM_AT(uint4, hx + lane * 16) = make_uint4(pack_f16(hc[0][0], hc[0][1]), pack_f16(hc[0][2], hc[0][3]),
                                                                  pack_f16(hc[1][0], hc[1][1]), pack_f16(hc[1][2], hc[1][3]));
                    } else {
                        SM_AT(float4, hx + 512 + lane * 16) = make_float4(hc[0][0], hc[0][1], hc[0][2], hc[0][3]);
                        SM_AT(float4, hx + 1024 + lane * 16) = make_float4(hc[1][0], hc[1][1], hc[1][2], hc[1][3]);
                    }
                } else {
#pragma unroll
                    for (int kb = 0; kb < 8; ++kb) {
                        const uint32_t koff = raw_off(ri + 8 * (mi & 1), 16 * kb + 8 * (mi >> 1));
                        uint32_t aK[4], bz[4];
                        ldsm_x4(prev2 + L_KB + koff, aK[0], aK[1], aK[2], aK[3]);
                        ldsm_x4(zt + 32 * kb, bz[0], bz[1], bz[2], bz[3]);
                        const float2 gl = SM_AT(const float2, prev + L_GAM + (16 * kb + 2 * t) * 4);
                        const float2 gh = SM_AT(const float2, prev + L_GAM + (16 * kb + 8 + 2 * t) * 4);
                        const uint32_t gk0 = pack_f16(gl.x, gl.y), gk1 = pack_f16(gh.x, gh.y);
                        mma_f16(hc[0], aK, hmul2(bz[0], gk0), hmul2(bz[1], gk1));
                        mma_f16(hc[1], aK, hmul2(bz[2], gk0), hmul2(bz[3], gk1));
                    }
                    // H''^T rows n = Z row (16 per warp), columns k = j
                    stsm_x4_t(sl + L_HP + (lw == 2 ? 0 : 512) + stsm_row, pack_f16(hc[0][0], hc[0][1]),
                              pack_f16(hc[0][2], hc[0][3]), pack_f16(hc[1][0], hc[1][1]), pack_f16(hc[1][2], hc[1][3]));
                    tc::fence_async_smem();  // H''^T is read by the tensor core
                }
            }
            __syncwarp();  // one arrival per warp, after all its lanes' stores and reads
            if (lane == 0) {
                mbar_arrive(bar(B_HRDY + 2 * ln + xb));
                if (n >= 2) mbar_arrive(bar(B_PREP_EMPTY + (n - 2) % NP));  // last read of slot n - 2
            }
        }
    } else {
        // ---------------------------------------------------------------- finishers
        // one warp per prep lane: A and P from the lane's partial sums, T' = (I + A)^-1 diag(beta),
        // M = P T', the TM and Phi operands and (H Phi^T)^T, then the slot is handed on.
        const int ln = warp - 14;
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
            const uint32_t gp = scr + S_GP + xb * 4096 + lane * 16, hx = scr + S_HX + xb * 1536;
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
            // TM rows 0..15 = T', Phi rows 0..15 = [-T', 0]
            uint32_t tw[2][2];
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
                const int col = 8 * nt + 2 * t;
                const float2 bc = SM_AT(const float2, bet + col * 4);
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    const int r = g + 8 * hh;
                    const uint32_t w = pack_f16(T.c[nt][2 * hh] * bc.x, T.c[nt][2 * hh + 1] * bc.y);
                    tw[nt][hh] = w;
                    SM_AT(uint32_t, sl + L_TM + cm16(r, col)) = w;
                    SM_AT(float2, sl + L_PHI + cm32(r, col)) = make_float2(-h_lo(w), -h_hi(w));
                    SM_AT(float2, sl + L_PHI + cm32(r, 16 + col)) = make_float2(0.f, 0.f);
                }
            }
            // M = P T' (B operand: transposed 8x8 blocks of T'); s M rounded to f16 once, shared by
            // TM rows 16..31, Phi rows 16..31 = [-s M, s I] and the correction
            uint32_t sm16[2][2];
            {
                uint32_t aP[4];
                frag_as_a(P, aP);
                float m[2][4];
#pragma unroll
                for (int nb = 0; nb < 2; ++nb) {
                    m[nb][0] = m[nb][1] = m[nb][2] = m[nb][3] = 0.f;
                    mma_f16(m[nb], aP, movm_t(tw[nb][0]), movm_t(tw[nb][1]));
                }
#pragma unroll
                for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                    for (int hh = 0; hh < 2; ++hh) {
                        const int r = g + 8 * hh, col = 8 * nt + 2 * t;
                        const uint32_t w = pack_f16(sc * m[nt][2 * hh], sc * m[nt][2 * hh + 1]);
                        sm16[nt][hh] = w;
                        SM_AT(uint32_t, sl + L_TM + cm16(16 + r, col)) = w;
                        SM_AT(float2, sl + L_PHI + cm32(16 + r, col)) = make_float2(-h_lo(w), -h_hi(w));
                        SM_AT(float2, sl + L_PHI + cm32(16 + r, 16 + col)) = make_float2(r == col ? sc : 0.f, r == col + 1 ? sc : 0.f);
                    }
            }
            if (!__all_sync(0xffffffffu, wait_bar(bar(B_HRDY + 2 * ln + xb), xpar, flags))) break;
            // (H Phi^T)^T = [H^w (-T')^T | H^w (-s M)^T + s H^q]: B[k = m][n] = -T'[n][m] and
            // -s M[n][m] come straight from the fragments of T' and s M
            {
                const uint4 ah = SM_AT(const uint4, hx + lane * 16);
                const uint32_t aH[4] = {ah.x, ah.y, ah.z, ah.w};
                const float4 q0 = SM_AT(const float4, hx + 512 + lane * 16), q1 = SM_AT(const float4, hx + 1024 + lane * 16);
                float cf[4][4];
#pragma unroll
                for (int i = 0; i < 4; ++i) cf[i][0] = cf[i][1] = cf[i][2] = cf[i][3] = 0.f;
                mma_f16(cf[0], aH, tw[0][0] ^ NEG2, tw[1][0] ^ NEG2);
                mma_f16(cf[1], aH, tw[0][1] ^ NEG2, tw[1][1] ^ NEG2);
                mma_f16(cf[2], aH, sm16[0][0] ^ NEG2, sm16[1][0] ^ NEG2);
                mma_f16(cf[3], aH, sm16[0][1] ^ NEG2, sm16[1][1] ^ NEG2);
                cf[2][0] = fmaf(sc, q0.x, cf[2][0]); cf[2][1] = fmaf(sc, q0.y, cf[2][1]);
                cf[2][2] = fmaf(sc, q0.z, cf[2][2]); cf[2][3] = fmaf(sc, q0.w, cf[2][3]);
                cf[3][0] = fmaf(sc, q1.x, cf[3][0]); cf[3][1] = fmaf(sc, q1.y, cf[3][1]);
                cf[3][2] = fmaf(sc, q1.z, cf[3][2]); cf[3][3] = fmaf(sc, q1.w, cf[3][3]);
#pragma unroll
                for (int nu = 0; nu < 4; nu += 2)
                    stsm_x4_t(sl + L_CC + nu * 256 + stsm_row, pack_f16(cf[nu][0], cf[nu][1]), pack_f16(cf[nu][2], cf[nu][3]),
                              pack_f16(cf[nu + 1][0], cf[nu + 1][1]), pack_f16(cf[nu + 1][2], cf[nu + 1][3]));
            }
            tc::fence_async_smem();
            if constexpr (DUMP) {
                // the slot is complete here: the lane's Z', V, Kbar, gamma and H''^T (HRDY), and
                // this warp's TM, Phi and (H Phi^T)^T
                if (blockIdx.x == 0 && n < p.dump_chunks) {
                    const uint4 *src = reinterpret_cast<const uint4 *>(smem + (sl - sb));
                    uint4 *dst = reinterpret_cast<uint4 *>(static_cast<uint8_t *>(p.dump) + static_cast<size_t>(n) * SLOT);
                    for (int i = lane; i < SLOT / 16; i += 32) dst[i] = src[i];
                }
            }
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(bar(B_FDONE + 2 * ln + xb));
                mbar_arrive(bar(B_PREP_FULL + n % NP));
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
