// kda_fwd.cu -- fused chunked forward pass of Kimi Delta Attention for GB300
// (sm_103a), and the C ABI declared in include/kda.h.
//
// One CTA owns one (sequence, head) state, or a slice of its V rows when there
// are too few states to fill the machine (the rows of S are independent).
// Warp roles inside the CTA:
//   warp 0       TMA producer: streams the 16-token q/k/v/g tiles of each
//                chunk into a 6-deep shared-memory ring.
//   warps 1..4   two "prep lanes" of two warps each, working on alternate
//                chunks: gate activation in base 2, in-chunk cumsum, the
//                exponent-scaled operand tiles, the 16x16 chunk matrix A and
//                the intra-chunk score matrix P (tf32 MMA), and the
//                unit-lower inverse T = (I + A)^-1 by forward substitution.
//   warps 5..    scan warps, 16 V rows each, holding their rows of the fp32
//                state S in registers across the whole sequence. Per chunk:
//                  Z   = S [K*Gamma ; Q*Gamma]^T              (bf16 MMA)
//                  R   = V^T - Z_k,  E = R (T diag(beta))^T   (fp16 MMA)
//                  O   = scale (Z_q + E P^T)                  (fp16 MMA)
//                  S   = S Diag(gamma) + E Kbar               (fp16 MMA)
//
// The chunk algebra follows from unrolling the gated delta rule over a chunk
// of rows r = 1..L starting from S0: with Gamma_r the in-chunk cumulative
// decay and gamma = Gamma_L, the written rows E satisfy
// (I + A) E = diag(beta) (V - (K*Gamma) S0^T), A[r,j] = beta_r sum_c
// k_r k_j Gamma_r/Gamma_j (j < r); the outputs are
// o_r = scale (S0 (q_r*Gamma_r) + sum_{j<=r} P[r,j] e_j) and the new state is
// S0 Diag(gamma) + E^T Kbar with Kbar_j = k_j * gamma / Gamma_j.
//
// Page references (title -- section):
//  * gate_scale = lower_bound * log2(e) folded on the host and the sigmoid via
//    tanh: "FlashKDA lower_bound Parameter: Controlling Exponentiation
//    Precision ..." -- "Conversion to the Gate Scale Factor".
//  * base-2 exponentials with ex2.approx.ftz.f32: "Base-2 Exponent
//    Optimization in FlashKDA ..." -- "Re-basing the Gate Activation",
//    "Hardware-Accelerated Instruction Selection".
//  * CHUNK = 16, the 16x16 unit-lower inverse: "How FlashKDA's CHUNK Size of
//    16 Improves Numerical Stability Over CHUNK 64" -- "bf16 Dynamic Range and
//    Exponential Terms", "Efficient 16x16 Matrix Inversion".
//  * tensor contract, states, varlen: "FlashKDA Input Tensor Shapes and
//    DTypes ..." -- all sections.
#include <cmath>
#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include "kda.h"
#include "ptx.cuh"

namespace kda {

constexpr int CHUNK = 16;
constexpr int DH = 128;  // K = V = 128

// ---------------------------------------------------------------- shared memory plan
constexpr int NR = 6;                 // raw q/k/v/g ring depth (chunks)
constexpr int NP = 2;                 // prep ring depth = number of prep lanes
constexpr int RAW_TILE = 4096;        // 16 rows x 128 bf16, as two 64-column TMA boxes
constexpr int RAW_BOX = 2048;
constexpr int RAW_STAGE = 4 * RAW_TILE;
constexpr int OFF_Q = 0, OFF_K = RAW_TILE, OFF_V = 2 * RAW_TILE, OFF_G = 3 * RAW_TILE;

constexpr int BZ_LD = 272;            // row pitch (bytes) of 128-wide 16-bit tiles (136 elements)
constexpr int SM_LD = 48;             // row pitch of 16x16 16-bit tiles (24 elements)
constexpr int P_BZ = 0;                           // bf16 [32][136]: K*Gamma rows 0-15, Q*Gamma rows 16-31
constexpr int P_KB = P_BZ + 32 * BZ_LD;           // f16  [16][136]: Kbar
constexpr int P_TT = P_KB + 16 * BZ_LD;           // f16  [16][24]:  T diag(beta)
constexpr int P_PP = P_TT + 16 * SM_LD;           // f16  [16][24]:  P
constexpr int P_GAM = P_PP + 16 * SM_LD;          // f32  [128]:     gamma = Gamma at chunk end
constexpr int PREP_SLOT = P_GAM + DH * 4;

constexpr int F_LD = 528;             // row pitch of fp32 [16][132] tiles
constexpr int A_LD = 80;              // row pitch of fp32 [16][20] tiles
constexpr int S_KL = 0;               // tf32 K * 2^(G - G_mid)
constexpr int S_QL = 16 * F_LD;       // tf32 Q * 2^(G - G_mid)
constexpr int S_KR = 32 * F_LD;       // tf32 K * 2^(G_mid - G)
constexpr int S_AM = 48 * F_LD;       // fp32 A
constexpr int S_BETA = S_AM + 16 * A_LD;
constexpr int SCR = S_BETA + 64;

constexpr int OFF_RAW = 0;
constexpr int OFF_PREP = OFF_RAW + NR * RAW_STAGE;
constexpr int OFF_SCR = OFF_PREP + NP * PREP_SLOT;
constexpr int OFF_BAR = OFF_SCR + NP * SCR;
constexpr int NBAR = 2 * NR + 2 * NP;
constexpr int OFF_FLAGS = OFF_BAR + NBAR * 8;
constexpr int SMEM_USED = OFF_FLAGS + 16;
constexpr int SMEM_ALLOC = SMEM_USED + 1024;  // the ring base is rounded up to 1024 B (128B swizzle)

static_assert(PREP_SLOT % 16 == 0 && SCR % 16 == 0 && OFF_PREP % 1024 == 0, "alignment");
static_assert(OFF_BAR % 8 == 0, "mbarrier alignment");
static_assert(SMEM_ALLOC <= 227 * 1024, "shared memory budget");

constexpr float LOG2E = 1.4426950408889634f;
// tf32 operands are taken from fp32 bit patterns (low mantissa bits ignored).
// Scaling by 1 + 2^-11 first centres that truncation error on zero.
constexpr float TRUNC_COMP = 1.00048828125f;

constexpr int SPIN_LIMIT = 1 << 22;

enum : unsigned { DEVERR_SEQLENS = 1u, DEVERR_TIMEOUT = 2u };
__device__ unsigned int g_dev_error;

struct Params {
    const uint16_t *beta;
    uint16_t *out;
    const float *A_log;
    const float *dt_bias;
    const void *init;
    void *fin;
    const int64_t *cu;
    int init_dtype, fin_dtype;
    int T;        // tokens per batch row (batched mode)
    int H;
    int nseq;     // B, or N in varlen mode
    int vsplit;   // CTAs per state
    int total;    // length of the flattened token axis (B * T)
    float scale;
    float half_gs;  // 0.5 * lower_bound * log2(e)
};

// Bounded wait on an mbarrier phase. Gives up when another role has already
// given up (abort flag) or after SPIN_LIMIT polls, which flags the device
// error word; the caller then leaves its loop so the CTA always terminates.
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile int *abort_flag)
{
#pragma unroll 1
    for (int i = 0; i < SPIN_LIMIT; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if (*abort_flag) return false;
    }
    atomicOr(&g_dev_error, DEVERR_TIMEOUT);
    *abort_flag = 1;
    return false;
}

// Bounded wait that ignores the abort flag (used to drain in-flight copies).
__device__ __forceinline__ void drain_bar(uint32_t bar, uint32_t parity)
{
#pragma unroll 1
    for (int i = 0; i < SPIN_LIMIT; ++i)
        if (mbar_try_wait(bar, parity)) return;
    atomicOr(&g_dev_error, DEVERR_TIMEOUT);
}

struct Span {
    int bos, len;
    bool ok;
};

__device__ __forceinline__ Span seq_span(const Params &p, int seq)
{
    if (p.cu) {
        const long long b = p.cu[seq], e = p.cu[seq + 1];
        if (b < 0 || e < b || e > p.total) return {0, 0, false};
        return {static_cast<int>(b), static_cast<int>(e - b), true};
    }
    return {seq * p.T, p.T, true};
}

// Byte offset of element (row r, channel c) inside a 16x128 bf16 tile loaded
// as two 64-column boxes with the 128-byte swizzle (16-byte chunk index XOR
// row mod 8).
__device__ __forceinline__ uint32_t raw_off(int r, int c)
{
    return (c >> 6) * RAW_BOX + r * 128 + ((((c & 63) >> 3) ^ (r & 7)) << 4) + (c & 7) * 2;
}

__device__ __forceinline__ uint16_t f2bf_bits(float x) { return __bfloat16_as_ushort(__float2bfloat16_rn(x)); }
__device__ __forceinline__ uint16_t f2h_bits(float x) { return __half_as_ushort(__float2half_rn(x)); }

template <int NS>
__global__ void __launch_bounds__(32 * (5 + NS), 1)
    kda_fwd_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                   const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap tg, const Params p)
{
    extern __shared__ uint8_t smem_dyn[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_dyn) + 1023) & ~uintptr_t(1023));
    const uint32_t sb = smem_u32(smem);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int unit = blockIdx.x / p.vsplit, slice = blockIdx.x % p.vsplit;
    const int seq = unit / p.H, h = unit % p.H;
    const Span sp = seq_span(p, seq);

    volatile int *flags = reinterpret_cast<volatile int *>(smem + OFF_FLAGS);
    const uint32_t raw_full = sb + OFF_BAR, raw_empty = raw_full + NR * 8;
    const uint32_t prep_full = raw_empty + NR * 8, prep_empty = prep_full + NP * 8;

    if (threadIdx.x == 0) {
        for (int i = 0; i < NR; ++i) {
            mbar_init(raw_full + 8 * i, 1);
            mbar_init(raw_empty + 8 * i, 1 + NS);
        }
        for (int i = 0; i < NP; ++i) {
            mbar_init(prep_full + 8 * i, 1);
            mbar_init(prep_empty + 8 * i, NS);
        }
        flags[0] = 0;
        fence_mbar_init();
        if (p.cu && blockIdx.x == 0 && (p.cu[0] != 0 || p.cu[p.nseq] != p.total))
            atomicOr(&g_dev_error, DEVERR_SEQLENS);
        if (!sp.ok && slice == 0 && h == 0) atomicOr(&g_dev_error, DEVERR_SEQLENS);
    }
    __syncthreads();
    if (!sp.ok) return;  // CTA-uniform
    const int nch = (sp.len + CHUNK - 1) / CHUNK;

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            tma_prefetch_desc(&tq);
            tma_prefetch_desc(&tk);
            tma_prefetch_desc(&tv);
            tma_prefetch_desc(&tg);
            int n = 0;
            for (; n < nch; ++n) {
                const int s = n % NR;
                const uint32_t ph = (n / NR) & 1;
                if (!wait_bar(raw_empty + 8 * s, ph ^ 1, flags)) break;
                const uint32_t fb = raw_full + 8 * s;
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
            // never leave while copies this thread issued may still be landing
            for (int m = (n > NR ? n - NR : 0); m < n; ++m) drain_bar(raw_full + 8 * (m % NR), (m / NR) & 1);
        }
        return;
    }

    if (warp < 5) {
        // ------------------------------------------------------------ prep lanes
        const int ln = (warp - 1) >> 1;            // prep lane 0 or 1
        const int lt = threadIdx.x - 32 - 64 * ln;  // 0..63
        const int lw = lt >> 5;                     // warp within the lane
        const uint32_t bar_id = 1 + ln;
        const uint32_t scr = sb + OFF_SCR + ln * SCR;
        const uint32_t pslot = sb + OFF_PREP + ln * PREP_SLOT;
        const int c0 = 2 * lt;                      // this thread's channels c0, c0 + 1
        float a_h = 1.f, bias0 = 0.f, bias1 = 0.f;
        if (p.A_log) a_h = ex2_approx(__ldg(p.A_log + h) * LOG2E);
        if (p.dt_bias) {
            bias0 = __ldg(p.dt_bias + h * DH + c0);
            bias1 = __ldg(p.dt_bias + h * DH + c0 + 1);
        }
        const float hs = p.half_gs;
        const int g = lane >> 2, t = lane & 3;

        for (int n = ln; n < nch; n += NP) {
            bool failed = false;  // this thread's waits gave up; OR-reduced at the end of the chunk
            const int rs = n % NR;
            const uint32_t rph = (n / NR) & 1, pph = (n / NP) & 1;
            const int tok0 = sp.bos + n * CHUNK;
            const int Lv = min(CHUNK, sp.len - n * CHUNK);
            float blogit = 0.f;
            if (lw == 1 && lane < Lv)
                blogit = __uint_as_float(static_cast<uint32_t>(__ldg(p.beta + static_cast<size_t>(tok0 + lane) * p.H + h)) << 16);
            if (!wait_bar(raw_full + 8 * rs, rph, flags)) failed = true;
            const uint32_t raw = sb + OFF_RAW + rs * RAW_STAGE;

            // gate in log2 units and its inclusive in-chunk cumsum
            float G0[CHUNK], G1[CHUNK];
            {
                float acc0 = 0.f, acc1 = 0.f;
#pragma unroll
                for (int r = 0; r < CHUNK; ++r) {
                    const uint32_t gw = lds32(raw + OFF_G + raw_off(r, c0));
                    const float x0 = a_h * (bf16_lo(gw) + bias0), x1 = a_h * (bf16_hi(gw) + bias1);
                    // gate_scale * sigmoid(x) = hs + hs * tanh(x / 2)
                    const float ga0 = fmaf(hs, tanh_approx(0.5f * x0), hs);
                    const float ga1 = fmaf(hs, tanh_approx(0.5f * x1), hs);
                    acc0 += (r < Lv) ? ga0 : 0.f;
                    acc1 += (r < Lv) ? ga1 : 0.f;
                    G0[r] = acc0;
                    G1[r] = acc1;
                }
            }
            if (!wait_bar(prep_empty + 8 * ln, pph ^ 1, flags)) failed = true;

            const float Gm0 = G0[7], Gm1 = G1[7];  // mid-chunk reference halves the exponent range
            const float sm0 = ex2_approx(-Gm0) * TRUNC_COMP, sm1 = ex2_approx(-Gm1) * TRUNC_COMP;
            const float se0 = ex2_approx(G0[15] - Gm0), se1 = ex2_approx(G1[15] - Gm1);
            stsf2(pslot + P_GAM + c0 * 4, ex2_approx(G0[15]), ex2_approx(G1[15]));
#pragma unroll
            for (int r = 0; r < CHUNK; ++r) {
                const uint32_t kw = lds32(raw + OFF_K + raw_off(r, c0));
                const uint32_t qw = lds32(raw + OFF_Q + raw_off(r, c0));
                const bool live = r < Lv;
                const float k0 = live ? bf16_lo(kw) : 0.f, k1 = live ? bf16_hi(kw) : 0.f;
                const float q0 = live ? bf16_lo(qw) : 0.f, q1 = live ? bf16_hi(qw) : 0.f;
                const float gm0 = ex2_approx(G0[r]), gm1 = ex2_approx(G1[r]);            // Gamma_r
                const float f0 = ex2_approx(Gm0 - G0[r]), f1 = ex2_approx(Gm1 - G1[r]);  // 2^(G_mid - G_r)
                sts32(pslot + P_BZ + r * BZ_LD + c0 * 2, pack_bf16(k0 * gm0, k1 * gm1));
                sts32(pslot + P_BZ + (16 + r) * BZ_LD + c0 * 2, pack_bf16(q0 * gm0, q1 * gm1));
                sts32(pslot + P_KB + r * BZ_LD + c0 * 2, pack_f16(k0 * f0 * se0, k1 * f1 * se1));
                const float u0 = gm0 * sm0, u1 = gm1 * sm1;                              // 2^(G_r - G_mid)
                stsf2(scr + S_KL + r * F_LD + c0 * 4, k0 * u0, k1 * u1);
                stsf2(scr + S_QL + r * F_LD + c0 * 4, q0 * u0, q1 * u1);
                stsf2(scr + S_KR + r * F_LD + c0 * 4, k0 * f0 * TRUNC_COMP, k1 * f1 * TRUNC_COMP);
            }
            if (lw == 1 && lane < CHUNK)
                stsf(scr + S_BETA + lane * 4, lane < Lv ? fmaf(0.5f, tanh_approx(0.5f * blogit), 0.5f) : 0.f);
            named_bar_sync(bar_id, 64);
            if (lt == 0) mbar_arrive(raw_empty + 8 * rs);

            // A (warp 0) and P (warp 1): [K|Q] * 2^(G - G_mid) times (K * 2^(G_mid - G))^T, tf32
            {
                const uint32_t X = scr + (lw == 0 ? S_KL : S_QL);
                float acc[2][4];
#pragma unroll
                for (int i = 0; i < 2; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
#pragma unroll
                for (int ks = 0; ks < 16; ++ks) {
                    const int cc = 8 * ks + t;
                    const float a0 = ldsf(X + g * F_LD + cc * 4), a1 = ldsf(X + (g + 8) * F_LD + cc * 4);
                    const float a2 = ldsf(X + g * F_LD + (cc + 4) * 4), a3 = ldsf(X + (g + 8) * F_LD + (cc + 4) * 4);
#pragma unroll
                    for (int nt = 0; nt < 2; ++nt) {
                        const float b0 = ldsf(scr + S_KR + (8 * nt + g) * F_LD + cc * 4);
                        const float b1 = ldsf(scr + S_KR + (8 * nt + g) * F_LD + (cc + 4) * 4);
                        mma_tf32(acc[nt], a0, a1, a2, a3, b0, b1);
                    }
                }
                if (lw == 0) {
#pragma unroll
                    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            const int r = g + 8 * (i >> 1), j = 8 * nt + 2 * t + (i & 1);
                            const float br = ldsf(scr + S_BETA + r * 4);
                            stsf(scr + S_AM + r * A_LD + j * 4, j < r ? acc[nt][i] * br : 0.f);
                        }
                } else {
#pragma unroll
                    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                        for (int hh = 0; hh < 2; ++hh) {
                            const int r = g + 8 * hh, j = 8 * nt + 2 * t;
                            const float v0 = j <= r ? acc[nt][2 * hh] : 0.f;
                            const float v1 = j + 1 <= r ? acc[nt][2 * hh + 1] : 0.f;
                            sts32(pslot + P_PP + r * SM_LD + j * 2, pack_f16(v0, v1));
                        }
                }
            }
            named_bar_sync(bar_id, 64);

            // T = (I + A)^-1 by forward substitution; lane c (mod 16) owns column c
            if (lw == 0) {
                const int c = lane & 15;
                float tc[CHUNK];
#pragma unroll
                for (int r = 0; r < CHUNK; ++r) {
                    float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
#pragma unroll
                    for (int j4 = 0; j4 < r; j4 += 4) {
                        const float4 a = ldsf4(scr + S_AM + r * A_LD + j4 * 4);
                        if (j4 + 0 < r) s0 = fmaf(a.x, tc[j4 + 0], s0);
                        if (j4 + 1 < r) s1 = fmaf(a.y, tc[j4 + 1], s1);
                        if (j4 + 2 < r) s2 = fmaf(a.z, tc[j4 + 2], s2);
                        if (j4 + 3 < r) s3 = fmaf(a.w, tc[j4 + 3], s3);
                    }
                    tc[r] = (r == c ? 1.f : 0.f) - ((s0 + s1) + (s2 + s3));
                }
                const float bc = ldsf(scr + S_BETA + c * 4);
#pragma unroll
                for (int j = 0; j < CHUNK; ++j)
                    if ((j >> 3) == (lane >> 4)) sts16(pslot + P_TT + j * SM_LD + c * 2, f2h_bits(tc[j] * bc));
            }
            const bool stop = named_bar_or(bar_id, 64, failed);
            if (lt == 0) mbar_arrive(prep_full + 8 * ln);
            if (stop) break;
        }
        return;
    }

    // ---------------------------------------------------------------- scan warps
    const int sw = warp - 5;
    const int g = lane >> 2, t = lane & 3;
    const int vr0 = slice * (16 * NS) + 16 * sw;
    const size_t st_base = (static_cast<size_t>(seq) * p.H + h) * (DH * DH);
    float S[16][4];
#pragma unroll
    for (int nt = 0; nt < 16; ++nt)
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            const size_t e = st_base + static_cast<size_t>(vr0 + g + 8 * hh) * DH + 8 * nt + 2 * t;
            float x = 0.f, y = 0.f;
            if (p.init) {
                if (p.init_dtype == KDA_DTYPE_FP32) {
                    const float2 w = *reinterpret_cast<const float2 *>(static_cast<const float *>(p.init) + e);
                    x = w.x;
                    y = w.y;
                } else {
                    const uint32_t w = *reinterpret_cast<const uint32_t *>(static_cast<const uint16_t *>(p.init) + e);
                    x = bf16_lo(w);
                    y = bf16_hi(w);
                }
            }
            S[nt][2 * hh] = x;
            S[nt][2 * hh + 1] = y;
        }

    const int mi = lane >> 3, ri = lane & 7;
    for (int n = 0; n < nch; ++n) {
        const int ps = n % NP, rs = n % NR;
        const uint32_t pph = (n / NP) & 1, rph = (n / NR) & 1;
        bool ok = wait_bar(prep_full + 8 * ps, pph, flags);
        ok = ok && wait_bar(raw_full + 8 * rs, rph, flags);
        if (!__all_sync(0xffffffffu, ok)) break;
        const int tok0 = sp.bos + n * CHUNK;
        const int Lv = min(CHUNK, sp.len - n * CHUNK);
        const uint32_t pb = sb + OFF_PREP + ps * PREP_SLOT;
        const uint32_t vt = sb + OFF_RAW + rs * RAW_STAGE + OFF_V;

        // Z = S [K*Gamma ; Q*Gamma]^T  (16 rows x 32 columns per warp)
        float z[4][4];
#pragma unroll
        for (int i = 0; i < 4; ++i) z[i][0] = z[i][1] = z[i][2] = z[i][3] = 0.f;
        const uint32_t bz = pb + P_BZ + (ri + 8 * (mi >> 1)) * BZ_LD + 16 * (mi & 1);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
            const uint32_t a[4] = {pack_bf16(S[2 * kk][0], S[2 * kk][1]), pack_bf16(S[2 * kk][2], S[2 * kk][3]),
                                   pack_bf16(S[2 * kk + 1][0], S[2 * kk + 1][1]),
                                   pack_bf16(S[2 * kk + 1][2], S[2 * kk + 1][3])};
            uint32_t b0, b1, b2, b3;
            ldsm_x4(bz + kk * 32, b0, b1, b2, b3);
            mma_bf16(z[0], a, b0, b1);
            mma_bf16(z[1], a, b2, b3);
            ldsm_x4(bz + 16 * BZ_LD + kk * 32, b0, b1, b2, b3);
            mma_bf16(z[2], a, b0, b1);
            mma_bf16(z[3], a, b2, b3);
        }

        // R = V^T - Z_k (rows past the chunk's end are zero)
        float R[2][4];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int j = 8 * nt + 2 * t + (i & 1), vr = vr0 + g + 8 * (i >> 1);
                const float vv = j < Lv ? __uint_as_float(static_cast<uint32_t>(lds16(vt + raw_off(j, vr))) << 16) : 0.f;
                R[nt][i] = vv - z[nt][i];
            }
        __syncwarp();
        if (lane == 0) mbar_arrive(raw_empty + 8 * rs);

        // E = R (T diag(beta))^T
        const uint32_t ra[4] = {pack_f16(R[0][0], R[0][1]), pack_f16(R[0][2], R[0][3]), pack_f16(R[1][0], R[1][1]),
                                pack_f16(R[1][2], R[1][3])};
        float e[2][4];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
            e[nt][0] = e[nt][1] = e[nt][2] = e[nt][3] = 0.f;
            const uint32_t row = pb + P_TT + (8 * nt + g) * SM_LD + 4 * t;
            mma_f16(e[nt], ra, lds32(row), lds32(row + 16));
        }
        const uint32_t ea[4] = {pack_f16(e[0][0], e[0][1]), pack_f16(e[0][2], e[0][3]), pack_f16(e[1][0], e[1][1]),
                                pack_f16(e[1][2], e[1][3])};

        // O = scale (Z_q + E P^T)
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
            const uint32_t row = pb + P_PP + (8 * nt + g) * SM_LD + 4 * t;
            mma_f16(z[2 + nt], ea, lds32(row), lds32(row + 16));
        }
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int r = 8 * nt + 2 * t + (i & 1), vr = vr0 + g + 8 * (i >> 1);
                if (r < Lv) p.out[(static_cast<size_t>(tok0 + r) * p.H + h) * DH + vr] = f2bf_bits(p.scale * z[2 + nt][i]);
            }

        // S = S Diag(gamma) + E Kbar
#pragma unroll
        for (int nt = 0; nt < 16; ++nt) {
            const float2 gm = ldsf2(pb + P_GAM + (8 * nt + 2 * t) * 4);
            S[nt][0] *= gm.x;
            S[nt][1] *= gm.y;
            S[nt][2] *= gm.x;
            S[nt][3] *= gm.y;
        }
        const uint32_t kb = pb + P_KB + (ri + 8 * (mi & 1)) * BZ_LD + 16 * (mi >> 1);
#pragma unroll
        for (int m = 0; m < 8; ++m) {
            uint32_t b0, b1, b2, b3;
            ldsm_x4_t(kb + m * 32, b0, b1, b2, b3);
            mma_f16(S[2 * m], ea, b0, b1);
            mma_f16(S[2 * m + 1], ea, b2, b3);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(prep_empty + 8 * ps);
    }

    if (p.fin) {
#pragma unroll
        for (int nt = 0; nt < 16; ++nt)
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                const size_t e = st_base + static_cast<size_t>(vr0 + g + 8 * hh) * DH + 8 * nt + 2 * t;
                if (p.fin_dtype == KDA_DTYPE_FP32)
                    *reinterpret_cast<float2 *>(static_cast<float *>(p.fin) + e) = make_float2(S[nt][2 * hh], S[nt][2 * hh + 1]);
                else
                    *reinterpret_cast<uint32_t *>(static_cast<uint16_t *>(p.fin) + e) = pack_bf16(S[nt][2 * hh], S[nt][2 * hh + 1]);
            }
    }
}

// ==================================================================== host side

static thread_local std::string t_last_error;

static kda_status fail(kda_status s, const char *fmt, ...) __attribute__((format(printf, 2, 3)));
static kda_status fail(kda_status s, const char *fmt, ...)
{
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    t_last_error = buf;
    return s;
}

static PFN_cuTensorMapEncodeTiled_v12000 get_encode()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    });
    return fn;
}

// [tokens, H, 128] bf16 tensor, boxes of 64 channels x 1 head x 16 tokens, 128-byte swizzle.
static bool make_map(CUtensorMap *m, const void *base, int64_t tokens, int64_t H)
{
    auto enc = get_encode();
    if (!enc) return false;
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(DH), static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(tokens)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(DH * 2), static_cast<cuuint64_t>(H * DH * 2)};
    cuuint32_t box[3] = {64, 1, CHUNK};
    cuuint32_t estr[3] = {1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

static void plan(int64_t units, int num_sms, int *vsplit, int64_t *grid)
{
    int vs = 1;
    for (int cand = 8; cand > 1; cand >>= 1)
        if (units * cand <= num_sms) {
            vs = cand;
            break;
        }
    *vsplit = vs;
    *grid = units * vs;
}

template <int NS>
static cudaError_t launch(int64_t grid, cudaStream_t s, const CUtensorMap &q, const CUtensorMap &k,
                          const CUtensorMap &v, const CUtensorMap &g, const Params &p)
{
    static thread_local int configured_dev = -1;
    int dev = 0;
    cudaGetDevice(&dev);
    if (configured_dev != dev) {
        cudaError_t e = cudaFuncSetAttribute(kda_fwd_kernel<NS>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_ALLOC);
        if (e != cudaSuccess) return e;
        configured_dev = dev;
    }
    kda_fwd_kernel<NS><<<static_cast<unsigned>(grid), 32 * (5 + NS), SMEM_ALLOC, s>>>(q, k, v, g, p);
    return cudaGetLastError();
}

static bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

}  // namespace kda

using namespace kda;

extern "C" {

KDA_API int kda_version(void) { return 100; }

KDA_API const char *kda_last_error(void) { return t_last_error.c_str(); }

KDA_API float kda_gate_scale(float lower_bound)
{
    return static_cast<float>(static_cast<double>(lower_bound) * 1.4426950408889634);
}

KDA_API kda_status kda_plan(int64_t units, int num_sms, int *v_split, int64_t *grid)
{
    if (!v_split || !grid) return fail(KDA_ERR_NULL, "kda_plan: null output pointer");
    if (units < 0 || num_sms < 1) return fail(KDA_ERR_SHAPE, "kda_plan: units=%lld num_sms=%d", (long long)units, num_sms);
    plan(units, num_sms, v_split, grid);
    return KDA_OK;
}

KDA_API kda_status kda_fwd(const void *q, const void *k, const void *v, const void *g, const void *beta, float scale,
                           void *out, const float *A_log, const float *dt_bias, float lower_bound,
                           const void *initial_state, kda_dtype initial_dtype, void *final_state,
                           kda_dtype final_dtype, const int64_t *cu_seqlens, int64_t N, int64_t B, int64_t T,
                           int64_t H, int64_t K, int64_t V, void *stream)
{
    t_last_error.clear();
    if (K != DH || V != DH) return fail(KDA_ERR_SHAPE, "K and V must be 128 (got K=%lld V=%lld)", (long long)K, (long long)V);
    if (B < 1 || T < 0 || H < 1) return fail(KDA_ERR_SHAPE, "bad sizes B=%lld T=%lld H=%lld", (long long)B, (long long)T, (long long)H);
    if (cu_seqlens && (B != 1 || N < 1))
        return fail(KDA_ERR_SHAPE, "varlen mode needs B == 1 and N >= 1 (B=%lld N=%lld)", (long long)B, (long long)N);
    const int64_t total = B * T;
    if (total > (int64_t(1) << 31) - 2 * CHUNK || H > (1 << 20))
        return fail(KDA_ERR_SHAPE, "problem too large (tokens=%lld H=%lld)", (long long)total, (long long)H);
    const int64_t nseq = cu_seqlens ? N : B;
    if (nseq * H > (int64_t(1) << 28)) return fail(KDA_ERR_SHAPE, "too many (sequence, head) pairs");
    if (total > 0 && (!q || !k || !v || !g || !beta || !out)) return fail(KDA_ERR_NULL, "q, k, v, g, beta and out are required");
    if (!std::isfinite(lower_bound) || lower_bound < -5.f || lower_bound > 0.f)
        return fail(KDA_ERR_RANGE, "lower_bound must lie in [-5, 0] (got %g)", (double)lower_bound);
    if (!std::isfinite(scale)) return fail(KDA_ERR_RANGE, "scale must be finite");
    auto dt_ok = [](const void *ptr, kda_dtype d) {
        return ptr ? (d == KDA_DTYPE_BF16 || d == KDA_DTYPE_FP32) : d == KDA_DTYPE_NONE;
    };
    if (!dt_ok(initial_state, initial_dtype) || !dt_ok(final_state, final_dtype))
        return fail(KDA_ERR_DTYPE, "state dtype codes must be BF16/FP32 for a given buffer and NONE for an absent one");
    const int64_t st_bytes = nseq * H * DH * DH * (initial_dtype == KDA_DTYPE_FP32 ? 4 : 2);
    if (initial_state && final_state) {
        if (initial_dtype != final_dtype) return fail(KDA_ERR_STATE_MISMATCH, "final_state must match initial_state's dtype");
        const uintptr_t a = reinterpret_cast<uintptr_t>(initial_state), b = reinterpret_cast<uintptr_t>(final_state);
        if (a != b && a < b + st_bytes && b < a + st_bytes)
            return fail(KDA_ERR_STATE_MISMATCH, "initial_state and final_state overlap partially");
    }
    if (total > 0) {
        const void *need16[] = {q, k, v, g, out};
        for (const void *ptr : need16)
            if (!aligned(ptr, 16)) return fail(KDA_ERR_ALIGN, "q, k, v, g and out must be 16-byte aligned");
        if (!aligned(beta, 2)) return fail(KDA_ERR_ALIGN, "beta must be 2-byte aligned");
    }
    if ((initial_state && !aligned(initial_state, 16)) || (final_state && !aligned(final_state, 16)))
        return fail(KDA_ERR_ALIGN, "state buffers must be 16-byte aligned");
    if ((A_log && !aligned(A_log, 4)) || (dt_bias && !aligned(dt_bias, 4)) || (cu_seqlens && !aligned(cu_seqlens, 8)))
        return fail(KDA_ERR_ALIGN, "A_log, dt_bias and cu_seqlens must be naturally aligned");

    CUtensorMap mq, mk, mv, mg;
    std::memset(&mq, 0, sizeof mq);
    std::memset(&mk, 0, sizeof mk);
    std::memset(&mv, 0, sizeof mv);
    std::memset(&mg, 0, sizeof mg);
    if (total > 0) {
        if (!make_map(&mq, q, total, H) || !make_map(&mk, k, total, H) || !make_map(&mv, v, total, H) ||
            !make_map(&mg, g, total, H))
            return fail(KDA_ERR_LAUNCH, "cuTensorMapEncodeTiled failed (driver entry point unavailable or bad geometry)");
    }
    int dev = 0, nsm = 0;
    cudaError_t ce = cudaGetDevice(&dev);
    if (ce == cudaSuccess) ce = cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
    if (ce != cudaSuccess) return fail(KDA_ERR_LAUNCH, "CUDA device query failed: %s", cudaGetErrorString(ce));

    Params p;
    p.beta = static_cast<const uint16_t *>(beta);
    p.out = static_cast<uint16_t *>(out);
    p.A_log = A_log;
    p.dt_bias = dt_bias;
    p.init = initial_state;
    p.fin = final_state;
    p.cu = cu_seqlens;
    p.init_dtype = initial_dtype;
    p.fin_dtype = final_dtype;
    p.T = static_cast<int>(T);
    p.H = static_cast<int>(H);
    p.nseq = static_cast<int>(nseq);
    p.total = static_cast<int>(total);
    p.scale = scale;
    p.half_gs = 0.5f * kda_gate_scale(lower_bound);
    int vs;
    int64_t grid;
    plan(nseq * H, nsm, &vs, &grid);
    p.vsplit = vs;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    switch (vs) {
        case 1: ce = launch<8>(grid, s, mq, mk, mv, mg, p); break;
        case 2: ce = launch<4>(grid, s, mq, mk, mv, mg, p); break;
        case 4: ce = launch<2>(grid, s, mq, mk, mv, mg, p); break;
        default: ce = launch<1>(grid, s, mq, mk, mv, mg, p); break;
    }
    if (ce != cudaSuccess) return fail(KDA_ERR_LAUNCH, "kernel launch failed: %s", cudaGetErrorString(ce));
    return KDA_OK;
}

KDA_API kda_status kda_check_device_status(void *stream)
{
    cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return fail(KDA_ERR_LAUNCH, "stream synchronize failed: %s", cudaGetErrorString(e));
    unsigned int word = 0, zero = 0;
    e = cudaMemcpyFromSymbol(&word, g_dev_error, sizeof word);
    if (e == cudaSuccess && word) e = cudaMemcpyToSymbol(g_dev_error, &zero, sizeof zero);
    if (e != cudaSuccess) return fail(KDA_ERR_LAUNCH, "reading the device status failed: %s", cudaGetErrorString(e));
    if (word)
        return fail(KDA_ERR_DEVICE, "device error word 0x%x:%s%s", word, (word & DEVERR_SEQLENS) ? " bad cu_seqlens" : "",
                    (word & DEVERR_TIMEOUT) ? " pipeline wait timed out" : "");
    return KDA_OK;
}

KDA_API kda_status kda_fwd_host(const void *q, const void *k, const void *v, const void *g, const void *beta,
                                float scale, void *out, const float *A_log, const float *dt_bias, float lower_bound,
                                const void *initial_state, kda_dtype initial_dtype, void *final_state,
                                kda_dtype final_dtype, const int64_t *cu_seqlens, int64_t N, int64_t B, int64_t T,
                                int64_t H, int64_t K, int64_t V, void *stream)
{
    t_last_error.clear();
    if (K != DH || V != DH || B < 1 || T < 0 || H < 1 || (cu_seqlens && N < 1))
        return fail(KDA_ERR_SHAPE, "bad sizes");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int64_t total = B * T, nseq = cu_seqlens ? N : B;
    const size_t act = static_cast<size_t>(total) * H * DH * 2, bet = static_cast<size_t>(total) * H * 2;
    const size_t st_in = initial_state ? static_cast<size_t>(nseq) * H * DH * DH * (initial_dtype == KDA_DTYPE_FP32 ? 4 : 2) : 0;
    const size_t st_out = final_state ? static_cast<size_t>(nseq) * H * DH * DH * (final_dtype == KDA_DTYPE_FP32 ? 4 : 2) : 0;
    const size_t cub = cu_seqlens ? static_cast<size_t>(N + 1) * 8 : 0;
    const size_t al = A_log ? static_cast<size_t>(H) * 4 : 0, db = dt_bias ? static_cast<size_t>(H) * DH * 4 : 0;
    auto up = [](size_t x) { return (x + 255) & ~size_t(255); };
    const size_t sizes[] = {act, act, act, act, bet, act, al, db, st_in, st_out, cub};
    size_t off[11], tot = 0;
    for (int i = 0; i < 11; ++i) {
        off[i] = tot;
        tot += up(sizes[i]);
    }
    uint8_t *d = nullptr;
    cudaError_t e = cudaMallocAsync(reinterpret_cast<void **>(&d), tot ? tot : 256, s);
    if (e != cudaSuccess) return fail(KDA_ERR_LAUNCH, "device staging allocation failed: %s", cudaGetErrorString(e));
    const void *src[] = {q, k, v, g, beta, nullptr, A_log, dt_bias, initial_state, nullptr, cu_seqlens};
    for (int i = 0; i < 11 && e == cudaSuccess; ++i)
        if (src[i] && sizes[i]) e = cudaMemcpyAsync(d + off[i], src[i], sizes[i], cudaMemcpyHostToDevice, s);
    kda_status st = KDA_ERR_LAUNCH;
    if (e == cudaSuccess) {
        st = kda_fwd(d + off[0], d + off[1], d + off[2], d + off[3], d + off[4], scale, d + off[5],
                     A_log ? reinterpret_cast<const float *>(d + off[6]) : nullptr,
                     dt_bias ? reinterpret_cast<const float *>(d + off[7]) : nullptr, lower_bound,
                     initial_state ? d + off[8] : nullptr, initial_dtype, final_state ? d + off[9] : nullptr,
                     final_dtype, cu_seqlens ? reinterpret_cast<const int64_t *>(d + off[10]) : nullptr, N, B, T, H, K,
                     V, stream);
        if (st == KDA_OK) {
            if (act) e = cudaMemcpyAsync(out, d + off[5], act, cudaMemcpyDeviceToHost, s);
            if (e == cudaSuccess && st_out) e = cudaMemcpyAsync(final_state, d + off[9], st_out, cudaMemcpyDeviceToHost, s);
            if (e != cudaSuccess) st = fail(KDA_ERR_LAUNCH, "device-to-host copy failed: %s", cudaGetErrorString(e));
        }
    } else {
        fail(KDA_ERR_LAUNCH, "host-to-device copy failed: %s", cudaGetErrorString(e));
    }
    cudaFreeAsync(d, s);
    cudaError_t se = cudaStreamSynchronize(s);
    if (st == KDA_OK && se != cudaSuccess) st = fail(KDA_ERR_LAUNCH, "stream synchronize failed: %s", cudaGetErrorString(se));
    return st;
}

}  // extern "C"
