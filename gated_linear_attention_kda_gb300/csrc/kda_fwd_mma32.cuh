// kda_fwd_mma32.cuh -- the warp-MMA KDA forward kernel with 32-token chunks:
// the chunk-size ablation of the 16-token kernels (KDA_FLAG_CHUNK32).
//
// "How FlashKDA's CHUNK Size of 16 Improves Numerical Stability Over CHUNK
// 64" -- "bf16 Dynamic Range and Exponential Terms", "Why CHUNK Size
// Determines Numerical Stability": the exponent factors K 2^{G - G_ref} and
// K 2^{G_ref - G} of the chunk matrix must stay inside bf16's range. With the
// reference at the chunk's middle (the cumulative gate after token 15) a
// 32-token chunk spans at most 16 |lower_bound| log2(e) <= 115.4 bits either
// way, as a 16-token chunk does with its reference at the start, so the same
// bf16 hi/lo chunk products hold. "Efficient 16x16 Matrix Inversion": the
// 32x32 unit-lower inverse is built from two 16x16 Neumann inverses,
//   (I + A)^-1 = [[T00, 0], [-T11 A10 T00, T11]],  T_ii = (I + A_ii)^-1.
//
// Roles (32 (9 + NS) threads):
//   warp 0      TMA producer: q/k/g tiles of each chunk into a 2-stage ring
//               (freed by the prep lane after its element-wise pass), v tiles
//               into a 3-stage ring (freed by the scan warps).
//   warps 1-8   two prep lanes of four warps, alternate chunks. A lane's warps
//               0-1 take tokens 0-15, warps 2-3 tokens 16-31 (two channels per
//               thread); the two halves exchange their gate sums through
//               shared memory. Chunk products: six 16x16 blocks (A00, A10, A11,
//               P00, P10, P11), 1.5 blocks per warp; inverse blocks on warps 0-1.
//   warps 9..   NS scan warps, 16 V rows each, fp32 state in registers:
//                 Z = S [K*Gamma ; Q*Gamma]^T (16 x 64), R = V^T - Z_k,
//                 E = R (T diag(beta))^T, O = scale (Z_q + E P^T),
//                 S = S Diag(gamma) + E Kbar (k = 32).
#pragma once
#include "kda_chunk.cuh"
#include "kda_common.cuh"

namespace kda {
namespace v32 {

constexpr int C2 = 32;                // tokens per chunk
constexpr int NP = 2;                 // prep lanes = prep slots
constexpr int NRQ = 2;                // q/k/g ring depth
constexpr int NRV = 3;                // v ring depth
constexpr int LANE_THREADS = 128;

constexpr int QKG_HALF = 3 * RAW_TILE;              // q, k, g tiles of 16 tokens
constexpr int QKG_STAGE = 2 * QKG_HALF;
constexpr int Q_OFF = 0, K_OFF = RAW_TILE, G_OFF = 2 * RAW_TILE;
constexpr int V_STAGE = 2 * RAW_TILE;

constexpr int LD = 272;               // row pitch (bytes) of 128-wide 16-bit tiles
constexpr int LD32 = 80;              // row pitch of 32x32 16-bit tiles (40 elements)
constexpr int P_BZ = 0;                           // bf16 [64][136]: K*Gamma rows 0-31, Q*Gamma rows 32-63
constexpr int P_KB = P_BZ + 64 * LD;              // f16  [32][136]: Kbar
constexpr int P_TT = P_KB + 32 * LD;              // f16  [32][40]:  T diag(beta) (lower)
constexpr int P_PP = P_TT + 32 * LD32;            // f16  [32][40]:  P (lower, with the diagonal)
constexpr int P_GAM = P_PP + 32 * LD32;           // f32  [128]:     gamma
constexpr int SLOT = P_GAM + DH * 4;

constexpr int S_KLH = 0;                          // bf16 K 2^(G - G_mid)
constexpr int S_QLH = S_KLH + 32 * LD;            // bf16 Q 2^(G - G_mid)
constexpr int S_KRH = S_QLH + 32 * LD;            // bf16 hi / lo of K 2^(G_mid - G)
constexpr int S_KRL = S_KRH + 32 * LD;
constexpr int S_BETA = S_KRL + 32 * LD;           // f32 [32]
constexpr int S_GX = S_BETA + 128;                // f32 [2 halves][128]: in-half gate sums
constexpr int S_XCH = S_GX + 1024;                // three 16x16 fp32 fragments (32 lanes x 8)
constexpr int SCR = S_XCH + 3 * 1024;

constexpr int OFF_QKG = 0;
constexpr int OFF_V = OFF_QKG + NRQ * QKG_STAGE;
constexpr int OFF_SLOT = OFF_V + NRV * V_STAGE;
constexpr int OFF_SCR = OFF_SLOT + NP * SLOT;
constexpr int OFF_BAR = OFF_SCR + NP * SCR;
constexpr int NBAR = 2 * NRQ + 2 * NRV + 2 * NP;
constexpr int OFF_FLAGS = OFF_BAR + NBAR * 8;
constexpr int SMEM_USED = OFF_FLAGS + 16;
constexpr int SMEM_ALLOC = SMEM_USED + 1024;  // the ring base is rounded up to 1024 B (128B swizzle)

static_assert(QKG_STAGE % 1024 == 0 && V_STAGE % 1024 == 0 && OFF_V % 1024 == 0, "swizzled TMA boxes need 1024-B alignment");
static_assert(SLOT % 16 == 0 && SCR % 16 == 0 && OFF_SLOT % 16 == 0 && OFF_SCR % 16 == 0, "alignment");
static_assert(OFF_BAR % 8 == 0, "mbarrier alignment");
static_assert(SMEM_ALLOC <= 227 * 1024, "shared memory budget");

// Fragment (Frag16) element (row g + 8 (i >> 1), col 8 nt + 2 t + (i & 1)) of the 16x16 block.
__device__ __forceinline__ void frag_store(uint8_t *p, const Frag16 &f, int lane)
{
    if (!smem_ok(smem_u32(p + lane * 32), 32)) return;
    float4 *q = reinterpret_cast<float4 *>(p + lane * 32);
    q[0] = make_float4(f.c[0][0], f.c[0][1], f.c[0][2], f.c[0][3]);
    q[1] = make_float4(f.c[1][0], f.c[1][1], f.c[1][2], f.c[1][3]);
}
__device__ __forceinline__ void frag_load_add(const uint8_t *p, Frag16 &f, int lane)
{
    if (!smem_ok(smem_u32(p + lane * 32), 32)) return;
    const float4 *q = reinterpret_cast<const float4 *>(p + lane * 32);
    const float4 a = q[0], b = q[1];
    f.c[0][0] += a.x; f.c[0][1] += a.y; f.c[0][2] += a.z; f.c[0][3] += a.w;
    f.c[1][0] += b.x; f.c[1][1] += b.y; f.c[1][2] += b.z; f.c[1][3] += b.w;
}

// A block of the chunk matrix: rows scaled by beta_(ro + r), strictly lower part only on a
// diagonal block (off-diagonal blocks below the diagonal are kept whole).
__device__ __forceinline__ void mask_rows_beta(Frag16 &f, const float *beta, int ro, bool diag, int g, int t)
{
    const float b0 = beta[ro + g], b8 = beta[ro + g + 8];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int r = g + 8 * (i >> 1), j = 8 * nt + 2 * t + (i & 1);
            f.c[nt][i] = (!diag || j < r) ? f.c[nt][i] * ((i >> 1) ? b8 : b0) : 0.f;
        }
}

// 16x16 block of a 32x32 f16 tile (pitch LD32) at (ro, co): columns scaled by beta_(co + j) when
// `beta` is given; on a diagonal block of P, entries above the diagonal are written as zero.
__device__ __forceinline__ void store_block(uint8_t *tile, const Frag16 &f, int ro, int co, const float *beta,
                                            bool lower_incl, int g, int t)
{
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
        const int j = 8 * nt + 2 * t;
        float2 bc = make_float2(1.f, 1.f);
        if (beta) bc = make_float2(beta[co + j], beta[co + j + 1]);
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            const int r = g + 8 * hh;
            float v0 = f.c[nt][2 * hh] * bc.x, v1 = f.c[nt][2 * hh + 1] * bc.y;
            if (lower_incl) {
                v0 = j <= r ? v0 : 0.f;
                v1 = j + 1 <= r ? v1 : 0.f;
            }
            uint8_t *dst = tile + (ro + r) * LD32 + (co + j) * 2;
            if (smem_ok(smem_u32(dst), 4)) *reinterpret_cast<uint32_t *>(dst) = pack_f16(v0, v1);
        }
    }
}

template <int NS>
__global__ void __launch_bounds__(32 * (1 + 4 * NP + NS), 1)
    kda_fwd32_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                     const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap tg, const Params p)
{
    extern __shared__ uint8_t smem_dyn[];
    uint8_t *smem = smem_dyn + ((1024u - (smem_u32(smem_dyn) & 1023u)) & 1023u);
    const uint32_t sb = smem_u32(smem);
#define SM_AT(T, a) (*reinterpret_cast<T *>(smem + (smem_checked((a), sizeof(T), sb) - sb)))
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int unit = blockIdx.x / p.vsplit, slice = blockIdx.x % p.vsplit;
    const int seq = unit / p.H, h = unit % p.H;
    const Span sp = seq_span(p, seq);

    volatile int *flags = reinterpret_cast<volatile int *>(smem + OFF_FLAGS);
    const uint32_t qkg_full = sb + OFF_BAR, qkg_empty = qkg_full + NRQ * 8;
    const uint32_t v_full = qkg_empty + NRQ * 8, v_empty = v_full + NRV * 8;
    const uint32_t prep_full = v_empty + NRV * 8, prep_empty = prep_full + NP * 8;

    if (threadIdx.x == 0) {
        for (int i = 0; i < NRQ; ++i) {
            mbar_init(qkg_full + 8 * i, 1);
            mbar_init(qkg_empty + 8 * i, 1);
        }
        for (int i = 0; i < NRV; ++i) {
            mbar_init(v_full + 8 * i, 1);
            mbar_init(v_empty + 8 * i, NS);
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
    const int nch = (sp.len + C2 - 1) / C2;

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            tma_prefetch_desc(&tq);
            tma_prefetch_desc(&tk);
            tma_prefetch_desc(&tv);
            tma_prefetch_desc(&tg);
            int nq = 0, nv = 0;  // chunks whose q/k/g and v copies were issued
            for (int n = 0; n < nch; ++n) {
                const int tok = sp.bos + n * C2;
                const int qs = n % NRQ;
                if (!wait_bar(qkg_empty + 8 * qs, ((n / NRQ) & 1) ^ 1, flags)) break;
                const uint32_t fq = qkg_full + 8 * qs;
                mbar_arrive_expect_tx(fq, QKG_STAGE);
                const uint32_t dq = sb + OFF_QKG + qs * QKG_STAGE;
#pragma unroll
                for (int hf = 0; hf < 2; ++hf)
#pragma unroll
                    for (int b = 0; b < 2; ++b) {
                        const uint32_t d = dq + hf * QKG_HALF + b * RAW_BOX;
                        tma_load_3d(d + Q_OFF, &tq, 64 * b, h, tok + 16 * hf, fq);
                        tma_load_3d(d + K_OFF, &tk, 64 * b, h, tok + 16 * hf, fq);
                        tma_load_3d(d + G_OFF, &tg, 64 * b, h, tok + 16 * hf, fq);
                    }
                nq = n + 1;
                const int vs = n % NRV;
                if (!wait_bar(v_empty + 8 * vs, ((n / NRV) & 1) ^ 1, flags)) break;
                const uint32_t fv = v_full + 8 * vs;
                mbar_arrive_expect_tx(fv, V_STAGE);
                const uint32_t dv = sb + OFF_V + vs * V_STAGE;
#pragma unroll
                for (int hf = 0; hf < 2; ++hf)
#pragma unroll
                    for (int b = 0; b < 2; ++b) tma_load_3d(dv + hf * RAW_TILE + b * RAW_BOX, &tv, 64 * b, h, tok + 16 * hf, fv);
                nv = n + 1;
            }
            // never leave while copies this thread issued may still be landing
            for (int m = (nq > NRQ ? nq - NRQ : 0); m < nq; ++m) drain_bar(qkg_full + 8 * (m % NRQ), (m / NRQ) & 1);
            for (int m = (nv > NRV ? nv - NRV : 0); m < nv; ++m) drain_bar(v_full + 8 * (m % NRV), (m / NRV) & 1);
        }
        return;
    }

    if (warp < 1 + 4 * NP) {
        // ------------------------------------------------------------ prep lanes
        const int ln = (warp - 1) >> 2;               // prep lane 0 .. NP - 1
        const int lt = threadIdx.x - 32 - LANE_THREADS * ln;  // 0..127
        const int lw = lt >> 5;                       // warp within the lane
        const int hf = lt >> 6;                       // token half: rows 16 hf .. 16 hf + 15
        const int c0 = 2 * (lt & 63);                 // this thread's channels c0, c0 + 1
        const uint32_t bar_id = 1 + ln;
        const uint32_t scr = sb + OFF_SCR + ln * SCR;
        const uint32_t pslot = sb + OFF_SLOT + ln * SLOT;
        uint8_t *scr_p = smem + (scr - sb);
        uint8_t *slot_p = smem + (pslot - sb);
        const float *beta_s = reinterpret_cast<const float *>(scr_p + S_BETA);
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
            const int qs = n % NRQ;
            const uint32_t qph = (n / NRQ) & 1, pph = (n / NP) & 1;
            const int tok0 = sp.bos + n * C2;
            const int Lv = min(C2, sp.len - n * C2);
            float blogit = 0.f;
            const size_t bi = static_cast<size_t>(tok0 + lt) * p.H + h;
            if (lt < C2 && lt < Lv && gmem_ok(bi, 1, tokhead_elems(p)))
                blogit = __uint_as_float(static_cast<uint32_t>(__ldg(p.beta + bi)) << 16);
            if (!wait_bar(qkg_full + 8 * qs, qph, flags)) failed = true;
            const uint32_t raw = sb + OFF_QKG + qs * QKG_STAGE + hf * QKG_HALF;

            // gate in log2 units and its inclusive cumsum within this thread's half
            float G0[16], G1[16];
            {
                float acc0 = 0.f, acc1 = 0.f;
#pragma unroll
                for (int r = 0; r < 16; ++r) {
                    const uint32_t gw = SM_AT(const uint32_t, raw + G_OFF + raw_off(r, c0));
                    const float x0 = a_h * (bf16_lo(gw) + bias0), x1 = a_h * (bf16_hi(gw) + bias1);
                    const float ga0 = fmaf(hs, tanh_approx(0.5f * x0), hs);
                    const float ga1 = fmaf(hs, tanh_approx(0.5f * x1), hs);
                    const bool live = 16 * hf + r < Lv;
                    acc0 += live ? ga0 : 0.f;
                    acc1 += live ? ga1 : 0.f;
                    G0[r] = acc0;
                    G1[r] = acc1;
                }
            }
            SM_AT(float2, scr + S_GX + hf * 512 + c0 * 4) = make_float2(G0[15], G1[15]);
            if (!wait_bar(prep_empty + 8 * ln, pph ^ 1, flags)) failed = true;
            named_bar_sync(bar_id, LANE_THREADS);
            // Gm = G after token 15 (the exponent reference), Ge = G after token 31;
            // this half's offset: G_r = off + (local sum)
            const float2 other = SM_AT(const float2, scr + S_GX + (hf ^ 1) * 512 + c0 * 4);
            float Gm0, Gm1, off0, off1, Ge0, Ge1;
            if (hf == 0) {
                Gm0 = G0[15];
                Gm1 = G1[15];
                off0 = off1 = 0.f;
                Ge0 = Gm0 + other.x;
                Ge1 = Gm1 + other.y;
            } else {
                Gm0 = other.x;
                Gm1 = other.y;
                off0 = Gm0;
                off1 = Gm1;
                Ge0 = Gm0 + G0[15];
                Ge1 = Gm1 + G1[15];
            }
            if (hf == 1) SM_AT(float2, pslot + P_GAM + c0 * 4) = make_float2(ex2_approx(Ge0), ex2_approx(Ge1));
            const float se0 = ex2_approx(Ge0 - Gm0), se1 = ex2_approx(Ge1 - Gm1);  // 2^(Ge - Gm)
            const float dm0 = off0 - Gm0, dm1 = off1 - Gm1;                        // G_r - Gm = dm + local
            // all raw loads first: stores below may alias them as far as the compiler knows
            uint32_t kwv[16], qwv[16];
#pragma unroll
            for (int r = 0; r < 16; ++r) {
                kwv[r] = SM_AT(const uint32_t, raw + K_OFF + raw_off(r, c0));
                qwv[r] = SM_AT(const uint32_t, raw + Q_OFF + raw_off(r, c0));
            }
#pragma unroll
            for (int r = 0; r < 16; ++r) {
                const int row = 16 * hf + r;
                const bool live = row < Lv;
                const float k0 = live ? bf16_lo(kwv[r]) : 0.f, k1 = live ? bf16_hi(kwv[r]) : 0.f;
                const float q0 = live ? bf16_lo(qwv[r]) : 0.f, q1 = live ? bf16_hi(qwv[r]) : 0.f;
                const float d0 = dm0 + G0[r], d1 = dm1 + G1[r];
                const float u0 = ex2_approx(d0), u1 = ex2_approx(d1);        // 2^(G_r - Gm)
                const float f0 = ex2_approx(-d0), f1 = ex2_approx(-d1);      // 2^(Gm - G_r)
                const float gm0 = ex2_approx(off0 + G0[r]), gm1 = ex2_approx(off1 + G1[r]);  // Gamma_r
                SM_AT(uint32_t, pslot + P_BZ + row * LD + c0 * 2) = pack_bf16(k0 * gm0, k1 * gm1);
                SM_AT(uint32_t, pslot + P_BZ + (C2 + row) * LD + c0 * 2) = pack_bf16(q0 * gm0, q1 * gm1);
                SM_AT(uint32_t, pslot + P_KB + row * LD + c0 * 2) = pack_f16(k0 * f0 * se0, k1 * f1 * se1);
                const uint32_t o = row * LD + c0 * 2;
                SM_AT(uint32_t, scr + S_KLH + o) = pack_bf16(k0 * u0, k1 * u1);
                SM_AT(uint32_t, scr + S_QLH + o) = pack_bf16(q0 * u0, q1 * u1);
                uint32_t hi, lo;
                split_bf16(k0 * f0, k1 * f1, hi, lo);
                SM_AT(uint32_t, scr + S_KRH + o) = hi;
                SM_AT(uint32_t, scr + S_KRL + o) = lo;
            }
            if (lt < C2) SM_AT(float, scr + S_BETA + lt * 4) = lt < Lv ? fmaf(0.5f, tanh_approx(0.5f * blogit), 0.5f) : 0.f;
            named_bar_sync(bar_id, LANE_THREADS);
            if (lt == 0) mbar_arrive(qkg_empty + 8 * qs);

            // chunk products, two bf16 products per entry (Kl, Ql rounded once, Kr as hi + lo):
            //   warp 0: A00, A10 over channels 0-63;   warp 1: A10 over 64-127, A11
            //   warp 2: P00, P10 over channels 0-63;   warp 3: P10 over 64-127, P11
            constexpr int R16 = 16 * LD;  // rows 16..31 of a scratch tile
            const uint32_t xl = scr + ((lw < 2) ? S_KLH : S_QLH);
            Frag16 d0f, d1f;
            if ((lw & 1) == 0) {
                chunk_gram_x2<8>(xl, scr + S_KRH, scr + S_KRL, d0f, lane, 0);           // X00
                chunk_gram_x2<4>(xl + R16, scr + S_KRH, scr + S_KRL, d1f, lane, 0);     // X10, first half
            } else {
                chunk_gram_x2<4>(xl + R16, scr + S_KRH, scr + S_KRL, d1f, lane, 4);     // X10, second half
                chunk_gram_x2<8>(xl + R16, scr + S_KRH + R16, scr + S_KRL + R16, d0f, lane, 0);  // X11
                frag_store(scr_p + S_XCH + (lw >> 1) * 1024, d1f, lane);
            }
            named_bar_sync(bar_id, LANE_THREADS);
            Frag16 y;  // warp 0: A10 T00, kept for T10
            if (lw == 0) {
                frag_load_add(scr_p + S_XCH, d1f, lane);                // A10
                mask_rows_beta(d0f, beta_s, 0, true, g, t);
                mask_rows_beta(d1f, beta_s, 16, false, g, t);
                Frag16 t00;
                unit_lower_inverse(d0f, t00, g, t);
                store_block(slot_p + P_TT, t00, 0, 0, beta_s, false, g, t);
                uint32_t a[4], b[2][2];
                frag_as_a(d1f, a);
                frag_as_b(t00, b);
                frag_mul(y, a, b);
            } else if (lw == 1) {
                mask_rows_beta(d0f, beta_s, 16, true, g, t);
                Frag16 t11;
                unit_lower_inverse(d0f, t11, g, t);
                store_block(slot_p + P_TT, t11, 16, 16, beta_s, false, g, t);
                frag_store(scr_p + S_XCH + 2048, t11, lane);
            } else if (lw == 2) {
                frag_load_add(scr_p + S_XCH + 1024, d1f, lane);         // P10
                store_block(slot_p + P_PP, d0f, 0, 0, nullptr, true, g, t);
                store_block(slot_p + P_PP, d1f, 16, 0, nullptr, false, g, t);
            } else {
                store_block(slot_p + P_PP, d0f, 16, 16, nullptr, true, g, t);
            }
            named_bar_sync(bar_id, LANE_THREADS);
            if (lw == 0) {
                // T10 = -T11 (A10 T00)
                Frag16 t11, t10;
                frag_zero(t11);
                frag_load_add(scr_p + S_XCH + 2048, t11, lane);
                uint32_t a[4], b[2][2];
                frag_as_a(t11, a);
                frag_as_b(y, b);
                frag_mul(t10, a, b);
#pragma unroll
                for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                    for (int i = 0; i < 4; ++i) t10.c[nt][i] = -t10.c[nt][i];
                store_block(slot_p + P_TT, t10, 16, 0, beta_s, false, g, t);
            }
            const bool stop = named_bar_or(bar_id, LANE_THREADS, failed);
            if (lt == 0) mbar_arrive(prep_full + 8 * ln);
            if (stop) break;
        }
        return;
    }

    // ---------------------------------------------------------------- scan warps
    const int sw = warp - (1 + 4 * NP);
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
            if (p.init && gmem_ok(e, 2, state_elems(p))) {
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
        const int ps = n % NP, vs = n % NRV;
        bool ok = wait_bar(prep_full + 8 * ps, (n / NP) & 1, flags);
        ok = ok && wait_bar(v_full + 8 * vs, (n / NRV) & 1, flags);
        if (!__all_sync(0xffffffffu, ok)) break;
        const int tok0 = sp.bos + n * C2;
        const int Lv = min(C2, sp.len - n * C2);
        const uint32_t pb = sb + OFF_SLOT + ps * SLOT;
        const uint32_t vt = sb + OFF_V + vs * V_STAGE;

        // Z = S [K*Gamma ; Q*Gamma]^T  (16 rows x 64 columns per warp; z[nt] = columns 8 nt ..)
        float z[8][4];
#pragma unroll
        for (int i = 0; i < 8; ++i) z[i][0] = z[i][1] = z[i][2] = z[i][3] = 0.f;
        const uint32_t bz = pb + P_BZ + (ri + 8 * (mi >> 1)) * LD + 16 * (mi & 1);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
            const uint32_t a[4] = {pack_bf16(S[2 * kk][0], S[2 * kk][1]), pack_bf16(S[2 * kk][2], S[2 * kk][3]),
                                   pack_bf16(S[2 * kk + 1][0], S[2 * kk + 1][1]),
                                   pack_bf16(S[2 * kk + 1][2], S[2 * kk + 1][3])};
#pragma unroll
            for (int zb = 0; zb < 4; ++zb) {
                uint32_t b0, b1, b2, b3;
                ldsm_x4(bz + zb * 16 * LD + kk * 32, b0, b1, b2, b3);
                mma_bf16(z[2 * zb], a, b0, b1);
                mma_bf16(z[2 * zb + 1], a, b2, b3);
            }
        }

        // R = V^T - Z_k (tokens past the chunk's end are zero), in place of Z_k
#pragma unroll
        for (int nt = 0; nt < 4; ++nt)
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int j = 8 * nt + 2 * t + (i & 1), vr = vr0 + g + 8 * (i >> 1);
                const float vv = j < Lv ? __uint_as_float(static_cast<uint32_t>(
                                                  SM_AT(const uint16_t, vt + (j >> 4) * RAW_TILE + raw_off(j & 15, vr)))
                                              << 16)
                                        : 0.f;
                z[nt][i] = vv - z[nt][i];
            }
        __syncwarp();
        if (lane == 0) mbar_arrive(v_empty + 8 * vs);

        // E = R (T diag(beta))^T; T is lower, so tokens 0-15 take no part of columns 16-31
        uint32_t ra[2][4];
#pragma unroll
        for (int ks = 0; ks < 2; ++ks) {
            ra[ks][0] = pack_f16(z[2 * ks][0], z[2 * ks][1]);
            ra[ks][1] = pack_f16(z[2 * ks][2], z[2 * ks][3]);
            ra[ks][2] = pack_f16(z[2 * ks + 1][0], z[2 * ks + 1][1]);
            ra[ks][3] = pack_f16(z[2 * ks + 1][2], z[2 * ks + 1][3]);
        }
        float e[4][4];
#pragma unroll
        for (int nt = 0; nt < 4; ++nt) {
            e[nt][0] = e[nt][1] = e[nt][2] = e[nt][3] = 0.f;
            const uint32_t row = pb + P_TT + (8 * nt + g) * LD32 + 4 * t;
#pragma unroll
            for (int ks = 0; ks < 2; ++ks) {
                if (ks == 1 && nt < 2) continue;
                mma_f16(e[nt], ra[ks], SM_AT(const uint32_t, row + 32 * ks), SM_AT(const uint32_t, row + 32 * ks + 16));
            }
        }
        uint32_t ea[2][4];
#pragma unroll
        for (int ks = 0; ks < 2; ++ks) {
            ea[ks][0] = pack_f16(e[2 * ks][0], e[2 * ks][1]);
            ea[ks][1] = pack_f16(e[2 * ks][2], e[2 * ks][3]);
            ea[ks][2] = pack_f16(e[2 * ks + 1][0], e[2 * ks + 1][1]);
            ea[ks][3] = pack_f16(e[2 * ks + 1][2], e[2 * ks + 1][3]);
        }

        // O = scale (Z_q + E P^T)
#pragma unroll
        for (int nt = 0; nt < 4; ++nt) {
            const uint32_t row = pb + P_PP + (8 * nt + g) * LD32 + 4 * t;
#pragma unroll
            for (int ks = 0; ks < 2; ++ks) {
                if (ks == 1 && nt < 2) continue;
                mma_f16(z[4 + nt], ea[ks], SM_AT(const uint32_t, row + 32 * ks), SM_AT(const uint32_t, row + 32 * ks + 16));
            }
        }
#pragma unroll
        for (int nt = 0; nt < 4; ++nt)
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int r = 8 * nt + 2 * t + (i & 1), vr = vr0 + g + 8 * (i >> 1);
                const size_t oi = (static_cast<size_t>(tok0 + r) * p.H + h) * DH + vr;
                if (r < Lv && gmem_ok(oi, 1, out_elems(p))) p.out[oi] = f2bf_bits(p.scale * z[4 + nt][i]);
            }

        // S = S Diag(gamma) + E Kbar
#pragma unroll
        for (int nt = 0; nt < 16; ++nt) {
            const float2 gm = SM_AT(const float2, pb + P_GAM + (8 * nt + 2 * t) * 4);
            S[nt][0] *= gm.x;
            S[nt][1] *= gm.y;
            S[nt][2] *= gm.x;
            S[nt][3] *= gm.y;
        }
        const uint32_t kb = pb + P_KB + (ri + 8 * (mi & 1)) * LD + 16 * (mi >> 1);
#pragma unroll
        for (int ks = 0; ks < 2; ++ks)
#pragma unroll
            for (int m = 0; m < 8; ++m) {
                uint32_t b0, b1, b2, b3;
                ldsm_x4_t(kb + ks * 16 * LD + m * 32, b0, b1, b2, b3);
                mma_f16(S[2 * m], ea[ks], b0, b1);
                mma_f16(S[2 * m + 1], ea[ks], b2, b3);
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
                if (!gmem_ok(e, 2, state_elems(p))) continue;
                if (p.fin_dtype == KDA_DTYPE_FP32)
                    *reinterpret_cast<float2 *>(static_cast<float *>(p.fin) + e) = make_float2(S[nt][2 * hh], S[nt][2 * hh + 1]);
                else
                    *reinterpret_cast<uint32_t *>(static_cast<uint16_t *>(p.fin) + e) = pack_bf16(S[nt][2 * hh], S[nt][2 * hh + 1]);
            }
    }
}

#undef SM_AT

}  // namespace v32
}  // namespace kda
