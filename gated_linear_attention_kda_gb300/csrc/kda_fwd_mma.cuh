// kda_fwd_mma.cuh -- the KDA forward kernel with warp-level MMA state
// products (state rows in registers). Used when a state's V rows are split
// across several CTAs (few states); see kda_fwd_tc.cuh for the tcgen05 kernel.
#pragma once
#include "kda_chunk.cuh"
#include "kda_common.cuh"

namespace kda {
namespace v1 {

// ---------------------------------------------------------------- shared memory plan
constexpr int BZ_LD = 272;            // row pitch (bytes) of 128-wide 16-bit tiles (136 elements)
constexpr int SM_LD = 48;             // row pitch of 16x16 16-bit tiles (24 elements)
constexpr int P_BZ = 0;                           // bf16 [32][136]: K*Gamma rows 0-15, Q*Gamma rows 16-31
constexpr int P_KB = P_BZ + 32 * BZ_LD;           // f16  [16][136]: Kbar
constexpr int P_TT = P_KB + 16 * BZ_LD;           // f16  [16][24]:  T diag(beta)
constexpr int P_PP = P_TT + 16 * SM_LD;           // f16  [16][24]:  P
constexpr int P_GAM = P_PP + 16 * SM_LD;          // f32  [128]:     gamma = Gamma at chunk end
constexpr int PREP_SLOT = P_GAM + DH * 4;

constexpr int H_LD = 272;             // row pitch of 16-bit [16][136] tiles
constexpr int S_KLH = 0;              // bf16 K * 2^(G - G_mid)
constexpr int S_QLH = S_KLH + 16 * H_LD;  // bf16 Q * 2^(G - G_mid)
constexpr int S_KRH = S_QLH + 16 * H_LD;  // bf16 hi / lo of K * 2^(G_mid - G)
constexpr int S_KRL = S_KRH + 16 * H_LD;
constexpr int S_BETA = S_KRL + 16 * H_LD;
constexpr int S_NRM = S_BETA + 64;    // f32 [2 warps][32]: row sums of squares of k (rows 0-15) and q (16-31)
constexpr int SCR = S_NRM + 256;

// Rings by the number of scan warps NS (16 V rows each). With few rows per CTA the scan of a chunk
// is short and the prep lanes pace the CTA: three lanes with two slots each, so a lane can prepare
// its next chunk while the scan still reads its previous one (raw ring 5 deep). With 64 rows
// (NS = 4) the scan takes longer: four lanes with one slot each (raw ring 6 deep).
template <int NS>
struct Layout {
    static constexpr int NP = NS >= 4 ? 4 : 3;             // prep lanes
    static constexpr int NSLOT = NS >= 4 ? NP : 2 * NP;    // prep slots; chunk n uses slot n % NSLOT
    static constexpr int NR = NS >= 4 ? 6 : 5;             // raw q/k/v/g ring depth (chunks)
    static constexpr int OFF_RAW = 0;
    static constexpr int OFF_PREP = OFF_RAW + NR * RAW_STAGE;
    static constexpr int OFF_SCR = OFF_PREP + NSLOT * PREP_SLOT;
    static constexpr int OFF_BAR = OFF_SCR + NP * SCR;
    static constexpr int NBAR = 2 * NR + 2 * NSLOT;
    static constexpr int OFF_FLAGS = OFF_BAR + NBAR * 8;
    static constexpr int SMEM_USED = OFF_FLAGS + 16;
    static constexpr int SMEM_ALLOC = SMEM_USED + 1024;  // the ring base is rounded up to 1024 B (128B swizzle)
    static constexpr int NTHREADS = 32 * (1 + 2 * NP + NS);
    static_assert(NSLOT % NP == 0, "each slot belongs to one lane");
    static_assert(PREP_SLOT % 16 == 0 && SCR % 16 == 0 && OFF_PREP % 1024 == 0, "alignment");
    static_assert(OFF_BAR % 8 == 0, "mbarrier alignment");
    static_assert(SMEM_ALLOC <= 227 * 1024, "shared memory budget");
};

// L2 scale factor 1 / sqrt(sum x^2 + 1e-6) of k row `lane` (lanes 0-15) or q row `lane - 16`
// (lanes 16-31) of a prep lane's chunk: each thread holds two channels of every row, a warp 64
// channels. The 32 per-thread sums of squares go through a reduce-scatter butterfly (lane l
// ends with its warp's sum of value l), the two warps' halves meet in shared memory.
__device__ __forceinline__ float qk_row_scale64(const uint32_t (&kw)[CHUNK], const uint32_t (&qw)[CHUNK], int lane,
                                                int lw, uint8_t *nrm, uint32_t bar_id)
{
    float v[32];
#pragma unroll
    for (int r = 0; r < CHUNK; ++r) {
        const float k0 = bf16_lo(kw[r]), k1 = bf16_hi(kw[r]), q0 = bf16_lo(qw[r]), q1 = bf16_hi(qw[r]);
        v[r] = fmaf(k0, k0, k1 * k1);
        v[CHUNK + r] = fmaf(q0, q0, q1 * q1);
    }
#pragma unroll
    for (int w = 16; w >= 1; w >>= 1) {
        const bool up = lane & w;
#pragma unroll
        for (int i = 0; i < w; ++i) {
            const float keep = up ? v[i + w] : v[i], send = up ? v[i] : v[i + w];
            v[i] = keep + __shfl_xor_sync(0xffffffffu, send, w);
        }
    }
    reinterpret_cast<float *>(nrm)[32 * lw + lane] = v[0];
    named_bar_sync(bar_id, 64);
    const float tot = reinterpret_cast<const float *>(nrm)[lane] + reinterpret_cast<const float *>(nrm)[32 + lane];
    return rsqrtf(tot + 1e-6f);
}

// QKN: L2-normalise the q and k rows in the element-wise pass (KDA_FLAG_QK_L2NORM).
template <int NS, bool QKN>
__global__ void __launch_bounds__(Layout<NS>::NTHREADS, 1)
    kda_fwd_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                   const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap tg, const Params p)
{
    using L = Layout<NS>;
    constexpr int NP = L::NP, NSLOT = L::NSLOT, NR = L::NR;
    constexpr int OFF_RAW = L::OFF_RAW, OFF_PREP = L::OFF_PREP, OFF_SCR = L::OFF_SCR, OFF_BAR = L::OFF_BAR,
                  OFF_FLAGS = L::OFF_FLAGS;
    extern __shared__ uint8_t smem_dyn[];
    // align to 1024 B by pointer arithmetic on the shared array, so that accesses
    // through `smem` stay in the shared address space
    uint8_t *smem = smem_dyn + ((1024u - (smem_u32(smem_dyn) & 1023u)) & 1023u);
    const uint32_t sb = smem_u32(smem);
#define SM_AT(T, a) (*reinterpret_cast<T *>(smem + (smem_checked((a), sizeof(T), sb) - sb)))
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int unit = blockIdx.x / p.vsplit, slice = blockIdx.x % p.vsplit;
    const int seq = unit / p.H, h = unit % p.H;
    const Span sp = seq_span(p, seq);

    volatile int *flags = reinterpret_cast<volatile int *>(smem + OFF_FLAGS);
    const uint32_t raw_full = sb + OFF_BAR, raw_empty = raw_full + NR * 8;
    const uint32_t prep_full = raw_empty + NR * 8, prep_empty = prep_full + NSLOT * 8;

    if (threadIdx.x == 0) {
        for (int i = 0; i < NR; ++i) {
            mbar_init(raw_full + 8 * i, 1);
            mbar_init(raw_empty + 8 * i, 1 + NS);
        }
        for (int i = 0; i < NSLOT; ++i) {
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

    if (warp < 1 + 2 * NP) {
        // ------------------------------------------------------------ prep lanes
        const int ln = (warp - 1) >> 1;            // prep lane 0 .. NP - 1
        const int lt = threadIdx.x - 32 - 64 * ln;  // 0..63
        const int lw = lt >> 5;                     // warp within the lane
        const uint32_t bar_id = 1 + ln;
        const uint32_t scr = sb + OFF_SCR + ln * SCR;
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
            const uint32_t rph = (n / NR) & 1, pph = (n / NSLOT) & 1;
            const int ps = n % NSLOT;  // slot ln or ln + NP
            const uint32_t pslot = sb + OFF_PREP + ps * PREP_SLOT;
            const int tok0 = sp.bos + n * CHUNK;
            const int Lv = min(CHUNK, sp.len - n * CHUNK);
            float blogit = 0.f;
            const size_t bi = static_cast<size_t>(tok0 + lane) * p.H + h;
            if (lw == 1 && lane < Lv && gmem_ok(bi, 1, tokhead_elems(p)))
                blogit = __uint_as_float(static_cast<uint32_t>(__ldg(p.beta + bi)) << 16);
            if (!wait_bar(raw_full + 8 * rs, rph, flags)) failed = true;
            const uint32_t raw = sb + OFF_RAW + rs * RAW_STAGE;

            // gate in log2 units and its inclusive in-chunk cumsum
            float G0[CHUNK], G1[CHUNK];
            {
                float acc0 = 0.f, acc1 = 0.f;
#pragma unroll
                for (int r = 0; r < CHUNK; ++r) {
                    const uint32_t gw = SM_AT(const uint32_t, raw + OFF_G + raw_off(r, c0));
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
            // all raw loads first: stores below may alias them as far as the compiler knows. With
            // in-kernel q/k normalisation the row scales need only these tiles, so they are formed
            // here, while the lane would otherwise wait for its slot
            uint32_t kwv[CHUNK], qwv[CHUNK];
#pragma unroll
            for (int r = 0; r < CHUNK; ++r) {
                kwv[r] = SM_AT(const uint32_t, raw + OFF_K + raw_off(r, c0));
                qwv[r] = SM_AT(const uint32_t, raw + OFF_Q + raw_off(r, c0));
            }
            float fqk = 1.f;
            if constexpr (QKN) fqk = qk_row_scale64(kwv, qwv, lane, lw, smem + (scr + S_NRM - sb), bar_id);
            if (!wait_bar(prep_empty + 8 * ps, pph ^ 1, flags)) failed = true;

            const float Gm0 = G0[7], Gm1 = G1[7];  // mid-chunk reference halves the exponent range
            const float sm0 = ex2_approx(-Gm0), sm1 = ex2_approx(-Gm1);
            const float se0 = ex2_approx(G0[15] - Gm0), se1 = ex2_approx(G1[15] - Gm1);
            SM_AT(float2, pslot + P_GAM + c0 * 4) = make_float2(ex2_approx(G0[15]), ex2_approx(G1[15]));
#pragma unroll
            for (int r = 0; r < CHUNK; ++r) {
                const uint32_t kw = kwv[r], qw = qwv[r];
                const bool live = r < Lv;
                float k0 = live ? bf16_lo(kw) : 0.f, k1 = live ? bf16_hi(kw) : 0.f;
                float q0 = live ? bf16_lo(qw) : 0.f, q1 = live ? bf16_hi(qw) : 0.f;
                if constexpr (QKN) {
                    const float fk = __shfl_sync(0xffffffffu, fqk, r), fq = __shfl_sync(0xffffffffu, fqk, CHUNK + r);
                    k0 *= fk;
                    k1 *= fk;
                    q0 *= fq;
                    q1 *= fq;
                }
                const float gm0 = ex2_approx(G0[r]), gm1 = ex2_approx(G1[r]);            // Gamma_r
                const float f0 = ex2_approx(Gm0 - G0[r]), f1 = ex2_approx(Gm1 - G1[r]);  // 2^(G_mid - G_r)
                SM_AT(uint32_t, pslot + P_BZ + r * BZ_LD + c0 * 2) = pack_bf16(k0 * gm0, k1 * gm1);
                SM_AT(uint32_t, pslot + P_BZ + (16 + r) * BZ_LD + c0 * 2) = pack_bf16(q0 * gm0, q1 * gm1);
                SM_AT(uint32_t, pslot + P_KB + r * BZ_LD + c0 * 2) = pack_f16(k0 * f0 * se0, k1 * f1 * se1);
                const float u0 = gm0 * sm0, u1 = gm1 * sm1;                              // 2^(G_r - G_mid)
                const uint32_t o = r * H_LD + c0 * 2;
                SM_AT(uint32_t, scr + S_KLH + o) = pack_bf16(k0 * u0, k1 * u1);
                SM_AT(uint32_t, scr + S_QLH + o) = pack_bf16(q0 * u0, q1 * u1);
                uint32_t hi, lo;
                split_bf16(k0 * f0, k1 * f1, hi, lo);
                SM_AT(uint32_t, scr + S_KRH + o) = hi;
                SM_AT(uint32_t, scr + S_KRL + o) = lo;
            }
            if (lw == 1 && lane < CHUNK)
                SM_AT(float, scr + S_BETA + lane * 4) = lane < Lv ? fmaf(0.5f, tanh_approx(0.5f * blogit), 0.5f) : 0.f;
            named_bar_sync(bar_id, 64);
            if (lt == 0) mbar_arrive(raw_empty + 8 * rs);

            // warp 0: A = strictly-lower(beta_r Kl Kr^T), T' = (I + A)^-1 diag(beta);
            // warp 1: P = lower(Ql Kr^T). Two bf16 products per entry: Kl, Ql rounded once, Kr as hi + lo.
            {
                Frag16 acc;
                if (lw == 0)
                    chunk_gram_x2<8>(scr + S_KLH, scr + S_KRH, scr + S_KRL, acc, lane, 0);
                else
                    chunk_gram_x2<8>(scr + S_QLH, scr + S_KRH, scr + S_KRL, acc, lane, 0);
                if (lw == 0) {
                    const float bg = SM_AT(const float, scr + S_BETA + g * 4), bg8 = SM_AT(const float, scr + S_BETA + (g + 8) * 4);
#pragma unroll
                    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            const int r = g + 8 * (i >> 1), j = 8 * nt + 2 * t + (i & 1);
                            acc.c[nt][i] = j < r ? acc.c[nt][i] * ((i >> 1) ? bg8 : bg) : 0.f;
                        }
                    Frag16 T;
                    unit_lower_inverse(acc, T, g, t);
#pragma unroll
                    for (int nt = 0; nt < 2; ++nt) {
                        const int col = 8 * nt + 2 * t;
                        const float2 bc = SM_AT(const float2, scr + S_BETA + col * 4);
#pragma unroll
                        for (int hh = 0; hh < 2; ++hh)
                            SM_AT(uint32_t, pslot + P_TT + (g + 8 * hh) * SM_LD + col * 2) =
                                pack_f16(T.c[nt][2 * hh] * bc.x, T.c[nt][2 * hh + 1] * bc.y);
                    }
                } else {
#pragma unroll
                    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                        for (int hh = 0; hh < 2; ++hh) {
                            const int r = g + 8 * hh, j = 8 * nt + 2 * t;
                            const float v0 = j <= r ? acc.c[nt][2 * hh] : 0.f;
                            const float v1 = j + 1 <= r ? acc.c[nt][2 * hh + 1] : 0.f;
                            SM_AT(uint32_t, pslot + P_PP + r * SM_LD + j * 2) = pack_f16(v0, v1);
                        }
                }
            }
            const bool stop = named_bar_or(bar_id, 64, failed);
            if (lt == 0) mbar_arrive(prep_full + 8 * ps);
            if (stop) break;
        }
        return;
    }

    // ---------------------------------------------------------------- scan warps
    const int sw = warp - (1 + 2 * NP);
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
        const int ps = n % NSLOT, rs = n % NR;
        const uint32_t pph = (n / NSLOT) & 1, rph = (n / NR) & 1;
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
                const float vv = j < Lv ? __uint_as_float(static_cast<uint32_t>(SM_AT(const uint16_t, vt + raw_off(j, vr))) << 16) : 0.f;
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
            mma_f16(e[nt], ra, SM_AT(const uint32_t, row), SM_AT(const uint32_t, row + 16));
        }
        const uint32_t ea[4] = {pack_f16(e[0][0], e[0][1]), pack_f16(e[0][2], e[0][3]), pack_f16(e[1][0], e[1][1]),
                                pack_f16(e[1][2], e[1][3])};

        // O = scale (Z_q + E P^T)
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
            const uint32_t row = pb + P_PP + (8 * nt + g) * SM_LD + 4 * t;
            mma_f16(z[2 + nt], ea, SM_AT(const uint32_t, row), SM_AT(const uint32_t, row + 16));
        }
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int r = 8 * nt + 2 * t + (i & 1), vr = vr0 + g + 8 * (i >> 1);
                const size_t oi = (static_cast<size_t>(tok0 + r) * p.H + h) * DH + vr;
                if (r < Lv && gmem_ok(oi, 1, out_elems(p))) p.out[oi] = f2bf_bits(p.scale * z[2 + nt][i]);
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
                if (!gmem_ok(e, 2, state_elems(p))) continue;
                if (p.fin_dtype == KDA_DTYPE_FP32)
                    *reinterpret_cast<float2 *>(static_cast<float *>(p.fin) + e) = make_float2(S[nt][2 * hh], S[nt][2 * hh + 1]);
                else
                    *reinterpret_cast<uint32_t *>(static_cast<uint16_t *>(p.fin) + e) = pack_bf16(S[nt][2 * hh], S[nt][2 * hh + 1]);
            }
    }
}


#undef SM_AT

}  // namespace v1
}  // namespace kda
