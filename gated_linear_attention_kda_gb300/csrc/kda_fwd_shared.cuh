// kda_fwd_shared.cuh -- the split-state warp-MMA forward kernel with each chunk prepared once
// per state: the VS CTAs that split a state's V rows form one thread-block cluster, CTA rank
// n % VS prepares chunk n (gate, cumsum, scaled operand tiles, the chunk matrices A and P, the
// inverse T = (I + A)^-1) exactly as the warp-MMA kernel's prep lanes do, and publishes the
// prepared operands to a workspace in global memory (a 16-entry ring per state, read back through
// L2); every CTA of the cluster, the owner included, copies each chunk's entry into a stage
// beside the chunk's V tile and scans it from there. Each CTA prepares only 1 / VS of the chunks, and the preparation
// never waits on the scan: a prep lane's staging slot is free again once it is copied out.
//
// Per chunk n, owner o = n % VS, workspace entry e = n % NG. Entry e is always written by the same
// owner (e % VS) and, since NG / VS is even, by the same one of its two prep lanes, so every
// barrier of an entry is waited on in phase order by a single waiter:
//   owner   prep lane -> staging slot (shared memory); once every CTA released entry e's previous
//           chunk (mbarrier `gfree[e]` of the owner, one arrival per CTA): copy the slot to entry
//           e; one thread then fences at cluster scope and arrives (relaxed) on `ready[e]` of
//           every CTA -- one fence per chunk, where release-qualified arrivals would fence once
//           per arrival.
//   all     the feeder thread waits for `ready[e]` (acquire at cluster scope) and bulk-copies
//           entry e into a stage beside the chunk's V tile; when it reuses that stage NST chunks
//           later (the copy has long landed and been scanned), it releases entry e with a relaxed
//           arrival on the owner's `gfree[e]` (nothing to order: the copy's reads completed
//           before its transaction count did). The scan warps never signal another CTA.
// The imported bytes are the prep lane's, so results equal the warp-MMA kernel's at the same
// split bit for bit. The rows of S are independent, which is what makes the split exact
// ("FlashKDA Input Tensor Shapes and DTypes ..." -- "Initial and Final States").
//
// Roles (9 warps, see NWARPS): warp 0 lane 0 the feeder (in chunk order: the V tile and the
// import of every chunk), two prep lanes of two warps (alternate own chunks; each lane loads its
// own q/k/g tiles), NS scan warps of 16 V rows (fp32 state in registers), on sub-partitions of
// their own.
#pragma once
#include "cluster.cuh"
#include "kda_chunk.cuh"
#include "kda_common.cuh"
#include "kda_fwd_mma.cuh"

namespace kda {
namespace v1s {

using v1::BZ_LD;
using v1::H_LD;
using v1::P_BZ;
using v1::P_GAM;
using v1::P_KB;
using v1::P_PP;
using v1::P_TT;
using v1::PREP_SLOT;
using v1::S_BETA;
using v1::S_KLH;
using v1::S_KRH;
using v1::S_KRL;
using v1::S_QLH;
using v1::SCR;
using v1::SM_LD;

constexpr int NG = 16;  // workspace ring entries per state (an even multiple of every split)
constexpr int NL = 2;   // prep lanes (own chunks alternate between them)
constexpr int NST = 7;  // stages: the V tile and the imported prepared operands of one chunk

constexpr int QKG_STAGE = 3 * RAW_TILE;  // q, k, g tiles of one chunk: one stage per prep lane
constexpr int QS_Q = 0, QS_K = RAW_TILE, QS_G = 2 * RAW_TILE;
constexpr int SLOT_PAD = (PREP_SLOT + 1023) / 1024 * 1024;
constexpr int STAGE = RAW_TILE + SLOT_PAD;  // V tile (128B-swizzled, at a 1024-byte boundary), then the slot
constexpr int OT_LD = 48;                   // row pitch of a scan warp's 16 x 16 bf16 output tile
constexpr int OT_BYTES = 16 * OT_LD;
constexpr int MAX_NS = 4;
constexpr int OFF_STG = 0;
constexpr int OFF_QKG = OFF_STG + NST * STAGE;
constexpr int OFF_OWN = OFF_QKG + NL * QKG_STAGE;  // one staging slot per prep lane
constexpr int OFF_SCR = OFF_OWN + NL * PREP_SLOT;
constexpr int OFF_OT = OFF_SCR + NL * SCR;
constexpr int OFF_BAR = OFF_OT + MAX_NS * OT_BYTES;
// barriers: stage full / empty [NST], q/k/g full [NL], ready [NG], gfree [NG]
constexpr int NBAR = 2 * NST + NL + 2 * NG;
constexpr int OFF_FLAGS = OFF_BAR + NBAR * 8;
constexpr int SMEM_USED = OFF_FLAGS + 16;
constexpr int SMEM_ALLOC = SMEM_USED + 1024;  // the ring base is rounded up to 1024 B (128B swizzle)

static_assert(PREP_SLOT % 16 == 0 && STAGE % 1024 == 0 && OFF_OWN % 16 == 0 && OFF_OT % 16 == 0,
              "bulk copies and 16-byte accesses need 16-byte units");
static_assert(RAW_TILE % 1024 == 0 && OFF_QKG % 1024 == 0, "128B-swizzled TMA boxes need 1024-byte alignment");
static_assert(NG % 16 == 0, "a workspace entry keeps one owner and one prep lane at every split");
static_assert(NG > NST, "an entry is released before its owner needs it again");
static_assert(OFF_BAR % 8 == 0, "mbarrier alignment");
static_assert(SMEM_ALLOC <= 227 * 1024, "shared memory budget");

// Workspace bytes per state: NG prepared chunks.
constexpr int64_t workspace_bytes_per_state() { return static_cast<int64_t>(NG) * PREP_SLOT; }

// Warp roles, placed so that scan warps and prep warps sit on different SM sub-partitions (warp
// w runs on sub-partition w % 4): warp 0 the feeder; warps 4 i + 1 and 4 i + 2 the scan warps
// (scan warp 2 i and 2 i + 1); warps 3, 4 prep lane 0 and warps 7, 8 prep lane 1. Warps left over
// at NS < 4 only take part in the cluster barriers.
constexpr int NWARPS = 9;
constexpr int NTHREADS = 32 * NWARPS;
__device__ __forceinline__ int scan_warp_index(int w) { return (w & 3) == 1 || (w & 3) == 2 ? 2 * (w >> 2) + (w & 3) - 1 : -1; }
__device__ __forceinline__ int prep_lane_of(int w) { return w == 3 || w == 4 ? 0 : (w == 7 || w == 8 ? 1 : -1); }

template <int NS>
__global__ void __launch_bounds__(NTHREADS, 1)
    kda_fwd_shared_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                          const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap tg, const Params p,
                          uint8_t *ws)
{
    constexpr int VS = 8 / NS;  // CTAs per state = the cluster
    extern __shared__ uint8_t smem_dyn[];
    uint8_t *smem = smem_dyn + ((1024u - (smem_u32(smem_dyn) & 1023u)) & 1023u);
    const uint32_t sb = smem_u32(smem);
#define SM_AT(T, a) (*reinterpret_cast<T *>(smem + (smem_checked((a), sizeof(T), sb) - sb)))
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int unit = blockIdx.x / VS;
    const int rank = static_cast<int>(cluster_ctarank());  // = blockIdx.x % VS: the V-row slice
    const int seq = unit / p.H, h = unit % p.H;
    const Span sp = seq_span(p, seq);
    uint8_t *wsu = ws + static_cast<size_t>(unit) * NG * PREP_SLOT;  // this state's workspace ring

    volatile int *flags = reinterpret_cast<volatile int *>(smem + OFF_FLAGS);
    const uint32_t st_full = sb + OFF_BAR, st_empty = st_full + NST * 8;
    const uint32_t qkg_full = st_empty + NST * 8;
    const uint32_t ready = qkg_full + NL * 8, gfree = ready + NG * 8;

    if (threadIdx.x == 0) {
        for (int i = 0; i < NST; ++i) {
            mbar_init(st_full + 8 * i, 1);
            mbar_init(st_empty + 8 * i, NS);  // every scan warp
        }
        for (int i = 0; i < NL; ++i) mbar_init(qkg_full + 8 * i, 1);
        for (int i = 0; i < NG; ++i) {
            mbar_init(ready + 8 * i, 1);   // the owner's prep lane
            mbar_init(gfree + 8 * i, VS);  // the feeder of every CTA of the cluster
        }
        flags[0] = 0;
        fence_mbar_init();
        if (p.cu && blockIdx.x == 0 && (p.cu[0] != 0 || p.cu[p.nseq] != p.total))
            atomicOr(&g_dev_error, DEVERR_SEQLENS);
        if (!sp.ok && rank == 0 && h == 0) atomicOr(&g_dev_error, DEVERR_SEQLENS);
    }
    if (!sp.ok) return;  // uniform over the cluster (one state per cluster), before any cluster barrier
    // every CTA's barriers are initialised before any arrival from another CTA reaches them
    __syncwarp();  // the cluster barrier is warp-aligned
    cluster_sync_all();
    const int nch = (sp.len + CHUNK - 1) / CHUNK;

    if (warp == 0) {
        if (lane == 0) {
            // -------------------------------------------- feeder: V tile and import of every chunk
            tma_prefetch_desc(&tv);
            int issued = 0;
            for (int n = 0; n < nch; ++n) {
                const int s = n % NST, e = n % NG;
                if (!wait_bar(st_empty + 8 * s, ((n / NST) & 1) ^ 1, flags)) break;
                if (n >= NST) {  // chunk n - NST has left stage s: its owner may reuse the workspace entry
                    // (the copy's reads completed before its transaction count did, so there is
                    // nothing to release: the arrival is relaxed)
                    const int m = n - NST;
                    mbar_arrive_cluster_relaxed(mapa_shared(gfree + 8 * (m % NG), static_cast<uint32_t>(m % VS)));
                }
                if (!wait_cluster(ready + 8 * e, (n / NG) & 1, flags)) break;
                fence_proxy_async_global();  // the owner's generic writes, seen by this thread's bulk copy
                const uint32_t fb = st_full + 8 * s, dst = sb + OFF_STG + s * STAGE;
                mbar_arrive_expect_tx(fb, RAW_TILE + PREP_SLOT);
                const int tok = sp.bos + n * CHUNK;
#pragma unroll
                for (int b = 0; b < 2; ++b) tma_load_3d(dst + b * RAW_BOX, &tv, 64 * b, h, tok, fb);
                bulk_load_global(dst + RAW_TILE, wsu + static_cast<size_t>(e) * PREP_SLOT, PREP_SLOT, fb);
                issued = n + 1;
            }
            // no copy is left in flight when the CTA exits
            for (int m = (issued > NST ? issued - NST : 0); m < issued; ++m)
                drain_bar(st_full + 8 * (m % NST), (m / NST) & 1);
        }
    } else if (prep_lane_of(warp) >= 0) {
        // ------------------------------------------------------------ prep lanes: own chunks
        const int ln = prep_lane_of(warp);
        const int lt = threadIdx.x - 32 * (ln == 0 ? 3 : 7);  // 0..63
        const int lw = lt >> 5;
        const uint32_t bar_id = 1 + ln;
        const uint32_t scr = sb + OFF_SCR + ln * SCR;
        const uint32_t pslot = sb + OFF_OWN + ln * PREP_SLOT;  // staging slot
        const uint32_t qkg = sb + OFF_QKG + ln * QKG_STAGE, qb = qkg_full + 8 * ln;
        const int c0 = 2 * lt;
        float a_h = 1.f, bias0 = 0.f, bias1 = 0.f;
        if (p.A_log) a_h = ex2_approx(__ldg(p.A_log + h) * LOG2E);
        if (p.dt_bias) {
            bias0 = __ldg(p.dt_bias + h * DH + c0);
            bias1 = __ldg(p.dt_bias + h * DH + c0 + 1);
        }
        const float hs = p.half_gs;
        const int g = lane >> 2, t = lane & 3;
        // this lane's k-th chunk is own chunk j = ln + NL k, chunk n = rank + VS j; its q/k/g
        // tiles land in the lane's stage, loaded by thread 0 of the lane one chunk ahead
        auto load_qkg = [&](int n) {
            mbar_arrive_expect_tx(qb, QKG_STAGE);
            const int tok = sp.bos + n * CHUNK;
#pragma unroll
            for (int b = 0; b < 2; ++b) {
                tma_load_3d(qkg + QS_Q + b * RAW_BOX, &tq, 64 * b, h, tok, qb);
                tma_load_3d(qkg + QS_K + b * RAW_BOX, &tk, 64 * b, h, tok, qb);
                tma_load_3d(qkg + QS_G + b * RAW_BOX, &tg, 64 * b, h, tok, qb);
            }
        };
        const int n_first = rank + VS * ln;
        int loaded = 0;  // loads issued by this lane
        if (lt == 0 && n_first < nch) {
            tma_prefetch_desc(&tq);
            tma_prefetch_desc(&tk);
            tma_prefetch_desc(&tg);
            load_qkg(n_first);
        }
        if (n_first < nch) loaded = 1;

        int k = 0;
        for (;; ++k) {
            const int j = ln + NL * k;
            const int n = rank + VS * j;
            if (n >= nch) break;
            bool failed = false;
            const int tok0 = sp.bos + n * CHUNK;
            const int Lv = min(CHUNK, sp.len - n * CHUNK);
            float blogit = 0.f;
            const size_t bi = static_cast<size_t>(tok0 + lane) * p.H + h;
            if (lw == 1 && lane < Lv && gmem_ok(bi, 1, tokhead_elems(p)))
                blogit = __uint_as_float(static_cast<uint32_t>(__ldg(p.beta + bi)) << 16);
            if (!wait_bar(qb, k & 1, flags)) failed = true;

            // gate in log2 units and its inclusive in-chunk cumsum
            float G0[CHUNK], G1[CHUNK];
            {
                float acc0 = 0.f, acc1 = 0.f;
#pragma unroll
                for (int r = 0; r < CHUNK; ++r) {
                    const uint32_t gw = SM_AT(const uint32_t, qkg + QS_G + raw_off(r, c0));
                    const float x0 = a_h * (bf16_lo(gw) + bias0), x1 = a_h * (bf16_hi(gw) + bias1);
                    const float ga0 = fmaf(hs, tanh_approx(0.5f * x0), hs);
                    const float ga1 = fmaf(hs, tanh_approx(0.5f * x1), hs);
                    acc0 += (r < Lv) ? ga0 : 0.f;
                    acc1 += (r < Lv) ? ga1 : 0.f;
                    G0[r] = acc0;
                    G1[r] = acc1;
                }
            }
            uint32_t kwv[CHUNK], qwv[CHUNK];
#pragma unroll
            for (int r = 0; r < CHUNK; ++r) {
                kwv[r] = SM_AT(const uint32_t, qkg + QS_K + raw_off(r, c0));
                qwv[r] = SM_AT(const uint32_t, qkg + QS_Q + raw_off(r, c0));
            }

            const float Gm0 = G0[7], Gm1 = G1[7];  // mid-chunk reference halves the exponent range
            const float sm0 = ex2_approx(-Gm0), sm1 = ex2_approx(-Gm1);
            const float se0 = ex2_approx(G0[15] - Gm0), se1 = ex2_approx(G1[15] - Gm1);
            SM_AT(float2, pslot + P_GAM + c0 * 4) = make_float2(ex2_approx(G0[15]), ex2_approx(G1[15]));
#pragma unroll
            for (int r = 0; r < CHUNK; ++r) {
                const uint32_t kw = kwv[r], qw = qwv[r];
                const bool live = r < Lv;
                const float k0 = live ? bf16_lo(kw) : 0.f, k1 = live ? bf16_hi(kw) : 0.f;
                const float q0 = live ? bf16_lo(qw) : 0.f, q1 = live ? bf16_hi(qw) : 0.f;
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
            // the stage has been read: load the lane's next chunk into it
            const int n_next = n + VS * NL;
            if (n_next < nch && !failed) {
                if (lt == 0) load_qkg(n_next);
                loaded = k + 2;
            }

            // warp 0: A and T' = (I + A)^-1 diag(beta); warp 1: P (two bf16 products per entry)
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
                            const int r = g + 8 * (i >> 1), jj = 8 * nt + 2 * t + (i & 1);
                            acc.c[nt][i] = jj < r ? acc.c[nt][i] * ((i >> 1) ? bg8 : bg) : 0.f;
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
                            const int r = g + 8 * hh, jj = 8 * nt + 2 * t;
                            const float v0 = jj <= r ? acc.c[nt][2 * hh] : 0.f;
                            const float v1 = jj + 1 <= r ? acc.c[nt][2 * hh + 1] : 0.f;
                            SM_AT(uint32_t, pslot + P_PP + r * SM_LD + jj * 2) = pack_f16(v0, v1);
                        }
                }
            }
            // publish: once every CTA has released this entry's previous chunk, copy the slot to the
            // workspace, fence, and signal every CTA of the cluster
            const int e = n % NG;
            if (!wait_cluster(gfree + 8 * e, ((n / NG) & 1) ^ 1, flags)) failed = true;
            named_bar_sync(bar_id, 64);  // the slot is complete
            {
                const uint4 *src = reinterpret_cast<const uint4 *>(smem + (pslot - sb));
                uint4 *dst = reinterpret_cast<uint4 *>(wsu + static_cast<size_t>(e) * PREP_SLOT);
                for (int i = lt; i < PREP_SLOT / 16; i += 64) dst[i] = src[i];
            }
            fence_proxy_async_global();  // these generic writes, for the bulk copies that read them
            if (named_bar_or(bar_id, 64, failed)) break;
            if (lt == 0) {
                // one release of the lane's writes (seen through the barrier), then the signals
                fence_acq_rel_cluster();
#pragma unroll 1
                for (int q = 0; q < VS; ++q) mbar_arrive_cluster_relaxed(mapa_shared(ready + 8 * e, static_cast<uint32_t>(q)));
            }
        }
        // the lane's last load, if it has not been waited for, lands before the CTA exits
        if (lt == 0 && loaded > k) drain_bar(qb, (loaded - 1) & 1);
    } else if (scan_warp_index(warp) >= 0 && scan_warp_index(warp) < NS) {
        // ---------------------------------------------------------------- scan warps
        const int sw = scan_warp_index(warp);
        const int g = lane >> 2, t = lane & 3;
        const int vr0 = rank * (16 * NS) + 16 * sw;
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
        const uint32_t ot = sb + OFF_OT + sw * OT_BYTES;  // this warp's output tile
        // ldmatrix / stmatrix row addresses: lane 8 i + r names row r of 8x8 matrix i, i.e. token
        // r + 8 (i >> 1) of the V-row block 8 (i & 1) of this warp's 16 rows
        const int mtok = (lane & 7) + 8 * (lane >> 4), mcol = 8 * ((lane >> 3) & 1);
        for (int n = 0; n < nch; ++n) {
            const int si = n % NST;
            const bool ok = wait_bar(st_full + 8 * si, (n / NST) & 1, flags);
            if (!__all_sync(0xffffffffu, ok)) break;
            const uint32_t vt = sb + OFF_STG + si * STAGE, pb = vt + RAW_TILE;
            const int tok0 = sp.bos + n * CHUNK;
            const int Lv = min(CHUNK, sp.len - n * CHUNK);

            // Z = S [K*Gamma ; Q*Gamma]^T  (16 rows x 32 columns per warp)
            float z[4][4];
#pragma unroll
            for (int q = 0; q < 4; ++q) z[q][0] = z[q][1] = z[q][2] = z[q][3] = 0.f;
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

            // Off the chain to the next chunk (Z -> R -> E -> S update -> next Z): decay S by gamma
            // now (Z has taken its bf16 copy), and load Kbar, T' and P while Z completes.
#pragma unroll
            for (int nt = 0; nt < 16; ++nt) {
                const float2 gm = SM_AT(const float2, pb + P_GAM + (8 * nt + 2 * t) * 4);
                S[nt][0] *= gm.x;
                S[nt][1] *= gm.y;
                S[nt][2] *= gm.x;
                S[nt][3] *= gm.y;
            }
            uint32_t kbf[8][4], ttf[2][2], ppf[2][2];
            {
                const uint32_t kb = pb + P_KB + (ri + 8 * (mi & 1)) * BZ_LD + 16 * (mi >> 1);
#pragma unroll
                for (int m = 0; m < 8; ++m) ldsm_x4_t(kb + m * 32, kbf[m][0], kbf[m][1], kbf[m][2], kbf[m][3]);
#pragma unroll
                for (int nt = 0; nt < 2; ++nt) {
                    const uint32_t rt = pb + P_TT + (8 * nt + g) * SM_LD + 4 * t, rp = pb + P_PP + (8 * nt + g) * SM_LD + 4 * t;
                    ttf[nt][0] = SM_AT(const uint32_t, rt);
                    ttf[nt][1] = SM_AT(const uint32_t, rt + 16);
                    ppf[nt][0] = SM_AT(const uint32_t, rp);
                    ppf[nt][1] = SM_AT(const uint32_t, rp + 16);
                }
            }

            // R = V^T - Z_k (rows past the chunk's end are zero): V^T in the accumulator layout
            // straight from the swizzled tile, matrix i = V^T rows 8 (i & 1).., tokens 8 (i >> 1)..
            float R[2][4];
            {
                uint32_t vw[4];
                ldsm_x4_t(vt + raw_off(mtok, vr0 + mcol), vw[0], vw[1], vw[2], vw[3]);
#pragma unroll
                for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const int jj = 8 * nt + 2 * t + (q & 1);
                        const uint32_t w = vw[2 * nt + (q >> 1)];
                        const float vv = jj < Lv ? ((q & 1) ? bf16_hi(w) : bf16_lo(w)) : 0.f;
                        R[nt][q] = vv - z[nt][q];
                    }
            }

            // E = R (T diag(beta))^T
            const uint32_t ra[4] = {pack_f16(R[0][0], R[0][1]), pack_f16(R[0][2], R[0][3]), pack_f16(R[1][0], R[1][1]),
                                    pack_f16(R[1][2], R[1][3])};
            float ev[2][4];
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
                ev[nt][0] = ev[nt][1] = ev[nt][2] = ev[nt][3] = 0.f;
                mma_f16(ev[nt], ra, ttf[nt][0], ttf[nt][1]);
            }
            const uint32_t ea[4] = {pack_f16(ev[0][0], ev[0][1]), pack_f16(ev[0][2], ev[0][3]), pack_f16(ev[1][0], ev[1][1]),
                                    pack_f16(ev[1][2], ev[1][3])};

            // S = S Diag(gamma) + E Kbar (the decay above): issued first, the next chunk waits on it
#pragma unroll
            for (int m = 0; m < 8; ++m) {
                mma_f16(S[2 * m], ea, kbf[m][0], kbf[m][1]);
                mma_f16(S[2 * m + 1], ea, kbf[m][2], kbf[m][3]);
            }

            // O = scale (Z_q + E P^T)
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) mma_f16(z[2 + nt], ea, ppf[nt][0], ppf[nt][1]);
            // the 16 x 16 output tile, transposed to [token][V row] in shared memory, then one
            // 16-byte store per lane (token lane / 2, V rows 8 (lane & 1)..)
            stsm_x4_t(ot + mtok * OT_LD + 2 * mcol, pack_bf16(p.scale * z[2][0], p.scale * z[2][1]),
                      pack_bf16(p.scale * z[2][2], p.scale * z[2][3]), pack_bf16(p.scale * z[3][0], p.scale * z[3][1]),
                      pack_bf16(p.scale * z[3][2], p.scale * z[3][3]));
            __syncwarp();
            {
                const int r = lane >> 1, c8 = 8 * (lane & 1);
                const uint4 o = SM_AT(const uint4, ot + r * OT_LD + 2 * c8);
                const size_t oi = (static_cast<size_t>(tok0 + r) * p.H + h) * DH + vr0 + c8;
                if (r < Lv && gmem_ok(oi, 8, out_elems(p))) *reinterpret_cast<uint4 *>(p.out + oi) = o;
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(st_empty + 8 * si);
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
    // no CTA leaves while another CTA of its cluster may still arrive on its barriers
    __syncwarp();  // warp 0's feeder lane ran a loop of its own
    cluster_sync_all();
#undef SM_AT
}

}  // namespace v1s
}  // namespace kda
