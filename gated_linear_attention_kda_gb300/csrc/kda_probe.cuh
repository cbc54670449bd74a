// kda_probe.cuh -- one 16-token chunk of one head through the element-wise and
// chunk-matrix steps of the forward pass, built from the same device helpers as
// the prep lanes (tanh-form sigmoid, ex2, bf16 factor tiles, the two-product
// chunk products, the unit-lower inverse), so that each step can be checked on
// its own against the fp64 chunk evaluation:
//   G2 (gate in log2 units, inclusive in-chunk cumsum), beta,
//   A = strictly-lower(beta_r sum_c k_r k_j 2^{G2_r - G2_j}), P = lower(sum_c q_r k_j 2^{..}),
//   T = (I + A)^-1.
// "FlashKDA lower_bound Parameter ..." -- "Conversion to the Gate Scale Factor";
// "How FlashKDA's CHUNK Size of 16 ..." -- "Efficient 16x16 Matrix Inversion".
// Test hook only: the forward kernels never call it.
#pragma once
#include "kda_common.cuh"
#include "kda_chunk.cuh"

namespace kda {
namespace probe {

constexpr int LD = 272;  // bytes per row of the [16][136] 16-bit tiles, as in the prep lanes

// q, k, g: one chunk [16][128] bf16 (row-major); beta: [16] bf16 logits; A_log: one float or
// NULL; dt_bias: [128] or NULL; rows >= L are padding (k = 0, beta = 0, no gate).
// Outputs (fp32): G2 [16][128], beta_act [16], A, P, T [16][16].
__global__ void __launch_bounds__(128)
    kda_probe_chunk_kernel(const uint16_t *q, const uint16_t *k, const uint16_t *g, const uint16_t *beta,
                           const float *A_log, const float *dt_bias, float half_gs, int L, float *G2, float *beta_act,
                           float *Aout, float *Pout, float *Tout)
{
    __shared__ __align__(16) uint8_t tiles[4 * 16 * LD];  // Kl, Ql, Kr hi, Kr lo (bf16)
    __shared__ float sbeta[16];
    const int c = threadIdx.x, warp = c >> 5, lane = c & 31;
    const uint32_t kl = smem_u32(tiles), ql = kl + 16 * LD, krh = ql + 16 * LD, krl = krh + 16 * LD;
    // gate: x / 2 = ah2 g + bb with x = exp(A_log) (g + dt_bias); g2 = gate_scale sigma(x)
    const float ah2 = A_log ? 0.5f * ex2_approx(A_log[0] * LOG2E) : 0.5f;
    const float bb = dt_bias ? ah2 * dt_bias[c] : 0.f;
    float Gc[CHUNK], acc = 0.f;
#pragma unroll
    for (int r = 0; r < CHUNK; ++r) {
        const float gx = __uint_as_float(static_cast<uint32_t>(g[r * DH + c]) << 16);
        acc += r < L ? fmaf(half_gs, tanh_approx(fmaf(ah2, gx, bb)), half_gs) : 0.f;
        Gc[r] = acc;
        G2[r * DH + c] = acc;
    }
    if (c < CHUNK) {
        const float b = c < L ? fmaf(0.5f, tanh_approx(0.5f * __uint_as_float(static_cast<uint32_t>(beta[c]) << 16)), 0.5f) : 0.f;
        sbeta[c] = b;
        beta_act[c] = b;
    }
    // factors with the exponent reference at row 7: Kl = K 2^{G - Gm}, Ql = Q 2^{G - Gm}, Kr = K 2^{Gm - G}
    const float gm = Gc[7];
#pragma unroll
    for (int r = 0; r < CHUNK; ++r) {
        const float d = Gc[r] - gm;
        const float u = ex2_approx(d), f = ex2_approx(-d);
        const float kv = r < L ? __uint_as_float(static_cast<uint32_t>(k[r * DH + c]) << 16) : 0.f;
        const float qv = __uint_as_float(static_cast<uint32_t>(q[r * DH + c]) << 16);
        uint32_t hi, lo;
        split_bf16_trunc(kv * f, kv * f, hi, lo);
        const uint32_t o = r * LD + c * 2;
        *reinterpret_cast<uint16_t *>(tiles + o) = static_cast<uint16_t>(pack_bf16(kv * u, 0.f));
        *reinterpret_cast<uint16_t *>(tiles + 16 * LD + o) = static_cast<uint16_t>(pack_bf16(qv * u, 0.f));
        *reinterpret_cast<uint16_t *>(tiles + 32 * LD + o) = static_cast<uint16_t>(hi);
        *reinterpret_cast<uint16_t *>(tiles + 48 * LD + o) = static_cast<uint16_t>(lo);
    }
    __syncthreads();
    if (warp >= 2) return;
    const int gq = lane >> 2, t = lane & 3;
    Frag16 acc16;
    chunk_gram_x2<8>(warp == 0 ? kl : ql, krh, krl, acc16, lane, 0);
    if (warp == 0) {
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int r = gq + 8 * (i >> 1), j = 8 * nt + 2 * t + (i & 1);
                acc16.c[nt][i] = j < r ? acc16.c[nt][i] * sbeta[r] : 0.f;
            }
        Frag16 T;
        unit_lower_inverse(acc16, T, gq, t);
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int r = gq + 8 * (i >> 1), j = 8 * nt + 2 * t + (i & 1);
                Aout[r * CHUNK + j] = acc16.c[nt][i];
                Tout[r * CHUNK + j] = T.c[nt][i];
            }
    } else {
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int r = gq + 8 * (i >> 1), j = 8 * nt + 2 * t + (i & 1);
                Pout[r * CHUNK + j] = j <= r ? acc16.c[nt][i] : 0.f;
            }
    }
}

// The bounded pipeline wait run out on purpose, with nothing left in flight: two lanes each wait
// on an mbarrier that nothing ever arrives on, through the kernels' own slow wait path with
// `polls` polls. Expected: both waits give up (result[0..1] = 0), the first to run out flags
// DEVERR_TIMEOUT in the device error word and sets the CTA's abort flag (result[2] = 1), which
// ends the other wait early; the kernel then returns normally and the context stays usable.
__global__ void __launch_bounds__(64) kda_probe_wait_kernel(int polls, int *result)
{
    __shared__ __align__(8) uint64_t bars[2];
    __shared__ int abort_flag;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bars[0]), 1);
        mbar_init(smem_u32(&bars[1]), 1);
        abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    if (lane == 0) {
        const uint32_t bar = smem_u32(&bars[warp]);
        const bool ok = mbar_try_wait(bar, 0) || wait_bar_slow(bar, 0, &abort_flag, polls);
        result[warp] = ok ? 1 : 0;
    }
    __syncthreads();
    if (threadIdx.x == 0) result[2] = abort_flag;
}

// The bounds checks themselves, with no access made: a shared address 16 bytes past the CTA's
// shared memory and a global index one past the end of a buffer of 10 elements. In the debug
// build both checks fail (result 0) and set DEVERR_BOUNDS; in the product build they compile to
// `true` (result 1) and set nothing.
__global__ void kda_probe_bounds_kernel(int *result)
{
    if (threadIdx.x != 0) return;
    result[0] = smem_ok(dbg_smem_end() + 16, 4) ? 1 : 0;
    result[1] = gmem_ok(10, 1, 10) ? 1 : 0;
}

}  // namespace probe
}  // namespace kda
