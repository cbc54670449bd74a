// kda_decode.cuh -- one token of KDA per (sequence, head) against a state kept in
// place: the recurrent step next to the chunked forward pass ("FlashKDA Input
// Tensor Shapes and DTypes ..." -- "Initial and Final States": the state carried
// from one call to the next).
//   a[c] = lower_bound sigmoid(exp(A_log[h]) (g[c] + dt_bias[h, c])),  beta = sigmoid(logit)
//   S <- S Diag(exp(a)),  p = S k,  S <- S + beta (v - p) k^T,  o = scale S q
// Bandwidth-bound (the state is read and written once per token). The S * H * 128 state rows
// are cut into one contiguous range per warp of a grid that fills the machine, so every warp
// streams the same number of rows (no partial last wave); a row's 128 channels are spread over
// the 32 lanes (four each, one 16-byte access), its two dot products are warp reductions, and a
// warp keeps four rows' loads in flight. The per-(sequence, head) terms (decay, key, query, beta)
// are formed again where a warp's range enters the next head. All arithmetic in fp32; a bf16
// state is widened on load and rounded to nearest on store.
#pragma once
#include "kda_common.cuh"

namespace kda {
namespace dec {

constexpr int THREADS = 128;       // 4 warps
constexpr int ROW_BATCH = 4;       // rows of one warp in flight

struct DecodeParams {
    const uint16_t *q, *k, *v, *g, *beta;  // bf16 [S, H, 128] ([S, H] for beta)
    uint16_t *out;                          // bf16 [S, H, 128]
    const float *A_log, *dt_bias;           // [H], [H, 128] or NULL
    void *state;                            // [S, H, 128 (V), 128 (K)], fp32 or bf16, in place
    int state_dtype;
    int H;
    float scale, lower_bound;
};

__device__ __forceinline__ float bf16_to_f(uint16_t x) { return __uint_as_float(static_cast<uint32_t>(x) << 16); }
__device__ __forceinline__ float sigmoid_f(float x) { return 1.f / (1.f + expf(-x)); }

// QKN: L2-normalise q and k before use (KDA_FLAG_QK_L2NORM).
template <bool QKN>
__global__ void __launch_bounds__(THREADS) kda_decode_kernel(const DecodeParams p, long long nrows)
{
    const int lane = threadIdx.x & 31;
    const long long nw = static_cast<long long>(gridDim.x) * (THREADS / 32);
    const long long w = static_cast<long long>(blockIdx.x) * (THREADS / 32) + (threadIdx.x >> 5);
    long long r = w * nrows / nw;                  // this warp's rows [r, r_end)
    const long long r_end = (w + 1) * nrows / nw;
    const int c0 = 4 * lane;
    while (r < r_end) {
        const long long unit = r / DH;             // (sequence, head)
        const int h = static_cast<int>(unit % p.H);
        const size_t tok = static_cast<size_t>(unit) * DH;  // [S, H, 128] offset of this (sequence, head)
        // this lane's four channels: decay, key, query
        const float ea = p.A_log ? expf(p.A_log[h]) : 1.f;
        float alpha[4], kk[4], qq[4];
        {
            const uint2 gw = *reinterpret_cast<const uint2 *>(p.g + tok + c0);
            const uint2 kw = *reinterpret_cast<const uint2 *>(p.k + tok + c0);
            const uint2 qw = *reinterpret_cast<const uint2 *>(p.q + tok + c0);
            const uint16_t gs[4] = {static_cast<uint16_t>(gw.x), static_cast<uint16_t>(gw.x >> 16),
                                    static_cast<uint16_t>(gw.y), static_cast<uint16_t>(gw.y >> 16)};
            const uint16_t ks[4] = {static_cast<uint16_t>(kw.x), static_cast<uint16_t>(kw.x >> 16),
                                    static_cast<uint16_t>(kw.y), static_cast<uint16_t>(kw.y >> 16)};
            const uint16_t qs[4] = {static_cast<uint16_t>(qw.x), static_cast<uint16_t>(qw.x >> 16),
                                    static_cast<uint16_t>(qw.y), static_cast<uint16_t>(qw.y >> 16)};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float b = p.dt_bias ? p.dt_bias[static_cast<size_t>(h) * DH + c0 + j] : 0.f;
                alpha[j] = expf(p.lower_bound * sigmoid_f(ea * (bf16_to_f(gs[j]) + b)));
                kk[j] = bf16_to_f(ks[j]);
                qq[j] = bf16_to_f(qs[j]);
            }
        }
        if constexpr (QKN) {  // x / sqrt(sum x^2 + 1e-6): the warp holds all 128 channels
            float sk = 0.f, sq = 0.f;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                sk = fmaf(kk[j], kk[j], sk);
                sq = fmaf(qq[j], qq[j], sq);
            }
#pragma unroll
            for (int m = 16; m >= 1; m >>= 1) {
                sk += __shfl_xor_sync(0xffffffffu, sk, m);
                sq += __shfl_xor_sync(0xffffffffu, sq, m);
            }
            const float fk = rsqrtf(sk + 1e-6f), fq = rsqrtf(sq + 1e-6f);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                kk[j] *= fk;
                qq[j] *= fq;
            }
        }
        const float beta = sigmoid_f(bf16_to_f(p.beta[unit]));
        const long long unit_end = r_end < (unit + 1) * DH ? r_end : (unit + 1) * DH;
        for (; r < unit_end; r += ROW_BATCH) {
            // up to ROW_BATCH rows of this head: all loads first, then the updates and stores
            float s[ROW_BATCH][4], vv[ROW_BATCH];
#pragma unroll
            for (int b = 0; b < ROW_BATCH; ++b) {
                s[b][0] = s[b][1] = s[b][2] = s[b][3] = 0.f;
                vv[b] = 0.f;
                if (r + b < unit_end) {
                    const int vr = static_cast<int>(r + b - unit * DH);
                    const size_t so = static_cast<size_t>(r + b) * DH + c0;
                    if (p.state_dtype == KDA_DTYPE_FP32) {
                        const float4 w4 = *reinterpret_cast<const float4 *>(static_cast<const float *>(p.state) + so);
                        s[b][0] = w4.x; s[b][1] = w4.y; s[b][2] = w4.z; s[b][3] = w4.w;
                    } else {
                        const uint2 w2 = *reinterpret_cast<const uint2 *>(static_cast<const uint16_t *>(p.state) + so);
                        s[b][0] = __uint_as_float(w2.x << 16); s[b][1] = __uint_as_float(w2.x & 0xffff0000u);
                        s[b][2] = __uint_as_float(w2.y << 16); s[b][3] = __uint_as_float(w2.y & 0xffff0000u);
                    }
                    vv[b] = bf16_to_f(p.v[tok + vr]);
                }
            }
#pragma unroll
            for (int b = 0; b < ROW_BATCH; ++b) {
                if (r + b >= unit_end) break;  // warp-uniform
                const int vr = static_cast<int>(r + b - unit * DH);
                const size_t so = static_cast<size_t>(r + b) * DH + c0;
                float pk = 0.f;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    s[b][j] *= alpha[j];
                    pk = fmaf(s[b][j], kk[j], pk);
                }
#pragma unroll
                for (int m = 16; m >= 1; m >>= 1) pk += __shfl_xor_sync(0xffffffffu, pk, m);
                const float wgt = beta * (vv[b] - pk);
                float o = 0.f;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    s[b][j] = fmaf(wgt, kk[j], s[b][j]);
                    o = fmaf(s[b][j], qq[j], o);
                }
#pragma unroll
                for (int m = 16; m >= 1; m >>= 1) o += __shfl_xor_sync(0xffffffffu, o, m);
                if (p.state_dtype == KDA_DTYPE_FP32) {
                    *reinterpret_cast<float4 *>(static_cast<float *>(p.state) + so) = make_float4(s[b][0], s[b][1], s[b][2], s[b][3]);
                } else {
                    *reinterpret_cast<uint2 *>(static_cast<uint16_t *>(p.state) + so) =
                        make_uint2(pack_bf16(s[b][0], s[b][1]), pack_bf16(s[b][2], s[b][3]));
                }
                if (lane == 0) p.out[tok + vr] = f2bf_bits(p.scale * o);
            }
        }
    }
}

}  // namespace dec
}  // namespace kda
