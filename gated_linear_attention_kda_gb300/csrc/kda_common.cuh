// kda_common.cuh -- definitions shared by the KDA forward kernels: launch
// parameters, the device error word, bounded mbarrier waits and the layout of
// the TMA-loaded q/k/v/g chunk tiles.
#pragma once
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "kda.h"
#include "ptx.cuh"

namespace kda {

constexpr int CHUNK = 16;
constexpr int DH = 128;  // K = V = 128
constexpr int RAW_TILE = 4096;        // 16 rows x 128 bf16, as two 64-column TMA boxes
constexpr int RAW_BOX = 2048;
constexpr int RAW_STAGE = 4 * RAW_TILE;
constexpr int OFF_Q = 0, OFF_K = RAW_TILE, OFF_V = 2 * RAW_TILE, OFF_G = 3 * RAW_TILE;

constexpr float LOG2E = 1.4426950408889634f;


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
    void *dump;       // slot-dump instance of the tcgen05 kernel only: finished prep slots of CTA 0
    int dump_chunks;  // ... for chunks 0 .. dump_chunks - 1
};

// Bounded wait on an mbarrier phase. Each poll may suspend the thread for up
// to WAIT_HINT_NS (it wakes when the phase completes), so a waiting warp costs
// no issue slots. Gives up when another role has already given up (abort
// flag) or after WAIT_LIMIT polls (a few seconds at most), which flags the
// device error word; the caller then leaves its loop so the CTA terminates.
constexpr uint32_t WAIT_HINT_NS = 20000;
constexpr int WAIT_LIMIT = 1 << 18;

// Slow path of wait_bar, kept out of line: the kernels wait at many sites and
// inlined copies of the loop would crowd the instruction cache. `limit` polls
// (WAIT_LIMIT in the kernels; the wait-timeout probe passes a shorter one).
__device__ __noinline__ bool wait_bar_slow(uint32_t bar, uint32_t parity, volatile int *abort_flag,
                                           int limit = WAIT_LIMIT)
{
#pragma unroll 1
    for (int i = 0; i < limit; ++i) {
        if (mbar_try_wait_sleep(bar, parity, WAIT_HINT_NS)) return true;
        if (*abort_flag) return false;
    }
    atomicOr(&g_dev_error, DEVERR_TIMEOUT);
    *abort_flag = 1;
    return false;
}

__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile int *abort_flag)
{
    if (mbar_try_wait(bar, parity)) return true;
    return wait_bar_slow(bar, parity, abort_flag);
}

// Bounded wait that ignores the abort flag (used to drain in-flight copies).
__device__ __noinline__ void drain_bar(uint32_t bar, uint32_t parity)
{
#pragma unroll 1
    for (int i = 0; i < WAIT_LIMIT; ++i)
        if (mbar_try_wait_sleep(bar, parity, WAIT_HINT_NS)) return;
    atomicOr(&g_dev_error, DEVERR_TIMEOUT);
}

// Sizes (elements) of the call's activation-shaped and state-shaped buffers, for the debug
// build's bounds checks.
__device__ __forceinline__ size_t tokhead_elems(const Params &p) { return static_cast<size_t>(p.total) * p.H; }
__device__ __forceinline__ size_t out_elems(const Params &p) { return tokhead_elems(p) * DH; }
__device__ __forceinline__ size_t state_elems(const Params &p) { return static_cast<size_t>(p.nseq) * p.H * DH * DH; }

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

// Varlen order, longest sequences first: CTA group `rank` (one group per sequence) takes the
// sequence of that rank in decreasing length, ties by index, so the long sequential chains start
// in the first wave. Every warp computes it alone (one pass over cu_seqlens per 32 sequences);
// used for up to 64 sequences, identity beyond. A permutation for any cu_seqlens contents.
constexpr int LPT_MAX_SEQS = 64;
__device__ __forceinline__ int lpt_sequence(const Params &p, int rank)
{
    const int lane = threadIdx.x & 31;
    int found = rank;
    for (int base = 0; base < p.nseq; base += 32) {
        const int i = base + lane;
        const long long li = i < p.nseq ? p.cu[i + 1] - p.cu[i] : -1;
        int r = 0;
        for (int j = 0; j < p.nseq; ++j) {
            const long long lj = p.cu[j + 1] - p.cu[j];
            r += (lj > li) || (lj == li && j < i);
        }
        const unsigned m = __ballot_sync(0xffffffffu, i < p.nseq && r == rank);
        if (m) found = base + __ffs(m) - 1;
    }
    return found;
}

// Byte offset of element (row r, channel c) inside a 16x128 bf16 tile loaded
// as two 64-column boxes with the 128-byte swizzle (16-byte chunk index XOR
// row mod 8).
__device__ __forceinline__ uint32_t raw_off(int r, int c)
{
    return (c >> 6) * RAW_BOX + r * 128 + ((((c & 63) >> 3) ^ (r & 7)) << 4) + (c & 7) * 2;
}

__device__ __forceinline__ uint16_t f2bf_bits(float x) { return __bfloat16_as_ushort(__float2bfloat16_rn(x)); }


}  // namespace kda
