// kda_fwd.cu -- fused chunked forward pass of Kimi Delta Attention for GB300
// (sm_103a), and the C ABI declared in include/kda.h.
//
// One CTA owns one (sequence, head) state, or a slice of its V rows when there
// are too few states to fill the machine (the rows of S are independent).
// Whole states run the tcgen05 kernel (kda_fwd_tc.cuh: state in tensor memory,
// state products on the 5th-generation tensor core); V-row slices run the
// warp-MMA kernel (kda_fwd_mma.cuh), whose warp roles are:
//   warp 0        TMA producer: streams the 16-token q/k/v/g tiles of each
//                 chunk into a 6-deep shared-memory ring.
//   warps 1..6    three "prep lanes" of two warps each, taking every third
//                 chunk: gate activation in base 2, in-chunk cumsum, the
//                 exponent-scaled operand tiles, the 16x16 chunk matrix A and
//                 the intra-chunk score matrix P (two bf16 warp-MMA products
//                 per entry), and the unit-lower inverse T = (I + A)^-1 as a
//                 four-factor Neumann product on fp16 warp MMA.
//   warps 7..     scan warps, 16 V rows each, holding their rows of the fp32
//                 state S in registers across the whole sequence. Per chunk:
//                   Z   = S [K*Gamma ; Q*Gamma]^T              (bf16 MMA)
//                   R   = V^T - Z_k,  E = R (T diag(beta))^T   (fp16 MMA)
//                   O   = scale (Z_q + E P^T)                  (fp16 MMA)
//                   S   = S Diag(gamma) + E Kbar               (fp16 MMA)
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
#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <string>

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include "kda.h"
#include "kda_common.cuh"
#include "kda_fwd_mma.cuh"
#include "kda_fwd_mma32.cuh"
#include "kda_fwd_shared.cuh"
#include "kda_fwd_tc.cuh"
#include "kda_probe.cuh"
#include "kda_decode.cuh"

namespace kda {

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

template <int NS, bool QKN>
static cudaError_t launch(int64_t grid, cudaStream_t s, const CUtensorMap &q, const CUtensorMap &k,
                          const CUtensorMap &v, const CUtensorMap &g, const Params &p)
{
    static thread_local int configured_dev = -1;
    int dev = 0;
    cudaGetDevice(&dev);
    if (configured_dev != dev) {
        cudaError_t e =
            cudaFuncSetAttribute(v1::kda_fwd_kernel<NS, QKN>, cudaFuncAttributeMaxDynamicSharedMemorySize, v1::Layout<NS>::SMEM_ALLOC);
        if (e != cudaSuccess) return e;
        configured_dev = dev;
    }
    v1::kda_fwd_kernel<NS, QKN><<<static_cast<unsigned>(grid), v1::Layout<NS>::NTHREADS, v1::Layout<NS>::SMEM_ALLOC, s>>>(q, k, v, g, p);
    return cudaGetLastError();
}

template <bool QKN, bool DUMP = false>
static cudaError_t launch_tc(int64_t grid, cudaStream_t s, const CUtensorMap &q, const CUtensorMap &k,
                             const CUtensorMap &v, const CUtensorMap &g, const Params &p)
{
    static thread_local int configured_dev = -1;
    int dev = 0;
    cudaGetDevice(&dev);
    if (configured_dev != dev) {
        cudaError_t e = cudaFuncSetAttribute(tcs::kda_fwd_tc_kernel<QKN, DUMP>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, tcs::SMEM_ALLOC);
        if (e != cudaSuccess) return e;
        configured_dev = dev;
    }
    tcs::kda_fwd_tc_kernel<QKN, DUMP><<<static_cast<unsigned>(grid), tcs::NTHREADS, tcs::SMEM_ALLOC, s>>>(q, k, v, g, p);
    return cudaGetLastError();
}

template <int NS>
static cudaError_t launch32(int64_t grid, cudaStream_t s, const CUtensorMap &q, const CUtensorMap &k,
                            const CUtensorMap &v, const CUtensorMap &g, const Params &p)
{
    static thread_local int configured_dev = -1;
    int dev = 0;
    cudaGetDevice(&dev);
    if (configured_dev != dev) {
        cudaError_t e =
            cudaFuncSetAttribute(v32::kda_fwd32_kernel<NS>, cudaFuncAttributeMaxDynamicSharedMemorySize, v32::SMEM_ALLOC);
        if (e != cudaSuccess) return e;
        configured_dev = dev;
    }
    v32::kda_fwd32_kernel<NS><<<static_cast<unsigned>(grid), 32 * (1 + 4 * v32::NP + NS), v32::SMEM_ALLOC, s>>>(q, k, v, g, p);
    return cudaGetLastError();
}

// The split-state kernel with shared chunk preparation: one cluster of VS = 8 / NS CTAs per state,
// the prepared operands handed between them through the workspace `ws`.
template <int NS>
static cudaLaunchConfig_t shared_config(int64_t grid, cudaStream_t s, cudaLaunchAttribute *attr)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(v1s::NTHREADS);
    cfg.dynamicSmemBytes = v1s::SMEM_ALLOC;
    cfg.stream = s;
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 8 / NS;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cfg;
}

// Clusters the device holds at once for this instance (0: cannot run), queried once per device.
template <int NS>
static int shared_capacity(int dev)
{
    static std::mutex mu;
    static int cache[256];
    static bool have[256] = {};
    if (dev < 0 || dev >= 256) return 0;
    std::lock_guard<std::mutex> lock(mu);
    if (!have[dev]) {
        int n = 0;
        cudaLaunchAttribute attr[1];
        cudaLaunchConfig_t cfg = shared_config<NS>(8 / NS, nullptr, attr);
        if (cudaFuncSetAttribute(v1s::kda_fwd_shared_kernel<NS>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 v1s::SMEM_ALLOC) != cudaSuccess ||
            cudaOccupancyMaxActiveClusters(&n, v1s::kda_fwd_shared_kernel<NS>, &cfg) != cudaSuccess)
            n = 0;
        cudaGetLastError();  // a refused query leaves no sticky error behind
        cache[dev] = n;
        have[dev] = true;
    }
    return cache[dev];
}

template <int NS>
static cudaError_t launch_shared(int64_t grid, cudaStream_t s, const CUtensorMap &q, const CUtensorMap &k,
                                 const CUtensorMap &v, const CUtensorMap &g, const Params &p, uint8_t *ws)
{
    cudaLaunchAttribute attr[1];
    const cudaLaunchConfig_t cfg = shared_config<NS>(grid, s, attr);
    const cudaError_t e = cudaLaunchKernelEx(&cfg, v1s::kda_fwd_shared_kernel<NS>, q, k, v, g, p, ws);
    return e == cudaSuccess ? cudaGetLastError() : e;
}

static int shared_capacity_for(int vs, int dev)
{
    switch (vs) {
        case 2: return shared_capacity<4>(dev);
        case 4: return shared_capacity<2>(dev);
        case 8: return shared_capacity<1>(dev);
        default: return 0;
    }
}

static cudaError_t launch_split_shared(int vs, int64_t grid, cudaStream_t s, const CUtensorMap &q, const CUtensorMap &k,
                                       const CUtensorMap &v, const CUtensorMap &g, const Params &p, uint8_t *ws)
{
    switch (vs) {
        case 2: return launch_shared<4>(grid, s, q, k, v, g, p, ws);
        case 4: return launch_shared<2>(grid, s, q, k, v, g, p, ws);
        default: return launch_shared<1>(grid, s, q, k, v, g, p, ws);
    }
}

// 32-token chunks (KDA_FLAG_CHUNK32): the warp-MMA kernel at every split, 128 / split V rows per CTA
static cudaError_t launch_split32(int vs, int64_t grid, cudaStream_t s, const CUtensorMap &q, const CUtensorMap &k,
                                  const CUtensorMap &v, const CUtensorMap &g, const Params &p)
{
    switch (vs) {
        case 1: return launch32<8>(grid, s, q, k, v, g, p);
        case 2: return launch32<4>(grid, s, q, k, v, g, p);
        case 4: return launch32<2>(grid, s, q, k, v, g, p);
        default: return launch32<1>(grid, s, q, k, v, g, p);
    }
}

template <bool QKN>
static cudaError_t launch_split(int vs, int64_t grid, cudaStream_t s, const CUtensorMap &q, const CUtensorMap &k,
                                const CUtensorMap &v, const CUtensorMap &g, const Params &p)
{
    switch (vs) {
        case 1: return launch_tc<QKN>(grid, s, q, k, v, g, p);
        case 2: return launch<4, QKN>(grid, s, q, k, v, g, p);
        case 4: return launch<2, QKN>(grid, s, q, k, v, g, p);
        default: return launch<1, QKN>(grid, s, q, k, v, g, p);
    }
}

static bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

// Per-device resources of kda_fwd_host, created on its first call on a device and kept until exit:
// a memory pool whose staging allocations stay mapped between calls (release threshold at its
// maximum), the streams and events of the pieces of a call, and pinned room for the rebased
// sequence bounds of each piece. Calls of kda_fwd_host on one device are serialised by `mu`.
constexpr int HOST_PIECES = 4;
constexpr int HOST_CU_MAX = 1 << 16;  // sequences per piece
struct HostLane {
    std::mutex mu;
    cudaMemPool_t pool = nullptr;
    cudaStream_t streams[HOST_PIECES] = {};
    cudaEvent_t start = nullptr, done[HOST_PIECES] = {};
    int64_t *cu_host = nullptr;
};

static HostLane *host_lane(int dev, cudaError_t *err)
{
    static std::mutex mu;
    static HostLane *lanes[256] = {};
    if (dev < 0 || dev >= 256) {
        *err = cudaErrorInvalidDevice;
        return nullptr;
    }
    std::lock_guard<std::mutex> lock(mu);
    if (lanes[dev]) {
        *err = cudaSuccess;
        return lanes[dev];
    }
    HostLane *hl = new HostLane;
    cudaMemPoolProps props = {};
    props.allocType = cudaMemAllocationTypePinned;
    props.location.type = cudaMemLocationTypeDevice;
    props.location.id = dev;
    cudaError_t e = cudaMemPoolCreate(&hl->pool, &props);
    if (e == cudaSuccess) {
        uint64_t keep = UINT64_MAX;
        e = cudaMemPoolSetAttribute(hl->pool, cudaMemPoolAttrReleaseThreshold, &keep);
    }
    for (int i = 0; i < HOST_PIECES && e == cudaSuccess; ++i) e = cudaStreamCreateWithFlags(&hl->streams[i], cudaStreamNonBlocking);
    for (int i = 0; i < HOST_PIECES && e == cudaSuccess; ++i) e = cudaEventCreateWithFlags(&hl->done[i], cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&hl->start, cudaEventDisableTiming);
    if (e == cudaSuccess)
        e = cudaMallocHost(reinterpret_cast<void **>(&hl->cu_host), sizeof(int64_t) * HOST_PIECES * (HOST_CU_MAX + 1));
    *err = e;
    if (e != cudaSuccess) return nullptr;  // partially created resources are left to process exit
    lanes[dev] = hl;
    return hl;
}

// Snapshot of the device error word, taken and cleared in one atomic step by status_take_kernel.
__device__ unsigned int g_dev_error_seen;

__global__ void status_take_kernel() { g_dev_error_seen = atomicExch(&g_dev_error, 0u); }

// An empty call (no tokens): every cu_seqlens entry must be 0, since cu[0] = 0 and cu[N] = B * T = 0.
__global__ void empty_seqlens_check_kernel(const int64_t *cu, int n)
{
    for (int i = threadIdx.x; i < n; i += blockDim.x)
        if (cu[i] != 0) atomicOr(&g_dev_error, DEVERR_SEQLENS);
}

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

// kda_fwd_ex with an optional split of the V rows (`split_vs` 1, 2, 4 or 8; 0 = planned, or the
// KDA_V_SPLIT override): kda_fwd_host runs the pieces of one call with the split of the whole call,
// so its results equal kda_fwd's bit for bit.
static kda_status fwd_impl(const void *q, const void *k, const void *v, const void *g, const void *beta, float scale,
                           void *out, const float *A_log, const float *dt_bias, float lower_bound,
                           const void *initial_state, kda_dtype initial_dtype, void *final_state, kda_dtype final_dtype,
                           const int64_t *cu_seqlens, int64_t N, int64_t B, int64_t T, int64_t H, int64_t K, int64_t V,
                           uint32_t flags, void *stream, int split_vs, void *dump = nullptr, int dump_chunks = 0,
                           void *ws = nullptr, size_t ws_bytes = 0)
{
    t_last_error.clear();
    constexpr uint32_t known = KDA_FLAG_QK_L2NORM | KDA_FLAG_CHUNK32;
    if (flags & ~known) return fail(KDA_ERR_RANGE, "unknown option bits 0x%x", flags & ~known);
    if ((flags & KDA_FLAG_CHUNK32) && (flags & KDA_FLAG_QK_L2NORM))
        return fail(KDA_ERR_RANGE, "KDA_FLAG_CHUNK32 does not combine with KDA_FLAG_QK_L2NORM");
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
    // KDA_V_SPLIT (1, 2, 4 or 8) overrides the planned split of each state's V rows, for tuning and tests
    int force_vs = split_vs;
    if (const char *env = std::getenv("KDA_V_SPLIT"); env && !split_vs) {
        force_vs = std::atoi(env);
        if (force_vs != 1 && force_vs != 2 && force_vs != 4 && force_vs != 8)
            return fail(KDA_ERR_RANGE, "KDA_V_SPLIT must be 1, 2, 4 or 8 (got '%s')", env);
    }

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (total == 0) {
        // No tokens: nothing to launch the forward kernels for. Every sequence is empty, so the
        // final state is the initial state (or zero); only cu_seqlens is still checked.
        cudaError_t e = cudaSuccess;
        if (cu_seqlens) {
            empty_seqlens_check_kernel<<<1, 256, 0, s>>>(cu_seqlens, static_cast<int>(N + 1));
            e = cudaGetLastError();
        }
        const size_t fin_bytes = static_cast<size_t>(nseq * H) * DH * DH * (final_dtype == KDA_DTYPE_FP32 ? 4 : 2);
        if (e == cudaSuccess && final_state && initial_state && initial_state != final_state)
            e = cudaMemcpyAsync(final_state, initial_state, fin_bytes, cudaMemcpyDeviceToDevice, s);
        else if (e == cudaSuccess && final_state && !initial_state)
            e = cudaMemsetAsync(final_state, 0, fin_bytes, s);
        if (e != cudaSuccess) return fail(KDA_ERR_LAUNCH, "empty call: %s", cudaGetErrorString(e));
        return KDA_OK;
    }

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
    p.dump = dump;
    p.dump_chunks = dump_chunks;
    int vs;
    int64_t grid;
    plan(nseq * H, nsm, &vs, &grid);
    if (force_vs) {
        vs = force_vs;
        grid = nseq * H * vs;
    }
    p.vsplit = vs;
    // split states with a workspace: the chunk preparation is shared by a state's CTAs
    const bool shared = ws && vs >= 2 && !dump && !(flags & (KDA_FLAG_CHUNK32 | KDA_FLAG_QK_L2NORM)) &&
                        shared_capacity_for(vs, dev) > 0;
    if (shared && static_cast<int64_t>(ws_bytes) < nseq * H * v1s::workspace_bytes_per_state())
        return fail(KDA_ERR_RANGE, "workspace of %zu bytes is smaller than the %lld this call needs", ws_bytes,
                    (long long)(nseq * H * v1s::workspace_bytes_per_state()));
    if (dump)
        ce = launch_tc<false, true>(grid, s, mq, mk, mv, mg, p);  // the per-step probe (split 1)
    else if (shared)
        ce = launch_split_shared(vs, grid, s, mq, mk, mv, mg, p, static_cast<uint8_t *>(ws));
    else if (flags & KDA_FLAG_CHUNK32)
        ce = launch_split32(vs, grid, s, mq, mk, mv, mg, p);
    else
        ce = (flags & KDA_FLAG_QK_L2NORM) ? launch_split<true>(vs, grid, s, mq, mk, mv, mg, p)
                                          : launch_split<false>(vs, grid, s, mq, mk, mv, mg, p);
    if (ce != cudaSuccess) return fail(KDA_ERR_LAUNCH, "kernel launch failed: %s", cudaGetErrorString(ce));
    return KDA_OK;
}

KDA_API kda_status kda_fwd_ex(const void *q, const void *k, const void *v, const void *g, const void *beta,
                              float scale, void *out, const float *A_log, const float *dt_bias, float lower_bound,
                              const void *initial_state, kda_dtype initial_dtype, void *final_state,
                              kda_dtype final_dtype, const int64_t *cu_seqlens, int64_t N, int64_t B, int64_t T,
                              int64_t H, int64_t K, int64_t V, uint32_t flags, void *stream)
{
    return fwd_impl(q, k, v, g, beta, scale, out, A_log, dt_bias, lower_bound, initial_state, initial_dtype, final_state,
                    final_dtype, cu_seqlens, N, B, T, H, K, V, flags, stream, 0);
}

KDA_API kda_status kda_fwd(const void *q, const void *k, const void *v, const void *g, const void *beta, float scale,
                           void *out, const float *A_log, const float *dt_bias, float lower_bound,
                           const void *initial_state, kda_dtype initial_dtype, void *final_state,
                           kda_dtype final_dtype, const int64_t *cu_seqlens, int64_t N, int64_t B, int64_t T,
                           int64_t H, int64_t K, int64_t V, void *stream)
{
    return kda_fwd_ex(q, k, v, g, beta, scale, out, A_log, dt_bias, lower_bound, initial_state, initial_dtype,
                      final_state, final_dtype, cu_seqlens, N, B, T, H, K, V, 0u, stream);
}

KDA_API kda_status kda_fwd_flat(const void *q, const void *k, const void *v, const void *g, const void *beta,
                                float scale, void *out, const float *A_log, const float *dt_bias, float lower_bound,
                                const void *initial_state, kda_dtype initial_dtype, void *final_state,
                                kda_dtype final_dtype, const int64_t *cu_seqlens, int64_t N, int64_t B, int64_t T,
                                int64_t H, int64_t K, int64_t V, void *stream)
{
    return kda_fwd(q, k, v, g, beta, scale, out, A_log, dt_bias, lower_bound, initial_state, initial_dtype,
                   final_state, final_dtype, cu_seqlens, N, B, T, H, K, V, stream);
}

KDA_API kda_status kda_fwd_packed(const kda_fwd_args *a, void *stream)
{
    if (!a) return fail(KDA_ERR_NULL, "kda_fwd_packed: NULL argument struct");
    return kda_fwd_ex(a->q, a->k, a->v, a->g, a->beta, a->scale, a->out, a->A_log, a->dt_bias, a->lower_bound,
                      a->initial_state, a->initial_dtype, a->final_state, a->final_dtype, a->cu_seqlens, a->N, a->B,
                      a->T, a->H, a->K, a->V, a->flags, stream);
}

KDA_API kda_status kda_decode_ex(const void *q, const void *k, const void *v, const void *g, const void *beta,
                                 float scale, void *out, const float *A_log, const float *dt_bias, float lower_bound,
                                 void *state, kda_dtype state_dtype, int64_t S, int64_t H, int64_t K, int64_t V,
                                 uint32_t flags, void *stream)
{
    t_last_error.clear();
    if (flags & ~KDA_FLAG_QK_L2NORM) return fail(KDA_ERR_RANGE, "unknown option bits 0x%x", flags & ~KDA_FLAG_QK_L2NORM);
    if (K != DH || V != DH) return fail(KDA_ERR_SHAPE, "K and V must be 128 (got K=%lld V=%lld)", (long long)K, (long long)V);
    if (S < 1 || H < 1 || S * H > (int64_t(1) << 28))
        return fail(KDA_ERR_SHAPE, "bad sizes S=%lld H=%lld", (long long)S, (long long)H);
    if (!q || !k || !v || !g || !beta || !out || !state)
        return fail(KDA_ERR_NULL, "q, k, v, g, beta, out and state are required");
    if (state_dtype != KDA_DTYPE_BF16 && state_dtype != KDA_DTYPE_FP32)
        return fail(KDA_ERR_DTYPE, "state dtype must be BF16 or FP32");
    if (!std::isfinite(lower_bound) || lower_bound < -5.f || lower_bound > 0.f)
        return fail(KDA_ERR_RANGE, "lower_bound must lie in [-5, 0] (got %g)", (double)lower_bound);
    if (!std::isfinite(scale)) return fail(KDA_ERR_RANGE, "scale must be finite");
    if (!aligned(q, 8) || !aligned(k, 8) || !aligned(g, 8) || !aligned(v, 2) || !aligned(beta, 2) || !aligned(out, 2) ||
        !aligned(state, 16) || (A_log && !aligned(A_log, 4)) || (dt_bias && !aligned(dt_bias, 4)))
        return fail(KDA_ERR_ALIGN, "q, k, g need 8-byte, state 16-byte and the others natural alignment");
    dec::DecodeParams p;
    p.q = static_cast<const uint16_t *>(q);
    p.k = static_cast<const uint16_t *>(k);
    p.v = static_cast<const uint16_t *>(v);
    p.g = static_cast<const uint16_t *>(g);
    p.beta = static_cast<const uint16_t *>(beta);
    p.out = static_cast<uint16_t *>(out);
    p.A_log = A_log;
    p.dt_bias = dt_bias;
    p.state = state;
    p.state_dtype = state_dtype;
    p.H = static_cast<int>(H);
    p.scale = scale;
    p.lower_bound = lower_bound;
    // one contiguous range of state rows per warp; enough CTAs to fill every SM, but no fewer than
    // eight rows per warp
    int dev = 0, nsm = 0;
    cudaError_t ce = cudaGetDevice(&dev);
    if (ce == cudaSuccess) ce = cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
    if (ce != cudaSuccess) return fail(KDA_ERR_LAUNCH, "CUDA device query failed: %s", cudaGetErrorString(ce));
    // resident CTAs per SM of the instance about to run (registers decide), queried once per device
    static thread_local int occ_dev = -1, occ[2] = {0, 0};
    if (occ_dev != dev) {
        ce = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ[0], dec::kda_decode_kernel<false>, dec::THREADS, 0);
        if (ce == cudaSuccess) ce = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ[1], dec::kda_decode_kernel<true>, dec::THREADS, 0);
        if (ce != cudaSuccess) return fail(KDA_ERR_LAUNCH, "occupancy query failed: %s", cudaGetErrorString(ce));
        occ_dev = dev;
    }
    const int per_sm = std::max(1, occ[(flags & KDA_FLAG_QK_L2NORM) ? 1 : 0]);
    const long long nrows = static_cast<long long>(S) * H * DH;
    const long long rows_per_cta = 8LL * (dec::THREADS / 32);
    const long long grid = std::min<long long>(static_cast<long long>(nsm) * per_sm, (nrows + rows_per_cta - 1) / rows_per_cta);
    if (flags & KDA_FLAG_QK_L2NORM)
        dec::kda_decode_kernel<true><<<static_cast<unsigned>(grid), dec::THREADS, 0, static_cast<cudaStream_t>(stream)>>>(p, nrows);
    else
        dec::kda_decode_kernel<false><<<static_cast<unsigned>(grid), dec::THREADS, 0, static_cast<cudaStream_t>(stream)>>>(p, nrows);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fail(KDA_ERR_LAUNCH, "decode launch failed: %s", cudaGetErrorString(e));
    return KDA_OK;
}

KDA_API kda_status kda_decode(const void *q, const void *k, const void *v, const void *g, const void *beta, float scale,
                              void *out, const float *A_log, const float *dt_bias, float lower_bound, void *state,
                              kda_dtype state_dtype, int64_t S, int64_t H, int64_t K, int64_t V, void *stream)
{
    return kda_decode_ex(q, k, v, g, beta, scale, out, A_log, dt_bias, lower_bound, state, state_dtype, S, H, K, V, 0u,
                         stream);
}

KDA_API kda_status kda_probe_chunk(const void *q, const void *k, const void *g, const void *beta, const float *A_log,
                                   const float *dt_bias, float lower_bound, int rows, float *G2, float *beta_act,
                                   float *A, float *P, float *T, void *stream)
{
    t_last_error.clear();
    if (!q || !k || !g || !beta || !G2 || !beta_act || !A || !P || !T)
        return fail(KDA_ERR_NULL, "kda_probe_chunk: q, k, g, beta and every output are required");
    if (rows < 1 || rows > CHUNK) return fail(KDA_ERR_SHAPE, "kda_probe_chunk: rows must lie in 1..16 (got %d)", rows);
    if (!std::isfinite(lower_bound) || lower_bound < -5.f || lower_bound > 0.f)
        return fail(KDA_ERR_RANGE, "lower_bound must lie in [-5, 0] (got %g)", (double)lower_bound);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    probe::kda_probe_chunk_kernel<<<1, 128, 0, s>>>(
        static_cast<const uint16_t *>(q), static_cast<const uint16_t *>(k), static_cast<const uint16_t *>(g),
        static_cast<const uint16_t *>(beta), A_log, dt_bias, 0.5f * kda_gate_scale(lower_bound), rows, G2, beta_act, A,
        P, T);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fail(KDA_ERR_LAUNCH, "probe launch failed: %s", cudaGetErrorString(e));
    return KDA_OK;
}

KDA_API kda_status kda_probe_wait_timeout(int polls, int *result, void *stream)
{
    t_last_error.clear();
    if (!result) return fail(KDA_ERR_NULL, "kda_probe_wait_timeout: result is required");
    if (polls < 1 || polls > WAIT_LIMIT)
        return fail(KDA_ERR_RANGE, "kda_probe_wait_timeout: polls must lie in 1..%d (got %d)", WAIT_LIMIT, polls);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    probe::kda_probe_wait_kernel<<<1, 64, 0, s>>>(polls, result);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fail(KDA_ERR_LAUNCH, "probe launch failed: %s", cudaGetErrorString(e));
    return KDA_OK;
}

KDA_API int kda_debug_build(void) { return kDebugChecks ? 1 : 0; }

KDA_API kda_status kda_fwd_workspace_bytes(int64_t states, int64_t H, uint32_t flags, size_t *bytes)
{
    t_last_error.clear();
    if (!bytes) return fail(KDA_ERR_NULL, "kda_fwd_workspace_bytes: bytes is required");
    if (states < 0 || H < 1) return fail(KDA_ERR_SHAPE, "bad sizes states=%lld H=%lld", (long long)states, (long long)H);
    int dev = 0, nsm = 0;
    cudaError_t ce = cudaGetDevice(&dev);
    if (ce == cudaSuccess) ce = cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
    if (ce != cudaSuccess) return fail(KDA_ERR_LAUNCH, "CUDA device query failed: %s", cudaGetErrorString(ce));
    int vs;
    int64_t grid;
    plan(states * H, nsm, &vs, &grid);
    if (const char *env = std::getenv("KDA_V_SPLIT")) {
        const int f = std::atoi(env);
        if (f == 1 || f == 2 || f == 4 || f == 8) vs = f;
    }
    const bool shared =
        vs >= 2 && !(flags & (KDA_FLAG_CHUNK32 | KDA_FLAG_QK_L2NORM)) && shared_capacity_for(vs, dev) > 0;
    *bytes = shared ? static_cast<size_t>(states * H * v1s::workspace_bytes_per_state()) : 0;
    return KDA_OK;
}

KDA_API kda_status kda_fwd_ws(const void *q, const void *k, const void *v, const void *g, const void *beta, float scale,
                              void *out, const float *A_log, const float *dt_bias, float lower_bound,
                              const void *initial_state, kda_dtype initial_dtype, void *final_state,
                              kda_dtype final_dtype, const int64_t *cu_seqlens, int64_t N, int64_t B, int64_t T,
                              int64_t H, int64_t K, int64_t V, uint32_t flags, void *workspace, size_t workspace_bytes,
                              void *stream)
{
    t_last_error.clear();
    if (workspace && !aligned(workspace, 16)) return fail(KDA_ERR_ALIGN, "workspace must be 16-byte aligned");
    return fwd_impl(q, k, v, g, beta, scale, out, A_log, dt_bias, lower_bound, initial_state, initial_dtype, final_state,
                    final_dtype, cu_seqlens, N, B, T, H, K, V, flags, stream, 0, nullptr, 0, workspace, workspace_bytes);
}

// ---------------------------------------------------------------------------------------------
// kda_fwd_static: kda_fwd_ws with a scratch array of the library's own (no allocation per call).
// Room for KDA_STATIC_SCRATCH_STATES states: the plan splits a state only when states x 2 fit on
// the SMs, at most 76 on a 152-SM GB300.
static __device__ __align__(256) uint8_t g_static_scratch[KDA_STATIC_SCRATCH_STATES * 16 * v1s::PREP_SLOT];
static_assert(KDA_STATIC_SCRATCH_STATES * 16 * v1s::PREP_SLOT == KDA_STATIC_SCRATCH_STATES * v1s::workspace_bytes_per_state(),
              "the static scratch holds KDA_STATIC_SCRATCH_STATES workspaces");

// The scratch array's device address on the current device, looked up once per device.
static kda_status static_scratch(void **ptr)
{
    static std::mutex mu;
    static void *addr[256];
    static bool have[256] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail(KDA_ERR_LAUNCH, "CUDA device query failed: %s", cudaGetErrorString(e));
    if (dev < 0 || dev >= 256) return fail(KDA_ERR_LAUNCH, "device ordinal %d out of range", dev);
    std::lock_guard<std::mutex> lock(mu);
    if (!have[dev]) {
        e = cudaGetSymbolAddress(&addr[dev], g_static_scratch);
        if (e != cudaSuccess) return fail(KDA_ERR_LAUNCH, "static scratch lookup failed: %s", cudaGetErrorString(e));
        have[dev] = true;
    }
    *ptr = addr[dev];
    return KDA_OK;
}

KDA_API kda_status kda_fwd_static(const void *q, const void *k, const void *v, const void *g, const void *beta,
                                  float scale, void *out, const float *A_log, const float *dt_bias, float lower_bound,
                                  const void *initial_state, kda_dtype initial_dtype, void *final_state,
                                  kda_dtype final_dtype, const int64_t *cu_seqlens, int64_t N, int64_t B, int64_t T,
                                  int64_t H, int64_t K, int64_t V, uint32_t flags, void *stream)
{
    t_last_error.clear();
    const int64_t nseq = cu_seqlens ? N : B;
    const bool sizes_ok = K == DH && V == DH && B >= 1 && T >= 0 && H >= 1 && H <= (1 << 20) &&
                          (!cu_seqlens || (B == 1 && N >= 1)) && nseq * H <= (int64_t(1) << 28);
    size_t need = 0;
    if (sizes_ok && B * T > 0 && kda_fwd_workspace_bytes(nseq, H, flags, &need) == KDA_OK && need > 0) {
        if (need > sizeof(g_static_scratch))
            return fail(KDA_ERR_RANGE,
                        "kda_fwd_static: %lld states need %zu bytes of scratch; the static scratch holds %d states "
                        "(%zu bytes): use kda_fwd_ws with a workspace",
                        (long long)(nseq * H), need, KDA_STATIC_SCRATCH_STATES, sizeof(g_static_scratch));
        void *ws = nullptr;
        if (const kda_status st = static_scratch(&ws); st != KDA_OK) return st;
        return fwd_impl(q, k, v, g, beta, scale, out, A_log, dt_bias, lower_bound, initial_state, initial_dtype,
                        final_state, final_dtype, cu_seqlens, N, B, T, H, K, V, flags, stream, 0, nullptr, 0, ws,
                        sizeof(g_static_scratch));
    }
    // no scratch needed (or an argument error, reported as kda_fwd_ex reports it)
    t_last_error.clear();
    return fwd_impl(q, k, v, g, beta, scale, out, A_log, dt_bias, lower_bound, initial_state, initial_dtype, final_state,
                    final_dtype, cu_seqlens, N, B, T, H, K, V, flags, stream, 0, nullptr, 0, nullptr, 0);
}

KDA_API int kda_probe_slot_bytes(void) { return tcs::SLOT; }

KDA_API kda_status kda_probe_slots(const void *q, const void *k, const void *v, const void *g, const void *beta,
                                   float scale, void *out, const float *A_log, const float *dt_bias, float lower_bound,
                                   int64_t T, void *dump, int nchunks, void *stream)
{
    t_last_error.clear();
    if (!dump) return fail(KDA_ERR_NULL, "kda_probe_slots: dump is required");
    if (T < 1 || nchunks < 1 || nchunks > (T + CHUNK - 1) / CHUNK)
        return fail(KDA_ERR_SHAPE, "kda_probe_slots: need T >= 1 and 1 <= nchunks <= ceil(T / 16) (T=%lld nchunks=%d)",
                    (long long)T, nchunks);
    if (!aligned(dump, 16)) return fail(KDA_ERR_ALIGN, "kda_probe_slots: dump must be 16-byte aligned");
    return fwd_impl(q, k, v, g, beta, scale, out, A_log, dt_bias, lower_bound, nullptr, KDA_DTYPE_NONE, nullptr,
                    KDA_DTYPE_NONE, nullptr, 0, 1, T, 1, DH, DH, 0, stream, 1, dump, nchunks);
}

KDA_API kda_status kda_probe_bounds(int *result, void *stream)
{
    t_last_error.clear();
    if (!result) return fail(KDA_ERR_NULL, "kda_probe_bounds: result is required");
    probe::kda_probe_bounds_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(result);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fail(KDA_ERR_LAUNCH, "probe launch failed: %s", cudaGetErrorString(e));
    return KDA_OK;
}

KDA_API kda_status kda_check_device_status(void *stream)
{
    t_last_error.clear();
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    unsigned int word = 0;
    // one thread exchanges the word with 0 (read and clear in one atomic step, so a bit that a
    // kernel on another stream sets meanwhile is kept for the next check), then the snapshot is
    // copied back behind it on the same stream
    status_take_kernel<<<1, 1, 0, s>>>();
    cudaError_t e = cudaGetLastError();
    if (e == cudaSuccess) e = cudaMemcpyFromSymbolAsync(&word, g_dev_error_seen, sizeof word, 0, cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return fail(KDA_ERR_LAUNCH, "reading the device status failed: %s", cudaGetErrorString(e));
    if (word)
        return fail(KDA_ERR_DEVICE, "device error word 0x%x:%s%s%s", word, (word & DEVERR_SEQLENS) ? " bad cu_seqlens" : "",
                    (word & DEVERR_TIMEOUT) ? " pipeline wait timed out" : "",
                    (word & DEVERR_BOUNDS) ? " out-of-bounds access caught (debug build)" : "");
    return KDA_OK;
}

KDA_API kda_status kda_fwd_host(const void *q, const void *k, const void *v, const void *g, const void *beta,
                                float scale, void *out, const float *A_log, const float *dt_bias, float lower_bound,
                                const void *initial_state, kda_dtype initial_dtype, void *final_state,
                                kda_dtype final_dtype, const int64_t *cu_seqlens, int64_t N, int64_t B, int64_t T,
                                int64_t H, int64_t K, int64_t V, void *stream)
{
    t_last_error.clear();
    if (K != DH || V != DH || B < 1 || T < 0 || H < 1 || (cu_seqlens && (N < 1 || B != 1)))
        return fail(KDA_ERR_SHAPE, "bad sizes");
    if (cu_seqlens)  // the host copy of the sequence bounds is read here to cut the call into pieces
        for (int64_t i = 0; i < N; ++i)
            if (cu_seqlens[i] < 0 || cu_seqlens[i + 1] < cu_seqlens[i] || cu_seqlens[i + 1] > T || cu_seqlens[0] != 0 ||
                cu_seqlens[N] != T)
                return fail(KDA_ERR_SHAPE, "cu_seqlens must rise from 0 to T");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int dev = 0, nsm = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
    HostLane *hl = e == cudaSuccess ? host_lane(dev, &e) : nullptr;
    if (!hl) return fail(KDA_ERR_LAUNCH, "staging set-up failed: %s", cudaGetErrorString(e));
    std::lock_guard<std::mutex> call_lock(hl->mu);
    const int64_t total = B * T, nseq = cu_seqlens ? N : B;
    const size_t act = static_cast<size_t>(total) * H * DH * 2, bet = static_cast<size_t>(total) * H * 2;
    const size_t sti = initial_state ? (initial_dtype == KDA_DTYPE_FP32 ? 4 : 2) : 0;
    const size_t sto = final_state ? (final_dtype == KDA_DTYPE_FP32 ? 4 : 2) : 0;
    const size_t st_row = static_cast<size_t>(H) * DH * DH;  // state elements per sequence
    const size_t cub = cu_seqlens ? static_cast<size_t>(N + 1 + HOST_PIECES) * 8 : 0;  // each piece's rebased bounds
    const size_t al = A_log ? static_cast<size_t>(H) * 4 : 0, db = dt_bias ? static_cast<size_t>(H) * DH * 4 : 0;
    auto up = [](size_t x) { return (x + 255) & ~size_t(255); };
    const size_t sizes[] = {act, act, act, act, bet, act, al, db, nseq * st_row * sti, nseq * st_row * sto, cub};
    size_t off[11], tot = 0;
    for (int i = 0; i < 11; ++i) {
        off[i] = tot;
        tot += up(sizes[i]);
    }
    // the whole call's V-row split, used by every piece (identical kernels, identical results)
    int vs = 1;
    int64_t grid = 0;
    plan(nseq * H, nsm, &vs, &grid);
    if (const char *env = std::getenv("KDA_V_SPLIT")) {  // a bad value is reported by the forward call itself
        const int ev = std::atoi(env);
        vs = (ev == 1 || ev == 2 || ev == 4 || ev == 8) ? ev : 0;
    }
    // pieces: groups of batch rows (or of sequences, by token count), each on its own stream, so the
    // copies of one piece overlap the kernel and copies of the others
    int np = static_cast<int>(nseq < HOST_PIECES ? nseq : HOST_PIECES);
    if (total == 0) np = 1;
    int64_t first[HOST_PIECES + 1];  // first batch row / sequence of each piece
    first[0] = 0;
    for (int i = 1; i < np; ++i) {
        if (!cu_seqlens) {
            first[i] = nseq * i / np;
        } else {  // the first sequence that starts at or after i / np of the tokens
            int64_t j = first[i - 1] + 1;
            while (j < nseq - (np - i) && cu_seqlens[j] * np < total * i) ++j;
            first[i] = j;
        }
    }
    first[np] = nseq;
    uint8_t *d = nullptr;
    e = cudaMallocFromPoolAsync(reinterpret_cast<void **>(&d), tot ? tot : 256, hl->pool, s);
    if (e != cudaSuccess) return fail(KDA_ERR_LAUNCH, "device staging allocation failed: %s", cudaGetErrorString(e));
    if (al) e = cudaMemcpyAsync(d + off[6], A_log, al, cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess && db) e = cudaMemcpyAsync(d + off[7], dt_bias, db, cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess) e = cudaEventRecord(hl->start, s);
    kda_status st = KDA_OK;
    for (int pi = 0; pi < np && e == cudaSuccess && st == KDA_OK; ++pi) {
        cudaStream_t ps = hl->streams[pi];
        const int64_t s0 = first[pi], s1 = first[pi + 1];
        const int64_t t0 = cu_seqlens ? cu_seqlens[s0] : s0 * T, t1 = cu_seqlens ? cu_seqlens[s1] : s1 * T;
        const size_t ao = static_cast<size_t>(t0) * H * DH * 2, an = static_cast<size_t>(t1 - t0) * H * DH * 2;
        const size_t bo = static_cast<size_t>(t0) * H * 2, bn = static_cast<size_t>(t1 - t0) * H * 2;
        e = cudaStreamWaitEvent(ps, hl->start, 0);
        const void *src[4] = {q, k, v, g};
        for (int i = 0; i < 4 && e == cudaSuccess; ++i)
            if (an) e = cudaMemcpyAsync(d + off[i] + ao, static_cast<const uint8_t *>(src[i]) + ao, an, cudaMemcpyHostToDevice, ps);
        if (e == cudaSuccess && bn)
            e = cudaMemcpyAsync(d + off[4] + bo, static_cast<const uint8_t *>(beta) + bo, bn, cudaMemcpyHostToDevice, ps);
        if (e == cudaSuccess && sti)
            e = cudaMemcpyAsync(d + off[8] + s0 * st_row * sti, static_cast<const uint8_t *>(initial_state) + s0 * st_row * sti,
                                (s1 - s0) * st_row * sti, cudaMemcpyHostToDevice, ps);
        const int64_t *dcu = nullptr;
        if (e == cudaSuccess && cu_seqlens) {  // this piece's bounds, rebased to its first token
            int64_t *host_cu = hl->cu_host + pi * (HOST_CU_MAX + 1);
            if (s1 - s0 > HOST_CU_MAX) {
                st = fail(KDA_ERR_SHAPE, "kda_fwd_host: at most %d sequences per piece", HOST_CU_MAX);
                break;
            }
            for (int64_t i = s0; i <= s1; ++i) host_cu[i - s0] = cu_seqlens[i] - t0;
            dcu = reinterpret_cast<const int64_t *>(d + off[10]) + s0 + pi;  // entries [s0 + pi, s1 + pi]
            e = cudaMemcpyAsync(const_cast<int64_t *>(dcu), host_cu, (s1 - s0 + 1) * 8, cudaMemcpyHostToDevice, ps);
        }
        if (e != cudaSuccess) break;
        const int64_t pB = cu_seqlens ? 1 : s1 - s0, pT = cu_seqlens ? t1 - t0 : T;
        st = fwd_impl(d + off[0] + ao, d + off[1] + ao, d + off[2] + ao, d + off[3] + ao, d + off[4] + bo, scale,
                      d + off[5] + ao, A_log ? reinterpret_cast<const float *>(d + off[6]) : nullptr,
                      dt_bias ? reinterpret_cast<const float *>(d + off[7]) : nullptr, lower_bound,
                      initial_state ? d + off[8] + s0 * st_row * sti : nullptr, initial_dtype,
                      final_state ? d + off[9] + s0 * st_row * sto : nullptr, final_dtype, dcu, s1 - s0, pB, pT, H, K, V, 0u,
                      ps, vs);
        if (st != KDA_OK) break;
        if (an) e = cudaMemcpyAsync(static_cast<uint8_t *>(out) + ao, d + off[5] + ao, an, cudaMemcpyDeviceToHost, ps);
        if (e == cudaSuccess && sto)
            e = cudaMemcpyAsync(static_cast<uint8_t *>(final_state) + s0 * st_row * sto, d + off[9] + s0 * st_row * sto,
                                (s1 - s0) * st_row * sto, cudaMemcpyDeviceToHost, ps);
        if (e == cudaSuccess) e = cudaEventRecord(hl->done[pi], ps);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(s, hl->done[pi], 0);
    }
    if (e != cudaSuccess && st == KDA_OK) st = fail(KDA_ERR_LAUNCH, "staging copy failed: %s", cudaGetErrorString(e));
    // the caller's stream waits for every piece (also after a failure, before the memory is freed)
    for (int pi = 0; pi < np; ++pi) {
        cudaEventRecord(hl->done[pi], hl->streams[pi]);
        cudaStreamWaitEvent(s, hl->done[pi], 0);
    }
    cudaFreeAsync(d, s);
    cudaError_t se = cudaStreamSynchronize(s);
    if (st == KDA_OK && se != cudaSuccess) st = fail(KDA_ERR_LAUNCH, "stream synchronize failed: %s", cudaGetErrorString(se));
    return st;
}

}  // extern "C"
