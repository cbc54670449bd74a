/*
 * kda.h -- C ABI of the KDA (Kimi Delta Attention) chunked forward pass for
 * GB300 (sm_103a). One shared library, libkda.so; plain pointers and sizes,
 * no framework types.
 *
 * The operation. For every sequence and head, with state S (V x K, stored
 * row-major [v][k]) and per token t:
 *
 *   a_t[c]  = lower_bound * sigmoid(exp(A_log[h]) * (g_t[c] + dt_bias[h,c]))
 *             (A_log NULL: factor 1; dt_bias NULL: bias 0)
 *   beta_t  = sigmoid(beta logit_t)
 *   S_t     = S_{t-1} Diag(exp(a_t)) (I - beta_t k_t k_t^T) + beta_t v_t k_t^T
 *   out_t   = scale * S_t q_t
 *
 * Sources (page title -- section):
 *  [LB]     "FlashKDA lower_bound Parameter: Controlling Exponentiation
 *           Precision in Selective State Space Models": "Conversion to the
 *           Gate Scale Factor" (gate_scale = lower_bound * log2(e)), "How does
 *           lower_bound interact with dt_bias?" (the gate), "Can lower_bound
 *           be positive?".
 *  [EX2]    "Base-2 Exponent Optimization in FlashKDA: How It Works and
 *           Performance Benefits": "Re-basing the Gate Activation".
 *  [CHUNK]  "How FlashKDA's CHUNK Size of 16 Improves Numerical Stability
 *           Over CHUNK 64": "Efficient 16x16 Matrix Inversion" (16-token
 *           chunks, the unit-lower chunk matrix and its inverse).
 *  [SHAPES] "FlashKDA Input Tensor Shapes and DTypes: Complete Specification
 *           for the Forward Pass": "Query, Key, and Value Tensors", "Gating
 *           Tensors and Output Buffer", "Global Scaling Factor", "Gating
 *           Parameters and Constraints", "Initial and Final States",
 *           "Variable-Length Mode", "Memory Layout and Hardware Requirements".
 * The pages name the method but do not print the state update; the update
 * above is the gated delta rule with a per-channel decay, the published
 * definition of KDA. How A_log enters the gate is not stated on the pages;
 * exp(A_log[h]) multiplying the biased gate is the reading adopted here.
 *
 * Ownership and execution. The caller owns every buffer; all pointers below
 * are DEVICE pointers except where noted. kda_fwd allocates no device memory,
 * keeps no per-call state, never synchronises, and runs asynchronously on the
 * caller's stream. Inputs are never modified. `out` is written in place
 * [SHAPES "Gating Tensors and Output Buffer"]. kda_fwd, kda_fwd_ex,
 * kda_fwd_packed and kda_decode(_ex) can be captured into a CUDA graph once
 * the same entry point has run eagerly on the device (the first call sets up
 * per-device kernel attributes on the host); kda_fwd_host and
 * kda_check_device_status synchronise and cannot.
 */
#ifndef KDA_H
#define KDA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define KDA_API __attribute__((visibility("default")))
#else
#define KDA_API
#endif

/* Status codes. Every entry point returns one; nothing aborts the process. */
typedef enum kda_status {
    KDA_OK = 0,
    KDA_ERR_NULL = 1,            /* a required pointer is NULL */
    KDA_ERR_SHAPE = 2,           /* K or V != 128, B/T/H/N out of range, varlen with B != 1 */
    KDA_ERR_DTYPE = 3,           /* unsupported state dtype code */
    KDA_ERR_RANGE = 4,           /* lower_bound outside [-5, 0] or not finite; scale not finite */
    KDA_ERR_STATE_MISMATCH = 5,  /* initial/final state dtypes differ, or buffers overlap partially */
    KDA_ERR_ALIGN = 6,           /* a pointer is not aligned as required */
    KDA_ERR_LAUNCH = 7,          /* a CUDA call failed; see kda_last_error() */
    KDA_ERR_DEVICE = 8           /* the device reported an error (kda_check_device_status) */
} kda_status;

/* Element type of the optional recurrent states [SHAPES "Initial and Final States"]. */
typedef enum kda_dtype {
    KDA_DTYPE_NONE = 0,          /* buffer absent (pointer must be NULL) */
    KDA_DTYPE_BF16 = 1,
    KDA_DTYPE_FP32 = 2
} kda_dtype;

/*
 * Option bits of kda_fwd_ex, kda_decode_ex and kda_fwd_args.flags (0 selects
 * the plain behaviour of kda_fwd / kda_decode).
 *   KDA_FLAG_QK_L2NORM  L2-normalise every (token, head) vector of q and k
 *                       inside the kernel before it is used:
 *                         x[c] <- x[c] / sqrt(sum_c' x[c']^2 + 1e-6)
 *                       in fp32 from the bf16 inputs (the inputs are not
 *                       modified). The pages do not say whether q and k arrive
 *                       normalised; without this bit they are used as given.
 *   KDA_FLAG_CHUNK32    run the forward pass with 32-token chunks (the
 *                       warp-MMA kernel at the planned split of the V rows,
 *                       the exponent reference after the chunk's 16th token,
 *                       the 32x32 inverse from two 16x16 blocks) instead of
 *                       CHUNK = 16: the chunk-size ablation of [CHUNK] "Why
 *                       CHUNK Size Determines Numerical Stability". Results
 *                       agree with the CHUNK = 16 path within the stated
 *                       tolerance, not bit for bit. Forward entry points
 *                       with option bits only (kda_fwd_ex, kda_fwd_packed);
 *                       with KDA_FLAG_QK_L2NORM, or in kda_decode_ex, it is
 *                       KDA_ERR_RANGE.
 * Any other bit is KDA_ERR_RANGE.
 */
#define KDA_FLAG_QK_L2NORM 1u
#define KDA_FLAG_CHUNK32 2u

/*
 * kda_fwd -- the chunked KDA forward pass (CHUNK = 16 [CHUNK]).
 *
 * Tensors (all row-major, contiguous, DEVICE memory):
 *   q, k, g   bf16  [B, T, H, K]        queries, keys, gate pre-activations (16-byte aligned)
 *   v         bf16  [B, T, H, V]        values (16-byte aligned)
 *   beta      bf16  [B, T, H]           beta logits (sigmoid applied inside)
 *   out       bf16  [B, T, H, V]        written for every token (16-byte aligned)
 *   A_log     fp32  [H]     or NULL     per-head log gate parameter
 *   dt_bias   fp32  [H, K]  or NULL     gate bias
 *   initial_state  [S, H, V, K] or NULL, dtype initial_dtype (S = B, or N)
 *   final_state    [S, H, V, K] or NULL, dtype final_dtype; receives the
 *                  state after each sequence's last token. It may be the
 *                  same buffer as initial_state (in-place update); partial
 *                  overlap is rejected. States are 16-byte aligned.
 *   cu_seqlens int64 [N+1] or NULL      varlen mode: B must be 1, T is the
 *                  packed length, sequence i spans tokens
 *                  [cu_seqlens[i], cu_seqlens[i+1]) [SHAPES "Variable-Length
 *                  Mode"]. Entries are read on the device only; a sequence
 *                  outside [0, T] or with a decreasing bound is skipped and
 *                  flags KDA_ERR_DEVICE for kda_check_device_status().
 * Scalars:
 *   scale        multiplies the output [SHAPES "Global Scaling Factor"].
 *   lower_bound  must lie in [-5, 0] [SHAPES "Gating Parameters and
 *                Constraints"]; the kernel uses gate_scale = lower_bound *
 *                log2(e) with base-2 exponentials [LB, EX2].
 *   B, T, H      batch, tokens per batch row (packed length in varlen), heads.
 *   K, V         head dimensions; both must be 128 [SHAPES "Memory Layout
 *                and Hardware Requirements"].
 *   N            number of sequences in varlen mode (>= 1); ignored otherwise.
 *   stream       a cudaStream_t (NULL = legacy default stream).
 * A state absent from the call is zero (initial) or not written (final).
 * A call with no tokens (B * T == 0) launches no forward kernel: final_state
 * (if given) receives initial_state, or zeros; in varlen mode every
 * cu_seqlens entry must then be 0, and a nonzero one flags KDA_ERR_DEVICE.
 * Returns KDA_OK once the work is enqueued. Argument errors are detected on
 * the host before anything is launched and leave every buffer untouched.
 * The environment variable KDA_V_SPLIT (1, 2, 4 or 8), when set, overrides the
 * planned split of each state's V rows across CTAs (kda_plan); any other value
 * is KDA_ERR_RANGE. Results do not depend on the split beyond rounding order.
 */
KDA_API kda_status kda_fwd(const void *q, const void *k, const void *v, const void *g,
                           const void *beta, float scale, void *out,
                           const float *A_log, const float *dt_bias, float lower_bound,
                           const void *initial_state, kda_dtype initial_dtype,
                           void *final_state, kda_dtype final_dtype,
                           const int64_t *cu_seqlens, int64_t N,
                           int64_t B, int64_t T, int64_t H, int64_t K, int64_t V,
                           void *stream);

/*
 * kda_fwd_flat -- the same call as kda_fwd under a second name, for callers
 * that pair it with the argument-struct form below.
 */
KDA_API kda_status kda_fwd_flat(const void *q, const void *k, const void *v, const void *g,
                                const void *beta, float scale, void *out,
                                const float *A_log, const float *dt_bias, float lower_bound,
                                const void *initial_state, kda_dtype initial_dtype,
                                void *final_state, kda_dtype final_dtype,
                                const int64_t *cu_seqlens, int64_t N,
                                int64_t B, int64_t T, int64_t H, int64_t K, int64_t V,
                                void *stream);

/*
 * kda_fwd_ex -- kda_fwd with option bits (`flags`, see KDA_FLAG_QK_L2NORM);
 * every other argument, check and error is kda_fwd's. flags == 0 is kda_fwd.
 */
KDA_API kda_status kda_fwd_ex(const void *q, const void *k, const void *v, const void *g,
                              const void *beta, float scale, void *out,
                              const float *A_log, const float *dt_bias, float lower_bound,
                              const void *initial_state, kda_dtype initial_dtype,
                              void *final_state, kda_dtype final_dtype,
                              const int64_t *cu_seqlens, int64_t N,
                              int64_t B, int64_t T, int64_t H, int64_t K, int64_t V,
                              uint32_t flags, void *stream);

/*
 * kda_fwd_ws -- kda_fwd_ex with a caller-owned DEVICE workspace that lets the
 * CTAs of a split state share the chunk preparation [CHUNK "Algorithm
 * Overview": gate, cumsum, intra-chunk matrices and their inverse, made once per
 * chunk]. When the plan splits a state's V rows across 2, 4 or 8 CTAs (kda_plan
 * or KDA_V_SPLIT) and flags == 0, those CTAs run as one thread-block cluster:
 * each prepares one chunk in `split`, publishes the prepared operands to
 * `workspace`, and reads the others' back through L2. Results equal kda_fwd_ex's
 * bit for bit.
 *   workspace        16-byte aligned device buffer of at least the
 *                    kda_fwd_workspace_bytes bytes for (N or B) x H states;
 *                    NULL (or a call that does not split, or any flag set, or
 *                    a device that cannot hold one cluster of the split's
 *                    size) runs kda_fwd_ex's kernels.
 *                    The contents need no initialisation and are scratch
 *                    after the call; calls that overlap in time must not share
 *                    a workspace.
 *   workspace_bytes  its size; smaller than needed is KDA_ERR_RANGE,
 *                    misaligned KDA_ERR_ALIGN.
 * Every other argument, check and error is kda_fwd_ex's. The library
 * allocates nothing.
 */
KDA_API kda_status kda_fwd_ws(const void *q, const void *k, const void *v, const void *g,
                              const void *beta, float scale, void *out,
                              const float *A_log, const float *dt_bias, float lower_bound,
                              const void *initial_state, kda_dtype initial_dtype,
                              void *final_state, kda_dtype final_dtype,
                              const int64_t *cu_seqlens, int64_t N,
                              int64_t B, int64_t T, int64_t H, int64_t K, int64_t V,
                              uint32_t flags, void *workspace, size_t workspace_bytes,
                              void *stream);

/*
 * kda_fwd_workspace_bytes -- the workspace kda_fwd_ws needs for `states`
 * sequences (N in varlen mode, else B) of H heads with option bits `flags` on
 * the current device: states x H x 16 prepared chunks of 15104 bytes when
 * kda_fwd_ws would share the preparation (the plan splits the state, no flag
 * is set and the device holds a cluster of the split's size), else 0. Needs a CUDA device (it reads the SM count);
 * KDA_ERR_NULL for a NULL `bytes`, KDA_ERR_SHAPE for states < 0 or H < 1.
 */
KDA_API kda_status kda_fwd_workspace_bytes(int64_t states, int64_t H, uint32_t flags, size_t *bytes);

/*
 * kda_fwd_static -- kda_fwd_ws with the library's own scratch instead of a
 * caller's workspace. The pages have no counterpart: it exists so that a
 * caller who cannot hand over device memory still gets the shared chunk
 * preparation, without any allocation. Arguments, checks and errors are
 * kda_fwd_ex's, plus:
 *   - the scratch is one file-scope device array of KDA_STATIC_SCRATCH_STATES
 *     workspaces (KDA_STATIC_SCRATCH_STATES x 16 x 15104 bytes = 18.4 MiB),
 *     part of the library's device image: no call allocates, frees or calls
 *     an allocating library function;
 *   - a call that would share the preparation for more than
 *     KDA_STATIC_SCRATCH_STATES (N or B) x H states is KDA_ERR_RANGE, with a
 *     message naming the limit; a call whose plan does not split the state
 *     (or with option bits set) uses no scratch and has no limit;
 *   - nothing in the scratch needs to start at zero: every entry is written
 *     before it is read within a call;
 *   - the first call on each device looks up the scratch array's device
 *     address (cudaGetSymbolAddress) and sets the kernel attributes on the
 *     host; later calls reuse them;
 *   - calls that overlap in time on one device (on different streams, or
 *     from several host threads) share the scratch and race: serialise them,
 *     for example by issuing them on one stream.
 */
#define KDA_STATIC_SCRATCH_STATES 80
KDA_API kda_status kda_fwd_static(const void *q, const void *k, const void *v, const void *g,
                                  const void *beta, float scale, void *out,
                                  const float *A_log, const float *dt_bias, float lower_bound,
                                  const void *initial_state, kda_dtype initial_dtype,
                                  void *final_state, kda_dtype final_dtype,
                                  const int64_t *cu_seqlens, int64_t N,
                                  int64_t B, int64_t T, int64_t H, int64_t K, int64_t V,
                                  uint32_t flags, void *stream);

/*
 * kda_fwd_args / kda_fwd_packed -- the same operation with its arguments in
 * one struct. Every field has the meaning, layout and ownership of the
 * kda_fwd argument of the same name; the struct itself is read during the
 * call only and may be reused or freed when it returns. A NULL `a` returns
 * KDA_ERR_NULL; every other check and error is kda_fwd's.
 */
typedef struct kda_fwd_args {
    const void *q, *k, *v, *g, *beta; /* bf16 [B, T, H, 128] / beta bf16 [B, T, H] */
    void *out;                         /* bf16 [B, T, H, 128], written */
    const float *A_log;                /* fp32 [H] or NULL */
    const float *dt_bias;              /* fp32 [H, 128] or NULL */
    const void *initial_state;         /* [B|N, H, 128, 128] or NULL */
    void *final_state;                 /* [B|N, H, 128, 128] or NULL, written */
    const int64_t *cu_seqlens;         /* int64 [N + 1] or NULL */
    kda_dtype initial_dtype, final_dtype;
    float scale, lower_bound;
    int64_t N, B, T, H, K, V;
    uint32_t flags;                    /* KDA_FLAG_* bits, as kda_fwd_ex; 0 for kda_fwd */
} kda_fwd_args;

KDA_API kda_status kda_fwd_packed(const kda_fwd_args *a, void *stream);

/*
 * kda_fwd_host -- the same operation on HOST buffers (same layouts and
 * arguments as kda_fwd, every pointer a host pointer; pinned memory gives
 * the fastest copies). It stages the inputs in device memory, runs the
 * forward pass, copies `out` and `final_state` back and synchronises
 * `stream` before it returns: the end-to-end entry point for callers whose
 * tensors live in host memory.
 *   The call is cut into up to four pieces -- groups of batch rows, or in
 * varlen mode groups of whole sequences of about equal token count -- each on
 * a stream of its own, so that the host-to-device copy of one piece overlaps
 * the kernel and the device-to-host copy of the others. Every piece uses the
 * V-row split planned for the whole call, so the results equal kda_fwd's bit
 * for bit. In varlen mode cu_seqlens is a host array here; it must rise from
 * 0 to T (else KDA_ERR_SHAPE before anything is copied).
 *   On its first call on a device it creates, and keeps until the process
 * exits, a stream-ordered memory pool for the staging buffers (they stay
 * mapped between calls), four streams and five events, and a small pinned
 * host buffer; calls on one device are serialised. Work already queued on
 * `stream` is ordered before the call, and the call's work before later work
 * on `stream`.
 */
KDA_API kda_status kda_fwd_host(const void *q, const void *k, const void *v, const void *g,
                                const void *beta, float scale, void *out,
                                const float *A_log, const float *dt_bias, float lower_bound,
                                const void *initial_state, kda_dtype initial_dtype,
                                void *final_state, kda_dtype final_dtype,
                                const int64_t *cu_seqlens, int64_t N,
                                int64_t B, int64_t T, int64_t H, int64_t K, int64_t V,
                                void *stream);

/*
 * kda_decode -- one token per (sequence, head) against a state updated in
 * place: the recurrent step that continues a chunked forward pass (its state
 * is kda_fwd's final_state) ["FlashKDA Input Tensor Shapes and DTypes ..." --
 * "Initial and Final States": the state carried between calls]. For each of
 * the S sequences and H heads, with the same gate, beta and scale as kda_fwd:
 *   S <- S Diag(exp(a)) (I - beta k k^T) + beta v k^T,   out = scale S q.
 *   q, k, v, g   bf16 [S, H, 128] (DEVICE; kda_fwd's [B, T, H, 128] with T = 1).
 *   beta         bf16 [S, H] logits.  out  bf16 [S, H, 128], written.
 *   A_log        fp32 [H] or NULL;    dt_bias  fp32 [H, 128] or NULL.
 *   state        [S, H, 128 (v), 128 (k)] in state_dtype (BF16 or FP32), read
 *                and written in place (the caller owns it).
 * All arithmetic is fp32 (exact sigmoid and exponential); a bf16 state is
 * rounded to nearest even when stored. Allocates nothing; asynchronous on
 * `stream`. Errors as kda_fwd: KDA_ERR_SHAPE (K or V != 128, S or H < 1),
 * KDA_ERR_NULL, KDA_ERR_DTYPE, KDA_ERR_RANGE, KDA_ERR_ALIGN (q, k, g 8-byte,
 * state 16-byte), KDA_ERR_LAUNCH.
 */
KDA_API kda_status kda_decode(const void *q, const void *k, const void *v, const void *g,
                              const void *beta, float scale, void *out,
                              const float *A_log, const float *dt_bias, float lower_bound,
                              void *state, kda_dtype state_dtype,
                              int64_t S, int64_t H, int64_t K, int64_t V, void *stream);

/*
 * kda_decode_ex -- kda_decode with option bits (`flags`, see
 * KDA_FLAG_QK_L2NORM); everything else is kda_decode's.
 */
KDA_API kda_status kda_decode_ex(const void *q, const void *k, const void *v, const void *g,
                                 const void *beta, float scale, void *out,
                                 const float *A_log, const float *dt_bias, float lower_bound,
                                 void *state, kda_dtype state_dtype,
                                 int64_t S, int64_t H, int64_t K, int64_t V, uint32_t flags,
                                 void *stream);

/*
 * kda_probe_chunk -- test hook: one 16-token chunk of one head through the
 * forward pass's per-chunk steps, built from the same device code as the
 * kernels, so that each step can be checked on its own.
 *   q, k, g      one chunk, bf16 [16][128] row-major (DEVICE); rows >= `rows`
 *                are padding (k = 0, beta = 0, no gate).
 *   beta         bf16 [16] logits (DEVICE).
 *   A_log        one fp32 (DEVICE) or NULL; dt_bias fp32 [128] (DEVICE) or NULL.
 *   lower_bound  in [-5, 0]; rows in 1..16.
 * Outputs (DEVICE fp32, written): G2 [16][128] gate in log2 units with its
 * inclusive in-chunk cumsum [LB "Conversion to the Gate Scale Factor"];
 * beta_act [16]; A [16][16] = beta_r sum_c k_r k_j 2^{G2_r - G2_j} for j < r
 * (else 0); P [16][16] = sum_c q_r k_j 2^{G2_r - G2_j} for j <= r (else 0);
 * T [16][16] = (I + A)^-1 [CHUNK "Efficient 16x16 Matrix Inversion"].
 * Asynchronous on `stream`; KDA_ERR_NULL / _SHAPE / _RANGE / _LAUNCH as kda_fwd.
 */
KDA_API kda_status kda_probe_chunk(const void *q, const void *k, const void *g, const void *beta,
                                   const float *A_log, const float *dt_bias, float lower_bound, int rows,
                                   float *G2, float *beta_act, float *A, float *P, float *T, void *stream);

/*
 * kda_probe_wait_timeout -- test hook for the kernels' bounded pipeline waits.
 * One CTA whose two waiting lanes each wait on a shared-memory mbarrier that
 * nothing ever arrives on, through the same slow wait path as the forward
 * kernels, giving up after `polls` polls (1 .. 2^18; each poll suspends the
 * thread for at most 20 us). The first wait to give up sets
 * KDA_ERR_DEVICE's timeout bit in the device error word (read and cleared
 * by kda_check_device_status) and the CTA's abort flag, which ends the other
 * wait. `result` (DEVICE int[3], written): result[0], result[1] = 1 if that
 * wait succeeded (never expected), result[2] = the abort flag (1 expected).
 * No copy or other work is in flight when the waits give up, so the kernel
 * returns normally and the context stays usable. The pages have no
 * counterpart: this checks the build's own failure path. Asynchronous on
 * `stream`; KDA_ERR_NULL for a NULL result, KDA_ERR_RANGE for `polls`
 * outside its range, KDA_ERR_LAUNCH for a failed launch.
 */
KDA_API kda_status kda_probe_wait_timeout(int polls, int *result, void *stream);

/*
 * kda_debug_build -- 1 in the bounds-checked build of the library
 * (libkda_debug.so, compiled with KDA_DEBUG), 0 in the product build. In the
 * checked build every shared-memory, tensor-memory, TMA and global access of
 * the forward kernels is checked first; an access outside its buffer is
 * skipped and sets the out-of-bounds bit of the device error word, reported
 * as KDA_ERR_DEVICE by kda_check_device_status. Host only.
 */
KDA_API int kda_debug_build(void);

/*
 * kda_probe_bounds -- test hook for those checks, making no access: one
 * thread checks a shared address 16 bytes past its CTA's shared memory and
 * a global index one past the end of a 10-element buffer. `result` (DEVICE
 * int[2], written): 1 where the check passed. Checked build: {0, 0} and the
 * out-of-bounds bit set; product build: {1, 1} and nothing set. No
 * counterpart on the pages. Asynchronous on `stream`; KDA_ERR_NULL for a NULL
 * result, KDA_ERR_LAUNCH for a failed launch.
 */
KDA_API kda_status kda_probe_bounds(int *result, void *stream);

/*
 * kda_probe_slots -- test hook: the per-step operands of the tcgen05 kernel
 * itself. One head (B = H = 1) of T tokens (q, k, v, g bf16 [T, 1, 128],
 * beta bf16 [T, 1], out bf16 [T, 1, 128], A_log one fp32 or NULL, dt_bias
 * fp32 [128] or NULL; DEVICE; no states) runs through the tcgen05 kernel
 * (one CTA holding the whole state), and the prep slot of each chunk
 * n < nchunks is copied, as the tensor core reads it, to `dump` + n *
 * kda_probe_slot_bytes() (DEVICE, 16-byte aligned, written). Slot layout
 * (byte offsets; "cm16" = 8x8 core matrices of 16-bit values, K-major,
 * 128 B between K blocks and 256 B between N blocks; "cm32" = 8x4 core
 * matrices of fp32, 128 B between K blocks, 1024 B between N blocks;
 * "sw128" = rows of 128 B, 16-byte chunk index XOR row mod 8, as TMA's
 * 128-byte swizzle):
 *     0  Z' bf16 [32 rows][128]: rows 0-15 K Gamma, 16-31 Q Gamma, both
 *        times gamma of the previous chunk; two 64-column blocks of 4 KB,
 *        sw128
 *  8192  V f16 [16 tokens][128], two 64-column blocks of 2 KB, sw128
 * 12288  Kbar f16 [16][128] = K 2^(G_end - G), same layout as V
 * 16384  Phi fp32 [32][32] = [[-T', 0], [-s M, s I]], cm32
 * 20480  TM f16 [32][16] = [T' ; s M], cm16 (T' = (I + A)^-1 diag(beta),
 *        M = P T', s = scale)
 * 21504  (H Phi^T)^T f16 [32][16] with H = Kbar_{n-1} [K Gamma ; Q Gamma]^T,
 *        cm16 (chunk 0: not used by the kernel)
 * 22528  H''^T f16 [32][16] with H'' = Kbar_{n-2} Diag(gamma_{n-1})
 *        [K Gamma ; Q Gamma]^T, cm16 (chunks 0, 1: not used)
 * 23552  gamma fp32 [128] = 2^(G_end)
 * (G: the gate's in-chunk inclusive cumsum in log2 units; Gamma = 2^G.)
 * No counterpart on the pages: it checks the kernel's own steps. Asynchronous
 * on `stream`; argument checks and errors as kda_fwd, plus KDA_ERR_NULL for a
 * NULL dump, KDA_ERR_SHAPE for nchunks outside 1..ceil(T / 16).
 */
KDA_API kda_status kda_probe_slots(const void *q, const void *k, const void *v, const void *g,
                                   const void *beta, float scale, void *out,
                                   const float *A_log, const float *dt_bias, float lower_bound,
                                   int64_t T, void *dump, int nchunks, void *stream);

/* Bytes of one dumped prep slot of kda_probe_slots. Host only. */
KDA_API int kda_probe_slot_bytes(void);

/* gate_scale = lower_bound * log2(e), rounded to float, exactly as the kernel
 * receives it [LB "Conversion to the Gate Scale Factor"]. Host only. */
KDA_API float kda_gate_scale(float lower_bound);

/*
 * kda_plan -- the launch plan kda_fwd would use (host only, no GPU needed):
 * for `units` independent (sequence, head) pairs on a device with `num_sms`
 * multiprocessors, writes the number of CTAs each state's V rows are split
 * across (1, 2, 4 or 8) and the grid size. Returns KDA_ERR_NULL for NULL
 * outputs and KDA_ERR_SHAPE for units < 0 or num_sms < 1.
 */
KDA_API kda_status kda_plan(int64_t units, int num_sms, int *v_split, int64_t *grid);

/* Text of the last error raised on the calling thread ("" if none). */
KDA_API const char *kda_last_error(void);

/*
 * kda_check_device_status -- reads and clears the library's device error
 * word of the current device (bad cu_seqlens entries, a pipeline wait that
 * hit its iteration limit, or -- in the bounds-checked build, see
 * kda_debug_build -- an access outside its buffer that was caught and
 * skipped) and synchronises `stream`. The word is shared by
 * every call of this library on the device: it is exchanged with 0 by one
 * atomic operation on `stream`, so a flag set by any earlier call is reported
 * once, by the first check that runs after it, and a flag raised meanwhile by
 * a kernel on another stream is kept for the next check. Returns KDA_OK,
 * KDA_ERR_DEVICE (details in kda_last_error()) or KDA_ERR_LAUNCH.
 */
KDA_API kda_status kda_check_device_status(void *stream);

/* Library version, major * 10000 + minor * 100 + patch. */
KDA_API int kda_version(void);

#ifdef __cplusplus
}
#endif

#endif /* KDA_H */
