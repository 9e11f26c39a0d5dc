/*
 * gdr.h -- C ABI of the GB300 (sm_103a) gated delta rule forward library
 * (libgdr.so).
 *
 * The operation (Gated DeltaNet forward, one value-head h, state S in
 * R^{V x K} held V-major as S[v][k] in fp32):
 *
 *   S~  = exp(g_t) S_{t-1}        (per-key-channel gate: S_{t-1} diag(exp(gk_t)))
 *   n_t = beta_t (v_t - S~ k_t)
 *   S_t = S~ + n_t k_t^T
 *   o_t = scale * S_t q_t         (read after the update)
 *
 * The step order, the raw (not cumulative) gate and the post-update read are
 * those of FlashQLA PR #1 ("Fused recurrent GDN decode + SGLang DFlash verify
 * kernel"), core decode-kernel commit.  Value-head h reads key/query head
 * h / (Hv / Hk) (same page, review commit: grouped-value attention mapping).
 *
 * Conventions for every entry point
 *   - All tensor pointers are DEVICE pointers unless stated otherwise, dense,
 *     row-major, in the layouts given, 16-byte aligned.
 *   - Token-major packed layout: the batch is folded into the token axis and
 *     sequence b owns tokens [cu_seqlens[b], cu_seqlens[b+1]).
 *   - dtype GDR_BF16 or GDR_F32 applies to q, k, v, beta and o.  Gates (g, gk)
 *     are always fp32; prefill states are always fp32.
 *   - The caller owns every buffer, including the workspace.  No entry point
 *     allocates, frees or synchronises the device (except
 *     gdr_get_device_status and GDR_VALIDATE, which say so), so calls can be
 *     captured in a CUDA graph.  Work is enqueued on `stream` (NULL = legacy
 *     default stream).
 *   - Inputs are never written.  Outputs must not alias inputs.
 *   - Return value: GDR_OK or a gdr_status error code; on error nothing was
 *     launched and gdr_last_error() describes the problem (thread-local).
 *     Argument and shape checks happen on the host before any launch.
 *   - Empty work (T_total == 0 or N == 0) returns GDR_OK without a launch.
 */
#ifndef GDR_H_
#define GDR_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define GDR_API __attribute__((visibility("default")))
#else
#define GDR_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t. */
typedef struct CUstream_st* gdr_stream_t;

typedef enum gdr_status {
    GDR_OK = 0,
    GDR_ERR_INVALID_ARG = 1,    /* null pointer, bad size, misaligned pointer  */
    GDR_ERR_UNSUPPORTED = 2,    /* shape / dtype / device not supported        */
    GDR_ERR_WORKSPACE = 3,      /* workspace missing or too small              */
    GDR_ERR_LAUNCH = 4,         /* a CUDA launch or runtime call failed        */
    GDR_ERR_DEVICE_TIMEOUT = 5, /* a bounded device-side wait gave up          */
    GDR_ERR_VALIDATION = 6      /* GDR_VALIDATE found bad input content        */
} gdr_status;

typedef enum gdr_dtype { GDR_BF16 = 0, GDR_F32 = 1 } gdr_dtype;

typedef enum gdr_gate_kind {
    GDR_GATE_SCALAR = 0,  /* g  [T, Hv]     one log-decay per token and value-head */
    GDR_GATE_CHANNEL = 1  /* gk [T, Hv, K]  one log-decay per key channel (KDA)    */
} gdr_gate_kind;

/* flags (bitwise or) */
#define GDR_QK_L2NORM  0x1 /* normalise q and k rows in-library: x * rsqrt(sum x^2 + 1e-6) */
#define GDR_NEG_EIGVAL 0x2 /* gdr_gating_fwd: beta = 2 * sigmoid(b)                         */
#define GDR_COMMIT     0x4 /* gdr_recurrent_fwd: write the final state back to the pool     */
#define GDR_VALIDATE   0x8 /* check input contents on the device first (synchronises).
                              * The findings land in one library-wide device word:
                              * validated calls from different host threads must be
                              * serialised by the caller, or one call's reset of the
                              * word can hide the other's findings.                  */
#define GDR_CHANNEL_GATE 0x10 /* gdr_recurrent_fwd: g is per key channel, [T_total, Hv, K]  */
#define GDR_CHUNK_SCAN 0x20   /* gdr_chunk_fwd: chunk-parallel state scan (long sequences)     */

/* Chunk length of the chunked prefill (tokens).  The pages' kernels use 64. */
#define GDR_CHUNK 64

/*
 * gdr_chunk_workspace_size -- bytes of device workspace gdr_chunk_fwd needs.
 * Host only; depends on sizes, never on cu_seqlens contents (the chunk count
 * is bounded by ceil(T_total / 64) + N, the "capacity" of attention-gym
 * PR #344's inter-chunk state kernel).  Returns GDR_OK and sets *bytes.
 */
GDR_API int gdr_chunk_workspace_size(int N, int64_t T_total, int Hk, int Hv, int K, int V,
                             int gate_kind, int dtype, int flags, size_t* bytes);

/*
 * gdr_chunk_fwd -- chunked (WY, 64-token chunks) prefill over packed
 * variable-length sequences.  Computes exactly the recurrence above; the
 * chunked form is an implementation choice (FlashQLA PR #1 names the
 * chunked-prefill pieces cumsum / A / kkt-solve; attention-gym PR #344 gives
 * the inter-chunk state kernel with its per-chunk state h and v_new).
 *
 *   q, k           [T_total, Hk, K]   dtype
 *   v              [T_total, Hv, V]   dtype
 *   g              [T_total, Hv] fp32 log-decay (<= 0), or NULL
 *   gk             [T_total, Hv, K] fp32 per-key-channel log-decay, or NULL;
 *                  exactly one of g / gk is non-NULL
 *   beta           [T_total, Hv]      dtype, in [0, 1] (or [0, 2])
 *   initial_state  [N, Hv, V, K] fp32, or NULL for zeros
 *   cu_seqlens     [N+1] int32 device, cu[0] = 0, non-decreasing,
 *                  cu[N] = T_total; every sequence non-empty.  A cu_seqlens
 *                  that breaks the first three rules is found on the device
 *                  and nothing is written (the call still returns GDR_OK;
 *                  GDR_VALIDATE turns it into GDR_ERR_VALIDATION)
 *   scale          read scale (usually 1/sqrt(K))
 *   o              [T_total, Hv, V]   dtype (written)
 *   final_state    [N, Hv, V, K] fp32 (written), or NULL
 *   workspace      device scratch of at least gdr_chunk_workspace_size bytes,
 *                  256-byte aligned; contents need no initialisation
 * Supported: Hv % Hk == 0, K == V, K in {64, 128}.  bf16 inputs run on the
 * tensor cores at both sizes (a 64-channel head as a 128-channel tile whose
 * upper channels are zero), fp32 inputs on the CUDA cores.  Any finite g <= 0 is
 * accepted: every exponential formed is of an in-chunk difference
 * exp(gam_i - gam_j), i >= j (cuLA PR #113 review on exp(-prefix) overflow).
 *
 * GDR_CHUNK_SCAN (bf16, K = V = 128; ignored otherwise, with the same
 * results): the serial chain over a sequence's chunks is cut into segments.
 * The state map of a segment is affine in its start state,
 * S_end = S_start P + B, with P [K, K] and B [V, K]; in one parallel pass
 * the first segment of each sequence runs from the initial state (writing
 * its part of o) while the others form their B (and P, but for the last),
 * a scan composes them into every segment's start state, and the later
 * segments then run in parallel again to write o.  It pays for long
 * sequences with few value heads: the plain chain runs Hv * K / 32 CTAs per
 * sequence, 64 tokens per step, and the scan costs about three chain passes
 * of work instead of one, so it wins while 12 * Hv * N is well under the
 * GPU's SM count (measured on GB300 with one 32768-token sequence: 5x at
 * Hv = 1, 2.5x at Hv = 4, 1.5x at Hv = 8, a loss at Hv = 16).  The caller
 * decides; the flag always takes the scan where it applies.  The workspace
 * grows by about
 * 2 * (ceil(T_total / 64 / G) + N + 1) * Hv * K * K * 4 bytes, G the segment
 * length in chunks (at least 4 where sequences allow) that the library derives
 * from N, T_total and Hv.
 */
GDR_API int gdr_chunk_fwd(const void* q, const void* k, const void* v, const float* g,
                  const float* gk, const void* beta, const float* initial_state,
                  const int32_t* cu_seqlens, int N, int64_t T_total, int Hk, int Hv,
                  int K, int V, float scale, int dtype, int flags, void* o,
                  float* final_state, void* workspace, size_t ws_bytes,
                  gdr_stream_t stream);

/*
 * gdr_chunk_fwd_noalloc -- gdr_chunk_fwd without a caller workspace.  There is
 * no counterpart on the reference pages; it exists for callers that cannot
 * allocate device memory (a serving engine whose arena already owns all device
 * memory, a plugin host that exposes no allocator, a decode loop that cannot
 * afford cudaMalloc's implicit synchronisation).
 *   Same arguments and results as gdr_chunk_fwd, minus workspace / ws_bytes.
 *   Scratch comes from an array of GDR_NOALLOC_WORKSPACE_BYTES compiled into
 *   the library; every GPU that loads the library holds it until exit.  A
 *   problem whose gdr_chunk_workspace_size exceeds it is rejected with
 *   GDR_ERR_WORKSPACE before anything runs.
 *   Every call looks up the array's device address in the context current on
 *   the calling thread (the address belongs to the context, so it stays right
 *   after cudaDeviceReset or with another context current on the device).
 *   The first call in a context may load the library's device code there:
 *   make it before any stream capture.
 *   Nothing is allocated or freed, by the library or any routine it calls.
 *   All calls share the one array and it keeps the previous call's contents
 *   (nothing in it has to start at zero): calls whose work overlaps on the
 *   GPU -- on different streams, or from different host threads -- race on it
 *   and must be serialised by the caller.
 */
#define GDR_NOALLOC_WORKSPACE_BYTES (64ull << 20)
GDR_API int gdr_chunk_fwd_noalloc(const void* q, const void* k, const void* v, const float* g,
                                  const float* gk, const void* beta, const float* initial_state,
                                  const int32_t* cu_seqlens, int N, int64_t T_total, int Hk, int Hv,
                                  int K, int V, float scale, int dtype, int flags, void* o,
                                  float* final_state, gdr_stream_t stream);

/*
 * gdr_recurrent_fwd -- slot-indexed recurrent decode / multi-step verify
 * (FlashQLA PR #1, paged verify commit and deployment-facts commit).
 *
 *   q, k           [T_total, Hk, K] dtype;   v [T_total, Hv, V] dtype
 *   g              [T_total, Hv] fp32 raw log-decay, or with GDR_CHANNEL_GATE
 *                  [T_total, Hv, K] fp32 per-key-channel log-decay (column c
 *                  of the state scaled by e^{g[t,h,c]}: the per-channel decode
 *                  of tokenspeed PR #834);  beta [T_total, Hv] dtype
 *   state_pool     [num_slots, Hv, V, K] (V-major), pool_dtype GDR_F32 or
 *                  GDR_BF16; read, and written in place only with GDR_COMMIT
 *   state_indices  [N] int32 device: pool slot of sequence b; -1 (any value
 *                  < 0) is padding: nothing of sequence b is read or written
 *                  (its o rows, pool slot and ibuf row stay untouched); slot 0
 *                  is a valid slot; valid slots must be unique and < num_slots
 *   cu_seqlens     [N+1] int32 device (decode: 0..N); a sequence may be empty
 *   o              [T_total, Hv, V] dtype (written for non-padding sequences)
 *   intermediate_states  [rows >= N, steps, Hv, V, K] pool dtype, or NULL:
 *                  row b, step t receives the state after token t of
 *                  sequence b (t < L_b), rounded to the pool dtype; rows of
 *                  padding sequences and steps >= L_b are untouched.  Requires
 *                  L_b <= steps (checked under GDR_VALIDATE).
 * The carried state stays fp32 between tokens; only stores round.
 */
GDR_API int gdr_recurrent_fwd(const void* q, const void* k, const void* v, const float* g,
                      const void* beta, void* state_pool, int pool_dtype, int num_slots,
                      const int32_t* state_indices, const int32_t* cu_seqlens, int N,
                      int64_t T_total, int Hk, int Hv, int K, int V, float scale, int dtype,
                      int flags, void* o, void* intermediate_states, int steps,
                      gdr_stream_t stream);

/*
 * gdr_recurrent_fwd_norm -- gdr_recurrent_fwd with the gated RMSNorm output
 * epilogue fused (tokenspeed PR #834, fused gated-norm epilogue commit): every
 * value row x = o[t,h,:] of the recurrence output is written as
 *   x / sqrt(mean_v(x^2) + eps) * norm_weight[v] * sigmoid(norm_gate[t,h,v])
 * norm_weight [V] fp32 device; norm_gate [T_total, Hv, V] dtype device;
 * eps >= 0.  The normalisation uses the fp32 output before any rounding (one
 * bf16 round trip fewer than a separate norm kernel).  Every other argument,
 * flag and guarantee is gdr_recurrent_fwd's.
 */
GDR_API int gdr_recurrent_fwd_norm(const void* q, const void* k, const void* v, const float* g,
                      const void* beta, void* state_pool, int pool_dtype, int num_slots,
                      const int32_t* state_indices, const int32_t* cu_seqlens, int N,
                      int64_t T_total, int Hk, int Hv, int K, int V, float scale, int dtype,
                      int flags, const float* norm_weight, const void* norm_gate, float eps,
                      void* o, void* intermediate_states, int steps, gdr_stream_t stream);

/*
 * gdr_recurrent_fwd_gated -- gdr_recurrent_fwd with the gates formed inside the
 * kernel from the raw projections (FlashQLA PR #1, in-kernel gating commit):
 *   g[t,h]    = -exp(A_log[h]) * softplus(a[t,h] + dt_bias[h])
 *               (softplus beta 1, threshold 20, as gdr_gating_fwd)
 *   beta[t,h] = sigmoid(b[t,h]), times 2 with GDR_NEG_EIGVAL
 *   a, b [T_total, Hv] dtype; A_log, dt_bias [Hv] fp32 device.
 * beta is kept in fp32 (it is not rounded to dtype as gdr_gating_fwd's output
 * is).  Every other argument, flag (GDR_QK_L2NORM, GDR_COMMIT, GDR_VALIDATE)
 * and guarantee is gdr_recurrent_fwd's; GDR_CHANNEL_GATE is not accepted.
 */
GDR_API int gdr_recurrent_fwd_gated(const void* q, const void* k, const void* v, const void* a,
                      const void* b, const float* A_log, const float* dt_bias, void* state_pool,
                      int pool_dtype, int num_slots, const int32_t* state_indices,
                      const int32_t* cu_seqlens, int N, int64_t T_total, int Hk, int Hv, int K,
                      int V, float scale, int dtype, int flags, void* o, void* intermediate_states,
                      int steps, gdr_stream_t stream);

/*
 * gdr_gating_fwd -- gate preparation from raw projections (FlashQLA PR #1,
 * host-gating and in-kernel-gating commits):
 *   g[t,h]    = -exp(A_log[h]) * softplus(a[t,h] + dt_bias[h])
 *               (softplus beta 1, threshold 20)
 *   beta[t,h] = sigmoid(b[t,h]), times 2 with GDR_NEG_EIGVAL
 *   a, b [T, Hv] dtype; dt_bias, A_log [Hv] fp32; g [T, Hv] fp32 (written);
 *   beta [T, Hv] dtype (written).
 */
GDR_API int gdr_gating_fwd(const void* a, const float* dt_bias, const float* A_log, const void* b,
                   int64_t T, int Hv, int dtype, int flags, float* g, void* beta,
                   gdr_stream_t stream);

/* Description of the last error on the calling thread ("" if none). */
GDR_API const char* gdr_last_error(void);

/*
 * gdr_get_device_status -- synchronises `stream`, then reads and clears the
 * library's device error word of the current device (set by a bounded device
 * wait that gave up).  *word receives the raw word (0 = clean).  Returns
 * GDR_OK if the word was 0, GDR_ERR_DEVICE_TIMEOUT otherwise.  Diagnostic only.
 */
GDR_API int gdr_get_device_status(gdr_stream_t stream, int* word);

/*
 * gdr_selftest_bounded_wait -- diagnostic for the failure path (no counterpart
 * on the pages): enqueues on `stream` one small kernel that waits on an
 * mbarrier nothing ever completes, using the same bounded wait as the
 * tensor-core kernels (about one second of %globaltimer); it then sets bit
 * 0x100 of the device error word and returns.  A following
 * gdr_get_device_status reports GDR_ERR_DEVICE_TIMEOUT, and the context stays
 * usable.  Nothing faults, traps or spins without a limit.
 */
GDR_API int gdr_selftest_bounded_wait(gdr_stream_t stream);

/*
 * Kernel timing for diagnostics (no counterpart on the pages; measurement
 * support).  gdr_profile_enable(1): from then on every kernel the library
 * launches is bracketed by two CUDA events on its stream (not capturable:
 * leave it off under stream capture).  gdr_profile_read: waits for the
 * recorded events, then reports per kernel name (sorted) the summed device
 * time in ms and the launch count since the previous read, and clears them.
 *   names      receives "name1,name2,...," (truncated to name_cap bytes)
 *   total_ms, launches  arrays of max_kernels entries
 *   *n_kernels number of entries filled
 */
GDR_API int gdr_profile_enable(int on);
GDR_API int gdr_profile_read(int max_kernels, char* names, size_t name_cap, double* total_ms,
                             int* launches, int* n_kernels);

/* Library version (major * 10000 + minor * 100 + patch). */
GDR_API int gdr_version(void);

#ifdef __cplusplus
}
#endif
#endif /* GDR_H_ */
