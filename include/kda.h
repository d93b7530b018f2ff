/*
 * kda.h -- C ABI of the GB300 (sm_103a) Kimi Delta Attention (KDA) hot path.
 *
 * KDA is a gated delta rule whose forget gate decays each KEY CHANNEL separately
 * (the "per-K-channel exp2(gk)" decay of vllm.cpp PR #110 "chunk_kda prefill AOT
 * port", commit description; vllm.cpp PR #122 "fold Kimi-Linear onto the shared
 * paged runner", block B2, contrasts it with GDN's per-head decay).  For one head
 * with state S (K x V, row = key channel) and token t:
 *
 *     S_t = (I - beta_t k_t k_t^T) Diag(exp(g_t)) S_{t-1} + beta_t k_t v_t^T
 *     o_t = scale * S_t^T q_t
 *
 * The library has the two halves of the prefill=chunk / decode=recurrent split
 * (PR #110 commit description; PR #113 "paged-incremental decode", commit body):
 *
 *   kda_chunk_prefill     -- the whole prompt of each packed sequence, chunk by
 *                            chunk (64 tokens), from an optional initial state;
 *                            returns the outputs and the final state per sequence
 *                            (the state carried into decode, PR #113).
 *   kda_chunk_prefill_ws  -- the same prefill with a caller-owned workspace instead of
 *                            the library's own scratch (any number of calls in flight).
 *   kda_chunk_prefill_paged -- the same prefill with the initial and final states in
 *                            paged pool slots selected per sequence (in place).
 *   kda_recurrent_decode  -- one token per sequence against the state held in a
 *                            paged pool slot, updated in place (state slots keyed
 *                            by per-sequence indices, PR #122 block B2); its
 *                            _bf16_state form keeps the pool in bf16.
 *   kda_chunk_prefill_host -- the prefill of a prompt held in HOST memory, outputs
 *                            returned to host memory, the copies overlapped with it.
 *   kda_causal_conv1d_fwd / _update -- the short causal convolution in front of the
 *                            op over the packed [q|k|v] channels, its taps carried per
 *                            slot (PR #122 block B2; PR #113 commit body).
 *
 * Conventions for every call
 * --------------------------
 *  * Pointers are DEVICE pointers (cudaMalloc / torch CUDA memory) unless stated;
 *    each must be 16-byte aligned.  All tensors are dense and row-major with the
 *    last dimension contiguous:
 *        q, k, g : [tokens, H, K]     v, out : [tokens, H, V]     beta : [tokens, H]
 *        states  : [.., H, K, V]      (V fastest; a state row is one key channel)
 *  * dtype (KDA_DTYPE_*) is the element type of q, k and v; out_dtype that of out
 *    (either may be fp32 or bf16; an fp32 out suits an fp32 residual stream, and a
 *    bf16 out holds exactly the fp32 result rounded to nearest).  g, beta and all
 *    states are fp32, except the bf16 pool of kda_recurrent_decode_bf16_state.  g is the NATURAL-log gate (g <= 0 for a decay); the kernels
 *    work in exp2 space internally.  Accumulation is fp32.
 *  * The caller owns every buffer.  The library allocates no device or host memory
 *    and synchronises nothing (except kda_chunk_prefill_status, which says so): all
 *    work is enqueued on `stream` (a cudaStream_t; NULL = the legacy default stream).
 *    (kda_chunk_prefill_host also uses two copy streams and a few events of its own,
 *    created on its first call per device and kept until exit.)
 *    Errors from the kernels themselves surface at the caller's next synchronisation.
 *  * Prefill scratch.  The tensor-core prefill (bf16 q/k/v, K = V = 128) runs one
 *    4-CTA thread-block cluster per (sequence, head); each CTA builds every fourth
 *    chunk's operands (gate cumsum, decayed factors, A_kk, A_qk, the triangular inverse)
 *    and all four read them back through a ring of records in device memory.  The _ws
 *    entry points take that ring from the caller; the others use one device array inside
 *    the library (25.7 MB per device, present from load), so on one device only ONE
 *    prefill without a workspace may be in flight at a time: calls on one stream are
 *    ordered and safe, calls whose executions overlap (several streams or host threads)
 *    race and give wrong results.  Every call runs on one GPU, and a ring must be device
 *    memory of the GPU that runs the call.
 *  * Bounded waits.  The CTAs of a cluster wait on one another and on their tensor-core
 *    work; every such wait is bounded in time (2 s by default, kda_set_prefill_wait_limit).
 *    A wait that runs out ends that cluster's work early and leaves a status word in the
 *    ring's header that kda_chunk_prefill_status reports as KDA_ERR_TIMEOUT; the outputs
 *    and final states of that launch are then incomplete.
 *  * Range.  The tensor-core prefill rounds its operands to fp16: v, the states scaled by
 *    2^m (m <= 0 for decays) and the per-chunk corrected values (about v minus the
 *    state's prediction) must stay below 65,504 in magnitude, and q and k are expected at
 *    unit scale (L2-normalised keys, as KDA uses them).  Gates of any strength are
 *    covered (a chunk whose gate spans more than 2^16 takes an exact-exponential path).
 *  * Return value: KDA_OK (0) or a negative kda_status; on error nothing has been
 *    enqueued.  kda_status_string() names a status.
 *  * Aliasing: no output may overlap an input byte range, except that the prefill's
 *    final_state may be EXACTLY init_state (in-place carry).  Violations give
 *    KDA_ERR_ALIAS (the byte-range guard idea of flare PR #23, "Kimi K3: fused
 *    decode pack and retained-buffer compaction", design notes).
 *  * Supported shapes: K, V in {64, 128}; H >= 1.
 */
#ifndef KDA_H_
#define KDA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define KDA_ABI_VERSION 5

#if defined(__GNUC__)
#define KDA_API __attribute__((visibility("default")))
#else
#define KDA_API
#endif

/* Element type of q, k, v (dtype) and of out (out_dtype). */
enum kda_dtype {
    KDA_DTYPE_F32 = 0,
    KDA_DTYPE_BF16 = 1
};

/*
 * Option bits of the `flags` argument of the prefill and decode calls.
 *
 * KDA_FLAG_QK_L2NORM: normalise every query and key row over the key dimension inside
 *   the kernel, q <- q / sqrt(sum_c q_c^2 + 1e-6) and likewise k, before it is used --
 *   the in-kernel half of the fused prologue of the prompt path (vllm.cpp PR #110,
 *   commit description: chunk_kda_with_fused_gate), which reads unit-scale keys.  The
 *   rows are normalised where the kernels load them, so the option reads no extra
 *   bytes.  Without it q and k are used as given (callers normalise them).
 */
#define KDA_FLAG_QK_L2NORM 1

enum kda_status {
    KDA_OK = 0,
    KDA_ERR_INVALID_ARG = -1,   /* null required pointer, negative size, misaligned pointer,
                                   non-finite scale */
    KDA_ERR_UNSUPPORTED = -2,   /* K or V outside {64, 128}, unknown dtype or out_dtype */
    KDA_ERR_ALIAS = -3,         /* an output overlaps an input */
    KDA_ERR_CUDA = -4,          /* a CUDA runtime call or launch failed (see kda_last_cuda_error) */
    KDA_ERR_TIMEOUT = -5        /* a bounded wait inside the prefill kernel ran out (reported by
                                   kda_chunk_prefill_status) */
};

/* KDA_ABI_VERSION of the loaded library. */
KDA_API int kda_abi_version(void);

/* Static, NUL-terminated name of a status code. */
KDA_API const char *kda_status_string(int status);

/* cudaError_t of the last failing CUDA call in this thread (0 if none). */
KDA_API int kda_last_cuda_error(void);

/*
 * Chunked prefill over packed variable-length sequences.
 *
 * Defined by the chunked prompt path of vllm.cpp PR #110 (commit description: the
 * in-chunk gate cumsum in exp2 space, the decayed intra-chunk k.k^T, the unit
 * lower-triangular solve, the w/u recompute, the inter-chunk state propagation and
 * the output), with the state carry of PR #113 (commit body: the final recurrent
 * state of the prompt is the state the decode continues from).
 *
 *   q, k         [total_tokens, H, K]  dtype     queries / keys (callers normally
 *                                                 L2-normalise them; not done here)
 *   v            [total_tokens, H, V]  dtype     values
 *   g            [total_tokens, H, K]  fp32      natural-log gate per key channel
 *   beta         [total_tokens, H]     fp32      delta-rule write strength
 *   scale                               fp32     output scale (e.g. 1/sqrt(K))
 *   init_state   [num_seqs, H, K, V]   fp32      initial state per sequence, or NULL
 *                                                 for zeros
 *   cu_seqlens   [num_seqs + 1]        int32     sequence n is tokens
 *                                                 [cu_seqlens[n], cu_seqlens[n+1]);
 *                                                 read on the device.  Bounds are
 *                                                 clamped to [0, total_tokens] and a
 *                                                 decreasing pair is an empty sequence,
 *                                                 so no access leaves the buffers.
 *   out          [total_tokens, H, V]  out_dtype written for every token of every
 *                                                 sequence; rows outside all sequences
 *                                                 are not written
 *   final_state  [num_seqs, H, K, V]   fp32      state after the last token of each
 *                                                 sequence (init_state, or zeros, for an
 *                                                 empty one), or NULL to skip.  May be
 *                                                 exactly init_state.
 *   total_tokens, num_seqs >= 0; H >= 1; K, V in {64, 128}; dtype, out_dtype kda_dtypes.
 *   flags        KDA_FLAG_* bits (KDA_FLAG_QK_L2NORM); any other bit: KDA_ERR_INVALID_ARG.
 *
 * bf16 q/k/v with K = V = 128 run on the tensor-core cluster kernel with the library's
 * scratch (one such call in flight per device, see "Prefill scratch"; any batch size: the
 * clusters are persistent and walk the (sequence, head) work items); other shapes and
 * fp32 inputs on an exact CUDA-core kernel that needs no scratch.
 */
KDA_API int kda_chunk_prefill(const void *q, const void *k, const void *v,
                              const float *g, const float *beta, float scale,
                              const float *init_state, const int32_t *cu_seqlens,
                              void *out, float *final_state,
                              int64_t total_tokens, int32_t num_seqs, int32_t num_heads,
                              int32_t head_dim_k, int32_t head_dim_v, int32_t dtype,
                              int32_t out_dtype, int32_t flags, void *stream);

/*
 * Bytes of workspace kda_chunk_prefill_ws needs for these sizes on the CURRENT device:
 * a 256-byte header (the device status word) and a ring of 8 records of 66,816 bytes for
 * each of min(num_seqs * H, clusters the device keeps resident) clusters (~20 MB on a
 * 152-SM GPU whatever num_seqs is).  0 when the call needs none: num_seqs == 0, or
 * shapes that do not run on the tensor-core kernel (dtype fp32, or K or V != 128).
 */
KDA_API size_t kda_chunk_prefill_workspace_bytes(int32_t num_seqs, int32_t num_heads,
                                                 int32_t head_dim_k, int32_t head_dim_v,
                                                 int32_t dtype);

/*
 * kda_chunk_prefill with a caller-owned device workspace.
 *
 * Same operation, arguments, conventions and results as kda_chunk_prefill (vllm.cpp PR
 * #110, commit description; PR #113, commit body), on the same kernel; only the ring
 * through which the four CTAs of a cluster share each chunk's operands is the caller's.
 *
 *   workspace        device memory of the CURRENT device, 16-byte aligned, at least
 *                    kda_chunk_prefill_workspace_bytes(num_seqs, num_heads, head_dim_k,
 *                    head_dim_v, dtype) bytes; may be NULL when that is 0.  It must be
 *                    ZERO-FILLED before its first use (cudaMemset): its header holds the
 *                    device status word, which the kernel only sets and
 *                    kda_chunk_prefill_status reads and clears; the rest needs no
 *                    initialisation.  It must not overlap any other argument
 *                    (KDA_ERR_ALIAS), and two calls in flight at once need two
 *                    workspaces.  Host or another device's memory: KDA_ERR_INVALID_ARG.
 *   workspace_bytes  its size; smaller than required -> KDA_ERR_INVALID_ARG.
 * Every other argument as for kda_chunk_prefill.
 */
KDA_API int kda_chunk_prefill_ws(const void *q, const void *k, const void *v,
                                 const float *g, const float *beta, float scale,
                                 const float *init_state, const int32_t *cu_seqlens,
                                 void *out, float *final_state,
                                 int64_t total_tokens, int32_t num_seqs, int32_t num_heads,
                                 int32_t head_dim_k, int32_t head_dim_v, int32_t dtype,
                                 int32_t out_dtype, void *workspace, size_t workspace_bytes,
                                 int32_t flags, void *stream);

/*
 * kda_chunk_prefill for callers that cannot allocate device memory.  The pages have no
 * counterpart of this entry point: it serves hosts whose allocator is not reachable
 * through the C ABI (a runtime that owns the device heap, a plug-in loaded into another
 * program), which can pass inputs and outputs but no workspace.  The scratch is the
 * library's own file-scope device array (25.7 MB per device: the status header and a ring
 * for 48 clusters; zero at load, present from load until exit); the address is looked up
 * on each call with cudaGetSymbolAddress, and no call allocates or frees anything.
 *
 * Arguments, results and errors as for kda_chunk_prefill (which uses the same array),
 * without the flags argument: q and k are used as given.
 * Every call on a device uses the SAME array, which keeps the last call's contents:
 * two calls whose executions overlap (on different streams, or from different host
 * threads without ordering) race on it and give wrong results; calls enqueued on one
 * stream are ordered and safe.
 */
KDA_API int kda_chunk_prefill_noalloc(const void *q, const void *k, const void *v,
                                      const float *g, const float *beta, float scale,
                                      const float *init_state, const int32_t *cu_seqlens,
                                      void *out, float *final_state,
                                      int64_t total_tokens, int32_t num_seqs, int32_t num_heads,
                                      int32_t head_dim_k, int32_t head_dim_v, int32_t dtype,
                                      int32_t out_dtype, void *stream);

/*
 * Device status of the last tensor-core prefill that used `workspace` (NULL: the
 * library's scratch on the current device), after `stream` has finished.
 *
 * SYNCHRONISES `stream`, reads the status word the kernel leaves in the scratch and
 * clears it.  KDA_OK: no wait ran out; KDA_ERR_TIMEOUT: a bounded wait inside the kernel
 * ran out (the clusters concerned abandoned their work, drained their own copies and
 * MMAs and exited; outputs and final states of that launch are incomplete); KDA_ERR_CUDA:
 * the stream reported an error or the read failed.  This is the failure report of the
 * bounded waits that the prefill's CTAs use to hand chunks to one another; there is no
 * counterpart on the pages.
 */
KDA_API int kda_chunk_prefill_status(const void *workspace, void *stream);

/*
 * Limit, in nanoseconds, of every wait inside the tensor-core prefill kernels launched
 * after this call (process-wide; 0 restores the default of 2 s).  A limit far below a
 * chunk's build time makes the waits run out on purpose, which is how the timeout path
 * is tested; no launch then hangs or faults.
 */
KDA_API void kda_set_prefill_wait_limit(uint64_t nanoseconds);

/*
 * Chunked prefill whose per-sequence states live in paged pool slots.
 *
 * The prompt path over the paged state group (vllm.cpp PR #122 "fold Kimi-Linear
 * onto the shared paged runner", block B2: the chunked prefill for fresh prompts
 * and the state gather / scatter over the group's slots keyed by per-sequence state
 * indices).  Same computation as kda_chunk_prefill, except that sequence n starts
 * from the state held in slot state_idx[n] of state_pool and its final state is
 * written back to that slot, in place.  A fresh prompt starts from a zeroed slot.
 *
 *   q, k, v, g, beta, scale, cu_seqlens, out   as for kda_chunk_prefill
 *   state_pool   [num_slots, H, K, V]  fp32   read and updated IN PLACE at the selected
 *                                              slots; every other slot is left bit-identical
 *   state_idx    [num_seqs]            int32  slot of each sequence, read on the device.
 *                                              Slots must be distinct (duplicates race).
 *                                              An index outside [0, num_slots) reads and
 *                                              writes no slot: that sequence runs from a
 *                                              zero state and its final state is dropped.
 * Runs on the library's scratch like kda_chunk_prefill (one such call in flight per
 * device).
 */
KDA_API int kda_chunk_prefill_paged(const void *q, const void *k, const void *v,
                                    const float *g, const float *beta, float scale,
                                    float *state_pool, const int32_t *state_idx,
                                    const int32_t *cu_seqlens, void *out,
                                    int64_t total_tokens, int32_t num_seqs, int32_t num_slots,
                                    int32_t num_heads, int32_t head_dim_k, int32_t head_dim_v,
                                    int32_t dtype, int32_t out_dtype, int32_t flags, void *stream);

/*
 * kda_chunk_prefill_paged with a caller workspace: the same operation with the
 * workspace rules and size of kda_chunk_prefill_ws (kda_chunk_prefill_workspace_bytes(
 * num_seqs, ...)).  The workspace must not overlap any other argument, the pool
 * included (KDA_ERR_ALIAS).
 */
KDA_API int kda_chunk_prefill_paged_ws(const void *q, const void *k, const void *v,
                                       const float *g, const float *beta, float scale,
                                       float *state_pool, const int32_t *state_idx,
                                       const int32_t *cu_seqlens, void *out,
                                       int64_t total_tokens, int32_t num_seqs, int32_t num_slots,
                                       int32_t num_heads, int32_t head_dim_k, int32_t head_dim_v,
                                       int32_t dtype, int32_t out_dtype, void *workspace,
                                       size_t workspace_bytes, int32_t flags, void *stream);

/*
 * One recurrent decode step for num_seqs sequences with paged states.
 *
 * Defined by the decode side of the split: one token per sequence advanced from
 * the carried state (vllm.cpp PR #113, commit body), over the paged state group
 * whose slots are selected per sequence (vllm.cpp PR #122, block B2: state
 * gather / scatter keyed by the per-sequence state indices).  Gather, update and
 * scatter are one pass: each selected state is read once and written once.
 *
 *   q, k         [num_seqs, H, K]  dtype
 *   v            [num_seqs, H, V]  dtype
 *   g            [num_seqs, H, K]  fp32   natural-log gate
 *   beta         [num_seqs, H]     fp32
 *   state_pool   [num_slots, H, K, V] fp32  updated IN PLACE at the selected slots;
 *                                           every other slot is left bit-identical
 *   state_idx    [num_seqs]        int32  slot of each sequence, read on the device.
 *                                           Slots must be distinct (duplicates race).
 *                                           An index outside [0, num_slots) touches
 *                                           no slot and gives zero outputs.
 *   out          [num_seqs, H, V]  out_dtype
 *   flags        KDA_FLAG_* bits as for kda_chunk_prefill (KDA_FLAG_QK_L2NORM normalises
 *                the token's q and k rows before the step)
 */
KDA_API int kda_recurrent_decode(const void *q, const void *k, const void *v,
                                 const float *g, const float *beta, float scale,
                                 float *state_pool, const int32_t *state_idx, void *out,
                                 int32_t num_seqs, int32_t num_slots, int32_t num_heads,
                                 int32_t head_dim_k, int32_t head_dim_v, int32_t dtype,
                                 int32_t out_dtype, int32_t flags, void *stream);

/*
 * kda_recurrent_decode over a pool stored in bf16: the same step, the same
 * arguments, with state_pool [num_slots, H, K, V] of bf16 elements.
 *
 * The state's element type is a configuration of the model runner (vllm.cpp PR #122,
 * block B3: the conv cache dtype mirrors kda_state_dtype); the pages give no rule for
 * how a narrower state is used, and the one taken here is storage only: the selected
 * state is read into fp32, the step runs in fp32 exactly as with an fp32 pool, the
 * output is read from the fp32 updated state, and only the stored state is rounded
 * (to nearest, ties to even).  Each step thus reads and writes half the bytes and
 * rounds the carried state once (relative error <= 2^-9 per element and step; the
 * same pages warn that bf16 rounding inside the recurrence can destabilise it, so
 * this form is opt-in).  Slots outside state_idx are left bit-identical; the errors,
 * alignment and aliasing rules are those of kda_recurrent_decode (the pool's byte
 * range is num_slots * H * K * V * 2).
 */
KDA_API int kda_recurrent_decode_bf16_state(const void *q, const void *k, const void *v,
                                            const float *g, const float *beta, float scale,
                                            void *state_pool, const int32_t *state_idx, void *out,
                                            int32_t num_seqs, int32_t num_slots, int32_t num_heads,
                                            int32_t head_dim_k, int32_t head_dim_v, int32_t dtype,
                                            int32_t out_dtype, int32_t flags, void *stream);

/*
 * kda_chunk_prefill_host -- kda_chunk_prefill of a prompt whose inputs are in HOST memory,
 * with the outputs and the final states returned to host memory.  The prompt path of
 * vllm.cpp PR #113 ("paged-incremental decode", commit body): the prompt is prefilled once
 * with the chunked kernel and its state carried into decode.
 *
 * The packed token range is cut into `pieces` (1..KDA_HOST_MAX_PIECES) pieces on 64-token
 * boundaries.  Piece s is copied host-to-device on a copy stream, prefilled on `stream`
 * (every sequence clipped to the piece, its state carried in place from the previous
 * piece), and its output rows are copied device-to-host on a second copy stream, so the
 * copies of neighbouring pieces overlap the prefill.  A prefill split at any token and
 * continued from the carried state is the unsplit prefill (up to rounding).
 *
 *   q, k, v, g, beta, cu_seqlens, init_state (or NULL: zeros)   HOST inputs, the layouts
 *                    of kda_chunk_prefill; page-locked memory lets the copies run
 *                    asynchronously (pageable memory works, with staged copies).
 *   out, final_state (or NULL: not returned)   HOST outputs, valid once `stream` has been
 *                    synchronised; final_state == init_state carries the state in place.
 *   device_buffer    device memory of the current GPU, 256-byte aligned, at least
 *                    kda_chunk_prefill_host_device_bytes(...) bytes, zero-filled before
 *                    its first use.  It starts with the prefill workspace, so
 *                    kda_chunk_prefill_status(device_buffer, stream) reports this call's
 *                    status.  One call at a time per buffer.
 *   flags            as for kda_chunk_prefill.
 * Errors: KDA_ERR_INVALID_ARG (sizes, pieces, a NULL input, the buffer), KDA_ERR_ALIAS (a
 * host output overlapping a host input or the other output, other than the in-place state
 * carry), KDA_ERR_UNSUPPORTED (dtypes,
 * head sizes); on those nothing is enqueued.  KDA_ERR_CUDA from the runtime (work already
 * enqueued by this call then stays enqueued).
 * The function only enqueues work; calls from several host threads are serialised while
 * they enqueue.
 */
#define KDA_HOST_MAX_PIECES 16
KDA_API size_t kda_chunk_prefill_host_device_bytes(int64_t total_tokens, int32_t num_seqs,
                                                   int32_t num_heads, int32_t head_dim_k,
                                                   int32_t head_dim_v, int32_t dtype,
                                                   int32_t out_dtype, int32_t pieces);
KDA_API int kda_chunk_prefill_host(const void *q, const void *k, const void *v, const float *g,
                                   const float *beta, float scale, const float *init_state,
                                   const int32_t *cu_seqlens, void *out, float *final_state,
                                   int64_t total_tokens, int32_t num_seqs, int32_t num_heads,
                                   int32_t head_dim_k, int32_t head_dim_v, int32_t dtype,
                                   int32_t out_dtype, int32_t pieces, void *device_buffer,
                                   size_t device_buffer_bytes, int32_t flags, void *stream);

/* Activation of the causal convolution. */
enum kda_conv_activation {
    KDA_CONV_ACT_NONE = 0,
    KDA_CONV_ACT_SILU = 1      /* z / (1 + exp(-z)) */
};

/*
 * The short causal convolution in front of the KDA op, over a packed prompt.
 *
 * Defined by the conv taps of the KDA block (vllm.cpp PR #122 "fold Kimi-Linear onto the
 * shared paged runner", block B2: CausalConv1dFwd over the varlen prompt, the carried
 * conv_state split as chunk(3) into [q|k|v]; vllm.cpp PR #113, commit body: the conv-tap
 * carry of the decode regime).  A depthwise convolution of width W over D channels (the
 * packed [q|k|v] projections): per sequence n and channel c, with the W - 1 taps carried
 * in slot state_idx[n] prepended to the sequence's inputs (oldest first),
 *     out_t = act(bias_c + sum_{j < W} weight[c][j] xe_{t+j})
 * so out_t sees x_t and the W - 1 inputs before it; afterwards the slot holds the last
 * W - 1 entries of [taps | inputs] (exact copies of inputs: a prompt split anywhere and
 * continued from its taps gives the unsplit result bit for bit).
 *
 *   x           [total_tokens, D]   dtype       inputs, packed by cu_seqlens
 *   weight      [D, W]              fp32        per-channel taps, weight[c][W-1] on x_t
 *   bias        [D]                 fp32        or NULL
 *   conv_state  [num_slots, W-1, D] dtype       carried taps, read and updated IN PLACE at
 *                                               the selected slots (every other slot is
 *                                               left bit-identical); NULL: zero taps,
 *                                               nothing kept.  A fresh prompt starts from
 *                                               a zeroed slot.
 *   state_idx   [num_seqs]          int32       slot of each sequence (with conv_state);
 *                                               read on the device; distinct (duplicates
 *                                               race); an index outside [0, num_slots)
 *                                               gives zero taps and keeps nothing
 *   cu_seqlens  [num_seqs + 1]      int32       non-decreasing sequence bounds (read on
 *                                               the device and clamped to [0, total_tokens])
 *   out         [total_tokens, D]   out_dtype   rows outside every sequence are not written
 *   D >= 4 and a multiple of 4; W in 1..4; activation a kda_conv_activation.
 * Pointers 16-byte aligned; out must not overlap any input, conv_state no input or out
 * (KDA_ERR_ALIAS).  Two kernels on `stream`: the outputs (reading the old taps), then the
 * new taps.
 */
KDA_API int kda_causal_conv1d_fwd(const void *x, const float *weight, const float *bias,
                                  void *conv_state, const int32_t *state_idx,
                                  const int32_t *cu_seqlens, void *out, int64_t total_tokens,
                                  int32_t num_seqs, int32_t num_slots, int32_t dim,
                                  int32_t width, int32_t dtype, int32_t out_dtype,
                                  int32_t activation, void *stream);

/*
 * One token per sequence through the same convolution, the taps of slot state_idx[n]
 * shifted by one in place (vllm.cpp PR #122, block B2: CausalConv1dUpdate for decode).
 *
 *   x    [num_seqs, D] dtype;   out [num_seqs, D] out_dtype;   every other argument as for
 *   kda_causal_conv1d_fwd.  One kernel on `stream`; a decode step after
 *   kda_causal_conv1d_fwd on the same slot continues the prompt exactly.
 */
KDA_API int kda_causal_conv1d_update(const void *x, const float *weight, const float *bias,
                                     void *conv_state, const int32_t *state_idx, void *out,
                                     int32_t num_seqs, int32_t num_slots, int32_t dim,
                                     int32_t width, int32_t dtype, int32_t out_dtype,
                                     int32_t activation, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* KDA_H_ */
