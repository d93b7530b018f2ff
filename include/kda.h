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
 *   kda_chunk_prefill_ws  -- the same prefill with a caller workspace, through which
 *                            the four value-tile CTAs of a head share the per-chunk
 *                            operands instead of each building them (faster; same
 *                            result up to fp32 rounding).
 *   kda_chunk_prefill_paged -- the same prefill with the initial and final states in
 *                            paged pool slots selected per sequence (in place); its _ws
 *                            form runs on the shared-operand kernel.
 *   kda_recurrent_decode  -- one token per sequence against the state held in a
 *                            paged pool slot, updated in place (state slots keyed
 *                            by per-sequence indices, PR #122 block B2); its
 *                            _bf16_state form keeps the pool in bf16.
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
 *  * The caller owns every buffer.  The library allocates no device or host memory,
 *    keeps no per-call state, and synchronises nothing: all work is enqueued on
 *    `stream` (a cudaStream_t; NULL = the legacy default stream).  Errors from the
 *    kernels themselves surface at the caller's next synchronisation.
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

#define KDA_ABI_VERSION 3

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

enum kda_status {
    KDA_OK = 0,
    KDA_ERR_INVALID_ARG = -1,   /* null required pointer, negative size, misaligned pointer,
                                   non-finite scale */
    KDA_ERR_UNSUPPORTED = -2,   /* K or V outside {64, 128}, unknown dtype or out_dtype */
    KDA_ERR_ALIAS = -3,         /* an output overlaps an input */
    KDA_ERR_CUDA = -4           /* a CUDA runtime call or launch failed (see kda_last_cuda_error) */
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
 */
KDA_API int kda_chunk_prefill(const void *q, const void *k, const void *v,
                              const float *g, const float *beta, float scale,
                              const float *init_state, const int32_t *cu_seqlens,
                              void *out, float *final_state,
                              int64_t total_tokens, int32_t num_seqs, int32_t num_heads,
                              int32_t head_dim_k, int32_t head_dim_v, int32_t dtype,
                              int32_t out_dtype, void *stream);

/*
 * Bytes of workspace kda_chunk_prefill_ws needs for these sizes on the CURRENT device
 * (the ring of per-chunk operand records of the clusters that can be resident at
 * once: at most (SMs / 4) x 8 x 66,816 bytes, ~20 MB on a 152-SM GPU, whatever
 * num_seqs is).  0 when the call needs none: num_seqs == 0, or shapes that do not run
 * on the shared-operand kernel (dtype fp32, or K or V != 128).
 */
KDA_API size_t kda_chunk_prefill_workspace_bytes(int32_t num_seqs, int32_t num_heads,
                                                 int32_t head_dim_k, int32_t head_dim_v,
                                                 int32_t dtype);

/*
 * kda_chunk_prefill with a caller-owned device workspace.
 *
 * Same operation, arguments, conventions and results as kda_chunk_prefill (vllm.cpp PR
 * #110, commit description; PR #113, commit body); only the schedule differs: the four
 * CTAs that hold the 32-column value tiles of one (sequence, head) form a thread-block
 * cluster, each builds the intra-chunk operands (gate cumsum, decayed factors, A_kk,
 * A_qk and the triangular inverse) of every fourth chunk, and all four read them back
 * through a ring in `workspace`.  Outputs agree with kda_chunk_prefill up to fp32
 * summation order.
 *
 *   workspace        device pointer, 16-byte aligned, at least
 *                    kda_chunk_prefill_workspace_bytes(num_seqs, num_heads, head_dim_k,
 *                    head_dim_v, dtype) bytes (queried on the device that runs the call);
 *                    may be NULL when that is 0.  Contents need no initialisation and
 *                    are garbage afterwards.  It must not overlap any other argument
 *                    (KDA_ERR_ALIAS), and two calls in flight at once need two workspaces.
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
                                 void *stream);

/*
 * kda_chunk_prefill_ws without a caller workspace: the record ring lives in a
 * file-scope device array of the library (48 clusters x 8 x 66,816 bytes = 25.7 MB per
 * device, there from the moment the library is loaded).  The pages have no counterpart
 * of this entry point; it exists for callers that cannot pass a workspace across the
 * C ABI.
 *
 * Arguments, results and errors as for kda_chunk_prefill_ws, plus:
 *   KDA_ERR_UNSUPPORTED  the device can keep more clusters resident than the array has
 *                        room for (more than 48, i.e. more than 192 SMs).
 * Every call on a device uses the SAME array: two calls whose executions overlap (on
 * different streams, or from different host threads without ordering) race on it and
 * give wrong results; calls enqueued on one stream are ordered and safe.  The array
 * needs no initialisation.  The first call on each device looks up the array's
 * address and queries the resident-cluster count, so make it before capturing the
 * stream into a CUDA graph.
 */
KDA_API int kda_chunk_prefill_noalloc(const void *q, const void *k, const void *v,
                                      const float *g, const float *beta, float scale,
                                      const float *init_state, const int32_t *cu_seqlens,
                                      void *out, float *final_state,
                                      int64_t total_tokens, int32_t num_seqs, int32_t num_heads,
                                      int32_t head_dim_k, int32_t head_dim_v, int32_t dtype,
                                      int32_t out_dtype, void *stream);

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
 */
KDA_API int kda_chunk_prefill_paged(const void *q, const void *k, const void *v,
                                    const float *g, const float *beta, float scale,
                                    float *state_pool, const int32_t *state_idx,
                                    const int32_t *cu_seqlens, void *out,
                                    int64_t total_tokens, int32_t num_seqs, int32_t num_slots,
                                    int32_t num_heads, int32_t head_dim_k, int32_t head_dim_v,
                                    int32_t dtype, int32_t out_dtype, void *stream);

/*
 * kda_chunk_prefill_paged with a caller workspace: the same operation on the
 * shared-operand cluster kernel of kda_chunk_prefill_ws (same workspace rules and size,
 * kda_chunk_prefill_workspace_bytes(num_seqs, ...)).  The workspace must not overlap
 * any other argument, the pool included (KDA_ERR_ALIAS).
 */
KDA_API int kda_chunk_prefill_paged_ws(const void *q, const void *k, const void *v,
                                       const float *g, const float *beta, float scale,
                                       float *state_pool, const int32_t *state_idx,
                                       const int32_t *cu_seqlens, void *out,
                                       int64_t total_tokens, int32_t num_seqs, int32_t num_slots,
                                       int32_t num_heads, int32_t head_dim_k, int32_t head_dim_v,
                                       int32_t dtype, int32_t out_dtype, void *workspace,
                                       size_t workspace_bytes, void *stream);

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
 */
KDA_API int kda_recurrent_decode(const void *q, const void *k, const void *v,
                                 const float *g, const float *beta, float scale,
                                 float *state_pool, const int32_t *state_idx, void *out,
                                 int32_t num_seqs, int32_t num_slots, int32_t num_heads,
                                 int32_t head_dim_k, int32_t head_dim_v, int32_t dtype,
                                 int32_t out_dtype, void *stream);

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
                                            int32_t out_dtype, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* KDA_H_ */
