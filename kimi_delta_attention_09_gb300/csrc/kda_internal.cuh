// kda_internal.cuh -- internal declarations shared by the KDA CUDA sources.
// Not part of the public ABI (include/kda.h is).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace kda {

// One prefill call, already validated by the C-ABI layer.
struct PrefillArgs {
    const void *q, *k, *v;        // [T, H, K] / [T, H, V], dtype
    const float *g, *beta;        // [T, H, K] fp32, [T, H] fp32
    float scale;
    const float *init_state;      // [N, H, K, V] or nullptr
    const int32_t *cu_seqlens;    // [N + 1]
    void *out;                    // [T, H, V], out_dtype
    float *final_state;           // [N, H, K, V] or nullptr
    float *state_pool;            // [S, H, K, V] or nullptr: states live in slots state_idx[n]
    const int32_t *state_idx;     // [N] (with state_pool)
    int32_t num_slots;
    int64_t total_tokens;
    int32_t num_seqs, num_heads, head_dim_k, head_dim_v, dtype, out_dtype;
    int32_t flags;                // kFlag* bits
};

// Base pointers of the (sequence n, head h) state for a prefill: the caller's
// init/final arrays, or slot state_idx[n] of the pool (nullptr for both when the
// slot index is out of range, which makes the sequence start from zeros and drop
// its final state).
__device__ __forceinline__ void prefill_state_ptrs(const PrefillArgs &a, int64_t n, int h,
                                                   const float *&init, float *&fin)
{
    const int64_t kv = (int64_t)a.head_dim_k * a.head_dim_v;
    if (a.state_pool) {
        const int32_t slot = a.state_idx[n];
        const bool ok = slot >= 0 && slot < a.num_slots;
        fin = ok ? a.state_pool + ((int64_t)slot * a.num_heads + h) * kv : nullptr;
        init = fin;
    } else {
        const int64_t off = (n * a.num_heads + h) * kv;
        init = a.init_state ? a.init_state + off : nullptr;
        fin = a.final_state ? a.final_state + off : nullptr;
    }
}

// One decode step, already validated by the C-ABI layer.
struct DecodeArgs {
    const void *q, *k, *v;        // [N, H, K] / [N, H, V], dtype
    const float *g, *beta;        // [N, H, K], [N, H]
    float scale;
    void *pool;                   // [S, H, K, V], state_dtype (fp32 or bf16 storage)
    const int32_t *state_idx;     // [N]
    void *out;                    // [N, H, V], out_dtype
    int32_t num_seqs, num_slots, num_heads, head_dim_k, head_dim_v, dtype, out_dtype, state_dtype;
    int32_t flags;                // kFlag* bits
};

constexpr int kFlagQkL2Norm = 1;        // normalise q and k rows over K in the kernel
constexpr float kQkL2NormEps = 1e-6f;   // q / sqrt(sum q^2 + eps)
constexpr int kDtypeF32 = 0;
constexpr int kDtypeBF16 = 1;
constexpr int kChunk = 64;              // tokens per prefill chunk
constexpr float kLog2e = 1.4426950408889634f;

// Chunked prefill on CUDA cores in fp32 (any supported dtype / head size).
cudaError_t launch_prefill_simt(const PrefillArgs &a, cudaStream_t stream);

// Chunked prefill on tensor cores (bf16 q/k/v with K = V = 128): one 4-CTA cluster per
// (sequence, head) work item; the per-chunk operands are built once per head and shared
// through a ring of records in a device workspace.
bool prefill_rr_supported(const PrefillArgs &a);
constexpr size_t kPrefillRrRecordBytes = 66816;   // one chunk's operand record
constexpr int kPrefillRrRing = 8;                 // records per cluster
constexpr size_t kPrefillRrHeaderBytes = 256;     // workspace header: device status word
constexpr int kStatusTimeout = 1;                 // status word: a bounded wait ran out
// bytes for min(N H, resident clusters) clusters on the current device
size_t prefill_rr_workspace_bytes(const PrefillArgs &a);
// the launch uses min(N H, resident clusters, clusters the workspace holds) clusters
cudaError_t launch_prefill_rr(const PrefillArgs &a, void *workspace, size_t workspace_bytes,
                              cudaStream_t stream);
// limit of every wait inside the prefill kernel (0: the default of 2 s)
void set_prefill_wait_limit_ns(unsigned long long ns);

// The short causal convolution over packed channels with carried taps.
constexpr int kConvActNone = 0, kConvActSilu = 1;
struct ConvArgs {
    const void *x;                // [T, D] (prompt) or [N, D] (decode), dtype
    const float *weight, *bias;   // [D, W], [D] or nullptr
    void *state;                  // [S, W - 1, D] dtype, or nullptr (zero taps, nothing kept)
    const int32_t *state_idx;     // [N] (with state)
    const int32_t *cu_seqlens;    // [N + 1] (prompt)
    void *out;                    // like x, out_dtype
    int64_t total_tokens;
    int32_t num_seqs, num_slots, dim, width, dtype, out_dtype, activation;
};
cudaError_t launch_conv_fwd(const ConvArgs &a, cudaStream_t stream);
cudaError_t launch_conv_update(const ConvArgs &a, cudaStream_t stream);

// The thread's last CUDA error as kda_last_cuda_error reports it (set by every entry point
// that returns KDA_ERR_CUDA).
void record_cuda_error(int e);

// One-token paged decode.
cudaError_t launch_decode(const DecodeArgs &a, cudaStream_t stream);

// ---------------------------------------------------------------- device helpers
__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename T> __device__ __forceinline__ T from_f32(float x);
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) {
    return __float2bfloat16_rn(x);
}

// Clamp a device-read sequence range to [0, total] (an inverted pair is empty).
__device__ __forceinline__ void clamp_range(int64_t total, int32_t b, int32_t e,
                                            int64_t &bos, int64_t &eos) {
    bos = b < 0 ? 0 : (b > total ? total : b);
    eos = e < 0 ? 0 : (e > total ? total : e);
    if (eos < bos) eos = bos;
}

}  // namespace kda
