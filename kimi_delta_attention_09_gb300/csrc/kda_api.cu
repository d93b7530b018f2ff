// kda_api.cu -- the C ABI of include/kda.h: argument validation, the byte-range
// alias guard and kernel selection.  No allocation, no synchronisation.
#include <cmath>
#include <cstdint>

#include "kda.h"
#include "kda_internal.cuh"

namespace {

thread_local int g_last_cuda_error = 0;

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

struct Range {
    const void *p;
    uint64_t bytes;
};

// [p, p + bytes) and [q, q + bytes) share at least one byte
bool overlaps(const Range &a, const Range &b)
{
    if (!a.p || !b.p || a.bytes == 0 || b.bytes == 0) return false;
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(a.p), a1 = a0 + a.bytes;
    const uintptr_t b0 = reinterpret_cast<uintptr_t>(b.p), b1 = b0 + b.bytes;
    return a0 < b1 && b0 < a1;
}

bool dims_supported(int32_t d) { return d == 64 || d == 128; }
bool dtype_supported(int32_t d) { return d == KDA_DTYPE_F32 || d == KDA_DTYPE_BF16; }

int finish(cudaError_t e)
{
    if (e != cudaSuccess) {
        g_last_cuda_error = (int)e;
        return KDA_ERR_CUDA;
    }
    return KDA_OK;
}

// Shapes the tensor-core kernel does not cover (fp32 inputs, K or V = 64) run on the
// exact CUDA-core kernel, which needs no workspace.
int launch_prefill_simt(const kda::PrefillArgs &a, void *stream)
{
    return finish(kda::launch_prefill_simt(a, static_cast<cudaStream_t>(stream)));
}

// The library's own prefill workspace: the status header and a record ring for 48
// clusters, in a file-scope device array (nothing is allocated; the array exists once per
// device for the life of the loaded library).  It serves every prefill entry point that
// takes no workspace argument; a device that can keep more than 48 clusters resident runs
// 48 (the clusters are persistent and walk the work items).
constexpr size_t kStaticClusters = 48;
constexpr size_t kStaticScratchBytes =
    kda::kPrefillRrHeaderBytes + kStaticClusters * kda::kPrefillRrRing * kda::kPrefillRrRecordBytes;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kStaticScratchBytes];

// Device address of the scratch on the current device.  Looked up on every call (cheap
// next to a prefill), so that a device reset, which reloads the module, cannot leave a
// stale address behind.
void *noalloc_scratch()
{
    void *p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) {
        g_last_cuda_error = (int)e;
        return nullptr;
    }
    return p;
}

// Tensor-core prefill on the library scratch (entry points without a workspace).
int launch_prefill_static(const kda::PrefillArgs &a, void *stream)
{
    if (!kda::prefill_rr_supported(a)) return launch_prefill_simt(a, stream);
    void *ws = noalloc_scratch();
    if (!ws) return KDA_ERR_CUDA;
    return finish(kda::launch_prefill_rr(a, ws, kStaticScratchBytes, static_cast<cudaStream_t>(stream)));
}

// Tensor-core prefill on a caller workspace, checked for size, alignment and overlap.
int launch_prefill_ws(const kda::PrefillArgs &a, const Range (&ranges)[9], void *workspace,
                      size_t workspace_bytes, void *stream)
{
    if (!kda::prefill_rr_supported(a)) return launch_prefill_simt(a, stream);
    const size_t need = kda::prefill_rr_workspace_bytes(a);
    if (!workspace || !aligned16(workspace) || workspace_bytes < need) return KDA_ERR_INVALID_ARG;
    const Range r_ws{workspace, (uint64_t)need};
    for (const Range &r : ranges)
        if (overlaps(r_ws, r)) return KDA_ERR_ALIAS;
    cudaPointerAttributes attr;
    int dev = -1;
    if (cudaPointerGetAttributes(&attr, workspace) != cudaSuccess || cudaGetDevice(&dev) != cudaSuccess ||
        attr.type != cudaMemoryTypeDevice || attr.device != dev) {
        cudaGetLastError();
        return KDA_ERR_INVALID_ARG;   // the workspace must be device memory of the current device
    }
    return finish(kda::launch_prefill_rr(a, workspace, need, static_cast<cudaStream_t>(stream)));
}

// Validation shared by kda_chunk_prefill and kda_chunk_prefill_ws: fills `a` and the
// byte ranges of every input and output (for the workspace alias check).
int check_prefill(const void *q, const void *k, const void *v, const float *g, const float *beta,
                  float scale, const float *init_state, const int32_t *cu_seqlens, void *out,
                  float *final_state, int64_t total_tokens, int32_t num_seqs, int32_t num_heads,
                  int32_t head_dim_k, int32_t head_dim_v, int32_t dtype, int32_t out_dtype,
                  kda::PrefillArgs &a, Range (&ranges)[9])
{
    if (total_tokens < 0 || num_seqs < 0 || num_heads < 1 || !std::isfinite(scale))
        return KDA_ERR_INVALID_ARG;
    if (!dtype_supported(dtype) || !dtype_supported(out_dtype)) return KDA_ERR_UNSUPPORTED;
    if (!dims_supported(head_dim_k) || !dims_supported(head_dim_v)) return KDA_ERR_UNSUPPORTED;
    if (num_seqs == 0) return KDA_OK;
    if (!cu_seqlens || !aligned16(cu_seqlens)) return KDA_ERR_INVALID_ARG;
    if (total_tokens > 0) {
        const void *req[] = {q, k, v, g, beta, out};
        for (const void *p : req)
            if (!p || !aligned16(p)) return KDA_ERR_INVALID_ARG;
    }
    if ((init_state && !aligned16(init_state)) || (final_state && !aligned16(final_state)))
        return KDA_ERR_INVALID_ARG;

    const uint64_t T = (uint64_t)total_tokens, H = (uint64_t)num_heads;
    const uint64_t K = (uint64_t)head_dim_k, V = (uint64_t)head_dim_v;
    const uint64_t es = dtype == KDA_DTYPE_BF16 ? 2 : 4;
    const uint64_t eo = out_dtype == KDA_DTYPE_BF16 ? 2 : 4;
    const uint64_t state_bytes = (uint64_t)num_seqs * H * K * V * 4;
    const Range in[] = {{q, T * H * K * es}, {k, T * H * K * es}, {v, T * H * V * es},
                        {g, T * H * K * 4}, {beta, T * H * 4},
                        {cu_seqlens, ((uint64_t)num_seqs + 1) * 4}};
    const Range r_out{out, T * H * V * eo}, r_init{init_state, state_bytes},
        r_final{final_state, state_bytes};
    for (const Range &r : in)
        if (overlaps(r_out, r) || overlaps(r_final, r)) return KDA_ERR_ALIAS;
    if (overlaps(r_out, r_init) || overlaps(r_out, r_final)) return KDA_ERR_ALIAS;
    if (overlaps(r_final, r_init) && final_state != init_state) return KDA_ERR_ALIAS;
    for (int i = 0; i < 6; ++i) ranges[i] = in[i];
    ranges[6] = r_out;
    ranges[7] = r_init;
    ranges[8] = r_final;

    a = kda::PrefillArgs{};
    a.q = q; a.k = k; a.v = v; a.g = g; a.beta = beta; a.scale = scale;
    a.init_state = init_state; a.cu_seqlens = cu_seqlens; a.out = out;
    a.final_state = final_state; a.total_tokens = total_tokens; a.num_seqs = num_seqs;
    a.num_heads = num_heads; a.head_dim_k = head_dim_k; a.head_dim_v = head_dim_v;
    a.dtype = dtype; a.out_dtype = out_dtype;
    return KDA_OK;
}

// Validation of the paged prefill entry points: fills `a` and the byte ranges of every
// input and of out and the pool (for the workspace alias check).
int check_prefill_paged(const void *q, const void *k, const void *v, const float *g,
                        const float *beta, float scale, float *state_pool,
                        const int32_t *state_idx, const int32_t *cu_seqlens, void *out,
                        int64_t total_tokens, int32_t num_seqs, int32_t num_slots,
                        int32_t num_heads, int32_t head_dim_k, int32_t head_dim_v, int32_t dtype,
                        int32_t out_dtype, kda::PrefillArgs &a, Range (&ranges)[9])
{
    if (total_tokens < 0 || num_seqs < 0 || num_slots < 0 || num_heads < 1 ||
        !std::isfinite(scale))
        return KDA_ERR_INVALID_ARG;
    if (!dtype_supported(dtype) || !dtype_supported(out_dtype)) return KDA_ERR_UNSUPPORTED;
    if (!dims_supported(head_dim_k) || !dims_supported(head_dim_v)) return KDA_ERR_UNSUPPORTED;
    if (num_seqs == 0) return KDA_OK;
    if (!cu_seqlens || !aligned16(cu_seqlens) || !state_idx || !aligned16(state_idx))
        return KDA_ERR_INVALID_ARG;
    if (num_slots > 0 && (!state_pool || !aligned16(state_pool))) return KDA_ERR_INVALID_ARG;
    if (total_tokens > 0) {
        const void *req[] = {q, k, v, g, beta, out};
        for (const void *p : req)
            if (!p || !aligned16(p)) return KDA_ERR_INVALID_ARG;
    }
    const uint64_t T = (uint64_t)total_tokens, H = (uint64_t)num_heads;
    const uint64_t K = (uint64_t)head_dim_k, V = (uint64_t)head_dim_v;
    const uint64_t es = dtype == KDA_DTYPE_BF16 ? 2 : 4;
    const uint64_t eo = out_dtype == KDA_DTYPE_BF16 ? 2 : 4;
    const Range in[] = {{q, T * H * K * es}, {k, T * H * K * es}, {v, T * H * V * es},
                        {g, T * H * K * 4}, {beta, T * H * 4},
                        {cu_seqlens, ((uint64_t)num_seqs + 1) * 4},
                        {state_idx, (uint64_t)num_seqs * 4}};
    const Range r_out{out, T * H * V * eo};
    const Range r_pool{state_pool, (uint64_t)num_slots * H * K * V * 4};
    for (const Range &r : in)
        if (overlaps(r_out, r) || overlaps(r_pool, r)) return KDA_ERR_ALIAS;
    if (overlaps(r_out, r_pool)) return KDA_ERR_ALIAS;
    for (int i = 0; i < 7; ++i) ranges[i] = in[i];
    ranges[7] = r_out;
    ranges[8] = r_pool;

    a = kda::PrefillArgs{};
    a.q = q; a.k = k; a.v = v; a.g = g; a.beta = beta; a.scale = scale;
    a.cu_seqlens = cu_seqlens; a.out = out;
    a.state_pool = state_pool; a.state_idx = state_idx; a.num_slots = num_slots;
    a.total_tokens = total_tokens; a.num_seqs = num_seqs;
    a.num_heads = num_heads; a.head_dim_k = head_dim_k; a.head_dim_v = head_dim_v;
    a.dtype = dtype; a.out_dtype = out_dtype;
    return KDA_OK;
}

}  // namespace

namespace kda {
void record_cuda_error(int e) { g_last_cuda_error = e; }
}  // namespace kda

extern "C" {

int kda_abi_version(void) { return KDA_ABI_VERSION; }

const char *kda_status_string(int status)
{
    switch (status) {
    case KDA_OK: return "KDA_OK";
    case KDA_ERR_INVALID_ARG: return "KDA_ERR_INVALID_ARG";
    case KDA_ERR_UNSUPPORTED: return "KDA_ERR_UNSUPPORTED";
    case KDA_ERR_ALIAS: return "KDA_ERR_ALIAS";
    case KDA_ERR_CUDA: return "KDA_ERR_CUDA";
    case KDA_ERR_TIMEOUT: return "KDA_ERR_TIMEOUT";
    default: return "KDA_ERR_UNKNOWN";
    }
}

int kda_last_cuda_error(void) { return g_last_cuda_error; }

int kda_chunk_prefill(const void *q, const void *k, const void *v,
                      const float *g, const float *beta, float scale,
                      const float *init_state, const int32_t *cu_seqlens,
                      void *out, float *final_state,
                      int64_t total_tokens, int32_t num_seqs, int32_t num_heads,
                      int32_t head_dim_k, int32_t head_dim_v, int32_t dtype,
                      int32_t out_dtype, int32_t flags, void *stream)
{
    kda::PrefillArgs a;
    Range ranges[9];
    const int st = check_prefill(q, k, v, g, beta, scale, init_state, cu_seqlens, out, final_state,
                                 total_tokens, num_seqs, num_heads, head_dim_k, head_dim_v, dtype,
                                 out_dtype, a, ranges);
    if (st != KDA_OK || num_seqs == 0) return st;
    if (flags & ~kda::kFlagQkL2Norm) return KDA_ERR_INVALID_ARG;
    a.flags = flags;
    return launch_prefill_static(a, stream);
}

size_t kda_chunk_prefill_workspace_bytes(int32_t num_seqs, int32_t num_heads, int32_t head_dim_k,
                                         int32_t head_dim_v, int32_t dtype)
{
    if (num_seqs <= 0 || num_heads < 1) return 0;
    kda::PrefillArgs a{};
    a.num_seqs = num_seqs; a.num_heads = num_heads; a.head_dim_k = head_dim_k;
    a.head_dim_v = head_dim_v; a.dtype = dtype;
    return kda::prefill_rr_workspace_bytes(a);
}

int kda_chunk_prefill_ws(const void *q, const void *k, const void *v,
                         const float *g, const float *beta, float scale,
                         const float *init_state, const int32_t *cu_seqlens,
                         void *out, float *final_state,
                         int64_t total_tokens, int32_t num_seqs, int32_t num_heads,
                         int32_t head_dim_k, int32_t head_dim_v, int32_t dtype,
                         int32_t out_dtype, void *workspace, size_t workspace_bytes, int32_t flags, void *stream)
{
    kda::PrefillArgs a;
    Range ranges[9];
    const int st = check_prefill(q, k, v, g, beta, scale, init_state, cu_seqlens, out, final_state,
                                 total_tokens, num_seqs, num_heads, head_dim_k, head_dim_v, dtype,
                                 out_dtype, a, ranges);
    if (st != KDA_OK || num_seqs == 0) return st;
    if (flags & ~kda::kFlagQkL2Norm) return KDA_ERR_INVALID_ARG;
    a.flags = flags;
    return launch_prefill_ws(a, ranges, workspace, workspace_bytes, stream);
}

int kda_chunk_prefill_noalloc(const void *q, const void *k, const void *v,
                              const float *g, const float *beta, float scale,
                              const float *init_state, const int32_t *cu_seqlens,
                              void *out, float *final_state,
                              int64_t total_tokens, int32_t num_seqs, int32_t num_heads,
                              int32_t head_dim_k, int32_t head_dim_v, int32_t dtype,
                              int32_t out_dtype, void *stream)
{
    kda::PrefillArgs a;
    Range ranges[9];
    const int st = check_prefill(q, k, v, g, beta, scale, init_state, cu_seqlens, out, final_state,
                                 total_tokens, num_seqs, num_heads, head_dim_k, head_dim_v, dtype,
                                 out_dtype, a, ranges);
    if (st != KDA_OK || num_seqs == 0) return st;
    return launch_prefill_static(a, stream);
}

int kda_chunk_prefill_paged(const void *q, const void *k, const void *v,
                            const float *g, const float *beta, float scale,
                            float *state_pool, const int32_t *state_idx,
                            const int32_t *cu_seqlens, void *out,
                            int64_t total_tokens, int32_t num_seqs, int32_t num_slots,
                            int32_t num_heads, int32_t head_dim_k, int32_t head_dim_v,
                            int32_t dtype, int32_t out_dtype, int32_t flags, void *stream)
{
    kda::PrefillArgs a;
    Range ranges[9];
    const int st = check_prefill_paged(q, k, v, g, beta, scale, state_pool, state_idx, cu_seqlens,
                                       out, total_tokens, num_seqs, num_slots, num_heads,
                                       head_dim_k, head_dim_v, dtype, out_dtype, a, ranges);
    if (st != KDA_OK || num_seqs == 0) return st;
    if (flags & ~kda::kFlagQkL2Norm) return KDA_ERR_INVALID_ARG;
    a.flags = flags;
    return launch_prefill_static(a, stream);
}

int kda_chunk_prefill_paged_ws(const void *q, const void *k, const void *v,
                               const float *g, const float *beta, float scale,
                               float *state_pool, const int32_t *state_idx,
                               const int32_t *cu_seqlens, void *out,
                               int64_t total_tokens, int32_t num_seqs, int32_t num_slots,
                               int32_t num_heads, int32_t head_dim_k, int32_t head_dim_v,
                               int32_t dtype, int32_t out_dtype, void *workspace,
                               size_t workspace_bytes, int32_t flags, void *stream)
{
    kda::PrefillArgs a;
    Range ranges[9];
    const int st = check_prefill_paged(q, k, v, g, beta, scale, state_pool, state_idx, cu_seqlens,
                                       out, total_tokens, num_seqs, num_slots, num_heads,
                                       head_dim_k, head_dim_v, dtype, out_dtype, a, ranges);
    if (st != KDA_OK || num_seqs == 0) return st;
    if (flags & ~kda::kFlagQkL2Norm) return KDA_ERR_INVALID_ARG;
    a.flags = flags;
    return launch_prefill_ws(a, ranges, workspace, workspace_bytes, stream);
}

int kda_chunk_prefill_status(const void *workspace, void *stream)
{
    void *ws = const_cast<void *>(workspace);
    if (!ws) ws = noalloc_scratch();
    if (!ws) return KDA_ERR_CUDA;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    int32_t word = 0;
    cudaError_t e = cudaStreamSynchronize(st);
    if (e == cudaSuccess) e = cudaMemcpy(&word, ws, sizeof(word), cudaMemcpyDeviceToHost);
    if (e == cudaSuccess && word != 0) e = cudaMemset(ws, 0, sizeof(word));
    if (e != cudaSuccess) {
        g_last_cuda_error = (int)e;
        return KDA_ERR_CUDA;
    }
    return word == kda::kStatusTimeout ? KDA_ERR_TIMEOUT : KDA_OK;
}

void kda_set_prefill_wait_limit(uint64_t nanoseconds)
{
    kda::set_prefill_wait_limit_ns((unsigned long long)nanoseconds);
}

static int recurrent_decode(const void *q, const void *k, const void *v,
                            const float *g, const float *beta, float scale,
                            void *state_pool, int32_t state_dtype, const int32_t *state_idx, void *out,
                            int32_t num_seqs, int32_t num_slots, int32_t num_heads,
                            int32_t head_dim_k, int32_t head_dim_v, int32_t dtype,
                            int32_t out_dtype, int32_t flags, void *stream)
{
    if (num_seqs < 0 || num_slots < 0 || num_heads < 1 || !std::isfinite(scale) ||
        (flags & ~kda::kFlagQkL2Norm))
        return KDA_ERR_INVALID_ARG;
    if (!dtype_supported(dtype) || !dtype_supported(out_dtype)) return KDA_ERR_UNSUPPORTED;
    if (!dims_supported(head_dim_k) || !dims_supported(head_dim_v)) return KDA_ERR_UNSUPPORTED;
    if (num_seqs == 0) return KDA_OK;
    const void *req[] = {q, k, v, g, beta, state_idx, out};
    for (const void *p : req)
        if (!p || !aligned16(p)) return KDA_ERR_INVALID_ARG;
    if (num_slots > 0 && (!state_pool || !aligned16(state_pool))) return KDA_ERR_INVALID_ARG;

    const uint64_t N = (uint64_t)num_seqs, H = (uint64_t)num_heads;
    const uint64_t K = (uint64_t)head_dim_k, V = (uint64_t)head_dim_v;
    const uint64_t es = dtype == KDA_DTYPE_BF16 ? 2 : 4;
    const uint64_t eo = out_dtype == KDA_DTYPE_BF16 ? 2 : 4;
    const uint64_t ep = state_dtype == KDA_DTYPE_BF16 ? 2 : 4;
    const Range in[] = {{q, N * H * K * es}, {k, N * H * K * es}, {v, N * H * V * es},
                        {g, N * H * K * 4}, {beta, N * H * 4}, {state_idx, N * 4}};
    const Range r_out{out, N * H * V * eo};
    const Range r_pool{state_pool, (uint64_t)num_slots * H * K * V * ep};
    for (const Range &r : in)
        if (overlaps(r_out, r) || overlaps(r_pool, r)) return KDA_ERR_ALIAS;
    if (overlaps(r_out, r_pool)) return KDA_ERR_ALIAS;

    kda::DecodeArgs a{};
    a.q = q; a.k = k; a.v = v; a.g = g; a.beta = beta; a.scale = scale;
    a.pool = state_pool; a.state_idx = state_idx; a.out = out;
    a.num_seqs = num_seqs; a.num_slots = num_slots; a.num_heads = num_heads;
    a.head_dim_k = head_dim_k; a.head_dim_v = head_dim_v; a.dtype = dtype;
    a.out_dtype = out_dtype; a.state_dtype = state_dtype; a.flags = flags;
    return finish(kda::launch_decode(a, static_cast<cudaStream_t>(stream)));
}

int kda_recurrent_decode(const void *q, const void *k, const void *v,
                         const float *g, const float *beta, float scale,
                         float *state_pool, const int32_t *state_idx, void *out,
                         int32_t num_seqs, int32_t num_slots, int32_t num_heads,
                         int32_t head_dim_k, int32_t head_dim_v, int32_t dtype,
                         int32_t out_dtype, int32_t flags, void *stream)
{
    return recurrent_decode(q, k, v, g, beta, scale, state_pool, KDA_DTYPE_F32, state_idx, out,
                            num_seqs, num_slots, num_heads, head_dim_k, head_dim_v, dtype,
                            out_dtype, flags, stream);
}

int kda_recurrent_decode_bf16_state(const void *q, const void *k, const void *v,
                                    const float *g, const float *beta, float scale,
                                    void *state_pool, const int32_t *state_idx, void *out,
                                    int32_t num_seqs, int32_t num_slots, int32_t num_heads,
                                    int32_t head_dim_k, int32_t head_dim_v, int32_t dtype,
                                    int32_t out_dtype, int32_t flags, void *stream)
{
    return recurrent_decode(q, k, v, g, beta, scale, state_pool, KDA_DTYPE_BF16, state_idx, out,
                            num_seqs, num_slots, num_heads, head_dim_k, head_dim_v, dtype,
                            out_dtype, flags, stream);
}

static int causal_conv(bool prompt, const void *x, const float *weight, const float *bias,
                       void *conv_state, const int32_t *state_idx, const int32_t *cu_seqlens,
                       void *out, int64_t total_tokens, int32_t num_seqs, int32_t num_slots,
                       int32_t dim, int32_t width, int32_t dtype, int32_t out_dtype,
                       int32_t activation, void *stream)
{
    if (total_tokens < 0 || num_seqs < 0 || num_slots < 0 || dim < 4 || (dim & 3) != 0 ||
        width < 1 || width > 4 || (activation != KDA_CONV_ACT_NONE && activation != KDA_CONV_ACT_SILU))
        return KDA_ERR_INVALID_ARG;
    if (!dtype_supported(dtype) || !dtype_supported(out_dtype)) return KDA_ERR_UNSUPPORTED;
    if (num_seqs == 0) return KDA_OK;
    const int64_t rows = prompt ? total_tokens : num_seqs;
    if (prompt && (!cu_seqlens || !aligned16(cu_seqlens))) return KDA_ERR_INVALID_ARG;
    if (rows > 0 && (!x || !aligned16(x) || !out || !aligned16(out))) return KDA_ERR_INVALID_ARG;
    if (!weight || !aligned16(weight) || (bias && !aligned16(bias))) return KDA_ERR_INVALID_ARG;
    if (conv_state && (!aligned16(conv_state) || !state_idx || !aligned16(state_idx)))
        return KDA_ERR_INVALID_ARG;

    const uint64_t D = (uint64_t)dim, W = (uint64_t)width;
    const uint64_t es = dtype == KDA_DTYPE_BF16 ? 2 : 4, eo = out_dtype == KDA_DTYPE_BF16 ? 2 : 4;
    const Range in[] = {{x, (uint64_t)rows * D * es}, {weight, D * W * 4}, {bias, D * 4},
                        {state_idx, conv_state ? (uint64_t)num_seqs * 4 : 0},
                        {cu_seqlens, prompt ? ((uint64_t)num_seqs + 1) * 4 : 0}};
    const Range r_out{out, (uint64_t)rows * D * eo};
    const Range r_state{conv_state, (uint64_t)num_slots * (W - 1) * D * es};
    for (const Range &r : in)
        if (overlaps(r_out, r) || overlaps(r_state, r)) return KDA_ERR_ALIAS;
    if (overlaps(r_out, r_state)) return KDA_ERR_ALIAS;

    kda::ConvArgs a{};
    a.x = x; a.weight = weight; a.bias = bias; a.state = conv_state; a.state_idx = state_idx;
    a.cu_seqlens = cu_seqlens; a.out = out; a.total_tokens = prompt ? total_tokens : num_seqs;
    a.num_seqs = num_seqs; a.num_slots = num_slots; a.dim = dim; a.width = width;
    a.dtype = dtype; a.out_dtype = out_dtype; a.activation = activation;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    return finish(prompt ? kda::launch_conv_fwd(a, st) : kda::launch_conv_update(a, st));
}

int kda_causal_conv1d_fwd(const void *x, const float *weight, const float *bias,
                          void *conv_state, const int32_t *state_idx,
                          const int32_t *cu_seqlens, void *out, int64_t total_tokens,
                          int32_t num_seqs, int32_t num_slots, int32_t dim,
                          int32_t width, int32_t dtype, int32_t out_dtype,
                          int32_t activation, void *stream)
{
    return causal_conv(true, x, weight, bias, conv_state, state_idx, cu_seqlens, out, total_tokens,
                       num_seqs, num_slots, dim, width, dtype, out_dtype, activation, stream);
}

int kda_causal_conv1d_update(const void *x, const float *weight, const float *bias,
                             void *conv_state, const int32_t *state_idx, void *out,
                             int32_t num_seqs, int32_t num_slots, int32_t dim,
                             int32_t width, int32_t dtype, int32_t out_dtype,
                             int32_t activation, void *stream)
{
    return causal_conv(false, x, weight, bias, conv_state, state_idx, nullptr, out, 0, num_seqs,
                       num_slots, dim, width, dtype, out_dtype, activation, stream);
}

}  // extern "C"
