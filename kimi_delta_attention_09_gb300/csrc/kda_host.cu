// kda_host.cu -- the host-to-host chunked prefill: inputs in host memory, outputs back in
// host memory, the copies overlapped with the prefill.
//
// The prompt path of vllm.cpp PR #113 ("paged-incremental decode", commit body: prefill
// the prompt once with the chunked kernel, carry the state) starts from a prompt on the
// host.  Here the packed token range is cut into pieces on 64-token boundaries; piece s is
// copied in on one stream, prefilled on the caller's stream (every sequence clipped to the
// piece, its state carried in place from the previous piece: a prefill split at any token
// and continued from the carried state is the unsplit prefill), and its output rows are
// copied back on a third stream, so that the copy-in of piece s + 1 and the copy-out of
// piece s - 1 run beside the prefill of piece s.
//
// Everything lives in one caller-owned device buffer: the prefill workspace first (its
// status word at the buffer's base), then the device copies of the inputs, the output,
// the carried state and the per-piece cu_seqlens (written by a small kernel from the
// copied cu_seqlens, so the host side needs no staging memory of its own).
#include <cstdint>
#include <cstring>
#include <mutex>

#include "kda.h"
#include "kda_internal.cuh"

namespace {

constexpr int kChunk = 64;
constexpr int kMaxPieces = KDA_HOST_MAX_PIECES;
constexpr int kMaxDevices = 64;

size_t up256(size_t x) { return (x + 255) & ~size_t(255); }

struct HostLayout {
    size_t ws, ws_bytes, q, k, v, g, beta, out, state, cu, cup, total;
    size_t row;                         // int32 entries per per-piece cu_seqlens row
    int pieces;
    int64_t bounds[kMaxPieces + 1];     // piece s = packed tokens [bounds[s], bounds[s + 1])
};

// Piece bounds: at most `pieces` pieces, inner bounds on 64-token boundaries, the pieces as
// even in chunks as the count allows.
void piece_bounds(int64_t T, int pieces, HostLayout &L)
{
    const int64_t nch = (T + kChunk - 1) / kChunk;
    int64_t segs = pieces;
    if (segs > (nch > 1 ? nch : 1)) segs = nch > 1 ? nch : 1;
    L.pieces = (int)segs;
    for (int s = 0; s < L.pieces; ++s) L.bounds[s] = kChunk * ((nch * s) / segs);
    L.bounds[L.pieces] = T;
}

bool host_layout(int64_t T, int32_t N, int32_t H, int32_t K, int32_t V, int32_t dtype,
                 int32_t out_dtype, int32_t pieces, HostLayout &L)
{
    if (T < 0 || N < 1 || H < 1 || pieces < 1 || pieces > kMaxPieces) return false;
    if ((dtype != KDA_DTYPE_F32 && dtype != KDA_DTYPE_BF16) ||
        (out_dtype != KDA_DTYPE_F32 && out_dtype != KDA_DTYPE_BF16))
        return false;
    if ((K != 64 && K != 128) || (V != 64 && V != 128)) return false;
    const size_t es = dtype == KDA_DTYPE_BF16 ? 2 : 4, eo = out_dtype == KDA_DTYPE_BF16 ? 2 : 4;
    const size_t rows = (size_t)T * H;
    piece_bounds(T, pieces, L);
    L.row = ((size_t)N + 1 + 3) / 4 * 4;
    L.ws_bytes = kda_chunk_prefill_workspace_bytes(N, H, K, V, dtype);
    size_t o = 0;
    L.ws = o;    o = up256(o + L.ws_bytes);
    L.q = o;     o = up256(o + rows * K * es);
    L.k = o;     o = up256(o + rows * K * es);
    L.v = o;     o = up256(o + rows * V * es);
    L.g = o;     o = up256(o + rows * K * 4);
    L.beta = o;  o = up256(o + rows * 4);
    L.out = o;   o = up256(o + rows * V * eo);
    L.state = o; o = up256(o + (size_t)N * H * K * V * 4);
    L.cu = o;    o = up256(o + L.row * 4);
    L.cup = o;   o = up256(o + (size_t)L.pieces * L.row * 4);
    L.total = o;
    return true;
}

struct PieceBounds {
    int64_t b[kMaxPieces + 1];
};

// cup[s][n] = cu[n] clipped to piece s and counted from its first token
__global__ void piece_cu_kernel(const int32_t *__restrict__ cu, int32_t *__restrict__ cup, int n1,
                                int pieces, int row, PieceBounds pb)
{
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= pieces * row) return;
    const int s = i / row, n = i % row;
    const int64_t b0 = pb.b[s], len = pb.b[s + 1] - b0;
    int64_t x = n < n1 ? (int64_t)cu[n] - b0 : 0;
    x = x < 0 ? 0 : (x > len ? len : x);
    cup[i] = (int32_t)x;
}

// Streams and events of the copy pipeline, created on first use per device and kept until
// exit; enqueueing is serialised by a mutex (the device work of separate calls may still
// overlap: each call has its own device buffer, and an event's earlier waits keep the
// record they were enqueued against).
struct Pipe {
    bool ready = false;
    cudaStream_t in = nullptr, out = nullptr;
    cudaEvent_t start = nullptr, end = nullptr, in_done[kMaxPieces] = {}, run_done[kMaxPieces] = {};
};
std::mutex g_pipe_mu;
Pipe g_pipe[kMaxDevices];

cudaError_t pipe_for_device(int dev, Pipe *&p)
{
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    p = &g_pipe[dev];
    if (p->ready) return cudaSuccess;
    cudaError_t e = cudaStreamCreateWithFlags(&p->in, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&p->out, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&p->start, cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&p->end, cudaEventDisableTiming);
    for (int s = 0; s < kMaxPieces && e == cudaSuccess; ++s) {
        e = cudaEventCreateWithFlags(&p->in_done[s], cudaEventDisableTiming);
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(&p->run_done[s], cudaEventDisableTiming);
    }
    if (e == cudaSuccess) p->ready = true;
    return e;
}

struct HostRange {
    const void *p;
    size_t bytes;
};
bool host_overlap(const HostRange &a, const HostRange &b)
{
    if (!a.p || !b.p || !a.bytes || !b.bytes) return false;
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(a.p), b0 = reinterpret_cast<uintptr_t>(b.p);
    return a0 < b0 + b.bytes && b0 < a0 + a.bytes;
}

int host_fail(cudaError_t e)
{
    kda::record_cuda_error((int)e);
    return KDA_ERR_CUDA;
}

}  // namespace

extern "C" {

size_t kda_chunk_prefill_host_device_bytes(int64_t total_tokens, int32_t num_seqs,
                                           int32_t num_heads, int32_t head_dim_k,
                                           int32_t head_dim_v, int32_t dtype, int32_t out_dtype,
                                           int32_t pieces)
{
    HostLayout L;
    if (!host_layout(total_tokens, num_seqs, num_heads, head_dim_k, head_dim_v, dtype, out_dtype,
                     pieces, L))
        return 0;
    return L.total;
}

int kda_chunk_prefill_host(const void *q, const void *k, const void *v, const float *g,
                           const float *beta, float scale, const float *init_state,
                           const int32_t *cu_seqlens, void *out, float *final_state,
                           int64_t total_tokens, int32_t num_seqs, int32_t num_heads,
                           int32_t head_dim_k, int32_t head_dim_v, int32_t dtype,
                           int32_t out_dtype, int32_t pieces, void *device_buffer,
                           size_t device_buffer_bytes, int32_t flags, void *stream)
{
    if (num_seqs == 0 && total_tokens >= 0 && num_heads >= 1) return KDA_OK;
    HostLayout L;
    if (!host_layout(total_tokens, num_seqs, num_heads, head_dim_k, head_dim_v, dtype, out_dtype,
                     pieces, L))
        return (pieces < 1 || pieces > kMaxPieces || total_tokens < 0 || num_seqs < 0 || num_heads < 1)
                   ? KDA_ERR_INVALID_ARG : KDA_ERR_UNSUPPORTED;
    if (flags & ~KDA_FLAG_QK_L2NORM) return KDA_ERR_INVALID_ARG;
    if (!cu_seqlens || (total_tokens > 0 && (!q || !k || !v || !g || !beta || !out)))
        return KDA_ERR_INVALID_ARG;
    {   // the host outputs are written while later pieces' inputs are still being read
        const size_t rows = (size_t)total_tokens * num_heads;
        const size_t es = dtype == KDA_DTYPE_BF16 ? 2 : 4, eo = out_dtype == KDA_DTYPE_BF16 ? 2 : 4;
        const size_t sb = (size_t)num_seqs * num_heads * head_dim_k * head_dim_v * 4;
        const HostRange in[] = {{q, rows * head_dim_k * es}, {k, rows * head_dim_k * es},
                                {v, rows * head_dim_v * es}, {g, rows * head_dim_k * 4},
                                {beta, rows * 4}, {init_state, sb},
                                {cu_seqlens, ((size_t)num_seqs + 1) * 4}};
        const HostRange ro{out, rows * head_dim_v * eo}, rf{final_state, sb};
        for (const HostRange &r : in) {
            if (host_overlap(ro, r)) return KDA_ERR_ALIAS;
            // final_state == init_state carries the state in place on the host: the initial
            // state's copy-in precedes the first prefill, the final copy-out follows the last
            const bool carry = r.p == init_state && final_state == init_state;
            if (!carry && host_overlap(rf, r)) return KDA_ERR_ALIAS;
        }
        if (host_overlap(ro, rf)) return KDA_ERR_ALIAS;
    }
    if (!device_buffer || (reinterpret_cast<uintptr_t>(device_buffer) & 255u) != 0 ||
        device_buffer_bytes < L.total)
        return KDA_ERR_INVALID_ARG;
    int dev = -1;
    cudaPointerAttributes attr;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaPointerGetAttributes(&attr, device_buffer) != cudaSuccess ||
        attr.type != cudaMemoryTypeDevice || attr.device != dev) {
        cudaGetLastError();
        return KDA_ERR_INVALID_ARG;   // the buffer must be device memory of the current device
    }

    const size_t H = (size_t)num_heads, K = (size_t)head_dim_k, V = (size_t)head_dim_v;
    const size_t es = dtype == KDA_DTYPE_BF16 ? 2 : 4, eo = out_dtype == KDA_DTYPE_BF16 ? 2 : 4;
    const size_t qrow = H * K * es, vrow = H * V * es, grow = H * K * 4, brow = H * 4, orow = H * V * eo;
    const size_t state_bytes = (size_t)num_seqs * H * K * V * 4;
    unsigned char *base = static_cast<unsigned char *>(device_buffer);
    unsigned char *dq = base + L.q, *dk = base + L.k, *dv = base + L.v, *dg = base + L.g,
                  *db = base + L.beta, *dout = base + L.out;
    float *dstate = reinterpret_cast<float *>(base + L.state);
    int32_t *dcu = reinterpret_cast<int32_t *>(base + L.cu), *dcup = reinterpret_cast<int32_t *>(base + L.cup);
    cudaStream_t main = static_cast<cudaStream_t>(stream);

    std::lock_guard<std::mutex> lock(g_pipe_mu);
    Pipe *p = nullptr;
    cudaError_t e = pipe_for_device(dev, p);
    if (e != cudaSuccess) return host_fail(e);
    auto h2d = [&](void *dst, const void *src, size_t n) {
        if (e == cudaSuccess && n) e = cudaMemcpyAsync(dst, src, n, cudaMemcpyHostToDevice, p->in);
    };
    // copies start after the caller's earlier work on `stream` (which may still use the buffer)
    e = cudaEventRecord(p->start, main);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(p->in, p->start, 0);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(p->out, p->start, 0);
    h2d(dcu, cu_seqlens, ((size_t)num_seqs + 1) * 4);
    if (e == cudaSuccess) {
        PieceBounds pb;
        std::memcpy(pb.b, L.bounds, sizeof(pb.b));
        const int n = L.pieces * (int)L.row;
        piece_cu_kernel<<<(n + 255) / 256, 256, 0, p->in>>>(dcu, dcup, num_seqs + 1, L.pieces, (int)L.row, pb);
        e = cudaGetLastError();
    }
    if (init_state) h2d(dstate, init_state, state_bytes);
    else if (e == cudaSuccess) e = cudaMemsetAsync(dstate, 0, state_bytes, p->in);
    for (int s = 0; s < L.pieces && e == cudaSuccess; ++s) {
        const size_t b0 = (size_t)L.bounds[s], n = (size_t)(L.bounds[s + 1] - L.bounds[s]);
        h2d(dq + b0 * qrow, static_cast<const unsigned char *>(q) + b0 * qrow, n * qrow);
        h2d(dk + b0 * qrow, static_cast<const unsigned char *>(k) + b0 * qrow, n * qrow);
        h2d(dv + b0 * vrow, static_cast<const unsigned char *>(v) + b0 * vrow, n * vrow);
        h2d(dg + b0 * grow, reinterpret_cast<const unsigned char *>(g) + b0 * grow, n * grow);
        h2d(db + b0 * brow, reinterpret_cast<const unsigned char *>(beta) + b0 * brow, n * brow);
        if (e == cudaSuccess) e = cudaEventRecord(p->in_done[s], p->in);
    }
    if (e != cudaSuccess) return host_fail(e);
    for (int s = 0; s < L.pieces; ++s) {
        const size_t b0 = (size_t)L.bounds[s], n = (size_t)(L.bounds[s + 1] - L.bounds[s]);
        e = cudaStreamWaitEvent(main, p->in_done[s], 0);
        if (e != cudaSuccess) return host_fail(e);
        const int st = kda_chunk_prefill_ws(dq + b0 * qrow, dk + b0 * qrow, dv + b0 * vrow,
                                            reinterpret_cast<const float *>(dg + b0 * grow),
                                            reinterpret_cast<const float *>(db + b0 * brow), scale,
                                            dstate, dcup + (size_t)s * L.row, dout + b0 * orow, dstate,
                                            (int64_t)n, num_seqs, num_heads, head_dim_k, head_dim_v,
                                            dtype, out_dtype, L.ws_bytes ? base + L.ws : nullptr,
                                            L.ws_bytes, flags, stream);
        if (st != KDA_OK) return st;
        e = cudaEventRecord(p->run_done[s], main);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(p->out, p->run_done[s], 0);
        if (e == cudaSuccess && n)
            e = cudaMemcpyAsync(static_cast<unsigned char *>(out) + b0 * orow, dout + b0 * orow, n * orow,
                                cudaMemcpyDeviceToHost, p->out);
        if (e != cudaSuccess) return host_fail(e);
    }
    if (final_state) e = cudaMemcpyAsync(final_state, dstate, state_bytes, cudaMemcpyDeviceToHost, p->out);
    if (e == cudaSuccess) e = cudaEventRecord(p->end, p->out);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(main, p->end, 0);   // `stream` covers every copy
    return e == cudaSuccess ? KDA_OK : host_fail(e);
}

}  // extern "C"
