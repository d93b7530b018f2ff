// kda_conv.cu -- the short causal convolution in front of the KDA op: a depthwise
// convolution of width W over the packed [q|k|v] channels, its last W - 1 inputs carried
// per sequence in paged tap slots.
//
// The pages place it before the KDA op as CausalConv1dFwd over the packed varlen prompt
// and CausalConv1dUpdate for the one-token decode step, with the carried conv_state
// split as chunk(3) into [q|k|v] (vllm.cpp PR #122 "fold Kimi-Linear onto the shared
// paged runner", block B2; vllm.cpp PR #113 "paged-incremental decode", commit body: the
// conv-tap carry).  Per sequence and channel c, with the carried taps prepended to the
// sequence's inputs (oldest first; zeros without a slot):
//     y_t = act(bias_c + sum_{j < W} w_{c,j} xe_{t+j}),   taps <- last W - 1 entries of xe
// act is the identity or SiLU.  Taps are stored with the inputs' element type and hold
// exact copies of inputs, so a prompt split anywhere and continued from its taps gives
// the unsplit result bit for bit.
//
// Mapping: a thread owns 4 adjacent channels (one 8- or 16-byte access per row); a CTA
// of 64 threads covers 256 channels over 128 tokens of the packed range and slides a
// register window of the W - 1 previous inputs down its tokens, so every input row is
// read from HBM once (plus a W - 1 row halo per tile) and every output row written once.
// Inside a sequence the tokens go in batches (8 rows of bf16, 4 of fp32) whose loads are
// all issued before the first is used: with one load in flight per thread the pass is
// bound by memory latency at about a third of the HBM bandwidth.
// The prompt pass reads the old taps; a second pass, ordered after it on the stream,
// writes the new taps (a sequence's old taps may be read by any of its tiles).
#include "kda_internal.cuh"

namespace kda {
namespace {

constexpr int kConvThreads = 64;
constexpr int kConvCh = 4;                               // channels per thread
constexpr int kConvTile = 128;                           // tokens per CTA
constexpr int kConvChPerCta = kConvThreads * kConvCh;    // 256
// tokens whose loads fly together: 64 bytes per thread (8 bf16 rows, 4 fp32 rows)
template <typename Tin> constexpr int conv_batch() { return sizeof(Tin) == 2 ? 8 : 4; }
constexpr int kConvUpdThreads = 256;                     // decode step: 1024 channels per CTA

__device__ __forceinline__ void load4(const float *p, float (&v)[4])
{
    const float4 x = *reinterpret_cast<const float4 *>(p);
    v[0] = x.x; v[1] = x.y; v[2] = x.z; v[3] = x.w;
}
__device__ __forceinline__ void load4(const __nv_bfloat16 *p, float (&v)[4])
{
    const uint2 x = *reinterpret_cast<const uint2 *>(p);
    const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&x.x));
    const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&x.y));
    v[0] = a.x; v[1] = a.y; v[2] = b.x; v[3] = b.y;
}
__device__ __forceinline__ void store4(float *p, const float (&v)[4])
{
    *reinterpret_cast<float4 *>(p) = make_float4(v[0], v[1], v[2], v[3]);
}
__device__ __forceinline__ void store4(__nv_bfloat16 *p, const float (&v)[4])
{
    __nv_bfloat162 a = __floats2bfloat162_rn(v[0], v[1]), b = __floats2bfloat162_rn(v[2], v[3]);
    uint2 x;
    x.x = *reinterpret_cast<uint32_t *>(&a);
    x.y = *reinterpret_cast<uint32_t *>(&b);
    *reinterpret_cast<uint2 *>(p) = x;
}
// raw copy of 4 elements (taps keep the inputs' exact bits)
template <typename T> struct Raw4;
template <> struct Raw4<float> { using type = float4; };
template <> struct Raw4<__nv_bfloat16> { using type = uint2; };

// SiLU with the fast reciprocal division (a few ulp; the IEEE division made the prompt
// pass issue-bound): z -> -inf gives z * 0 = -0, the limit
__device__ __forceinline__ float act(float z, int activation)
{
    return activation == kConvActSilu ? __fdividef(z, 1.f + __expf(-z)) : z;
}

// the W taps of channels c..c+3 (weight [D, W] row-major: 4W contiguous floats, 16-byte
// aligned because c is a multiple of 4 and the pointer is)
template <int W>
__device__ __forceinline__ void load_weights(const float *weight, const float *bias, int c,
                                             float (&w)[W][kConvCh], float (&b)[kConvCh])
{
    float f[kConvCh * W];
#pragma unroll
    for (int v = 0; v < W; ++v) {
        const float4 x = __ldg(reinterpret_cast<const float4 *>(weight + (int64_t)c * W) + v);
        f[4 * v] = x.x; f[4 * v + 1] = x.y; f[4 * v + 2] = x.z; f[4 * v + 3] = x.w;
    }
#pragma unroll
    for (int i = 0; i < kConvCh; ++i)
#pragma unroll
        for (int j = 0; j < W; ++j) w[j][i] = f[i * W + j];
    if (bias) {
        const float4 x = __ldg(reinterpret_cast<const float4 *>(bias + c));
        b[0] = x.x; b[1] = x.y; b[2] = x.z; b[3] = x.w;
    } else {
        b[0] = b[1] = b[2] = b[3] = 0.f;
    }
}

// the sequence holding token t: the largest n with cu[n] <= t (cu non-decreasing)
__device__ __forceinline__ int seq_of(const int32_t *cu, int N, int64_t t)
{
    int lo = 0, hi = N - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if ((int64_t)cu[mid] <= t) lo = mid;
        else hi = mid - 1;
    }
    return lo;
}

template <typename Tin>
__device__ __forceinline__ const Tin *tap_base(const ConvArgs &a, int n, int W)
{
    if (!a.state || W == 1) return nullptr;
    const int32_t slot = a.state_idx[n];
    if (slot < 0 || slot >= a.num_slots) return nullptr;
    return static_cast<const Tin *>(a.state) + (int64_t)slot * (W - 1) * a.dim;
}

template <typename Tin, typename Tout, int W>
__global__ void __launch_bounds__(kConvThreads, 16)
kda_conv_fwd_kernel(const ConvArgs a)
{
    const int c = (blockIdx.y * kConvThreads + threadIdx.x) * kConvCh;
    if (c >= a.dim) return;
    const int64_t T = a.total_tokens, D = a.dim;
    const int64_t t0 = (int64_t)blockIdx.x * kConvTile;
    const int64_t t1 = t0 + kConvTile < T ? t0 + kConvTile : T;
    const Tin *x = static_cast<const Tin *>(a.x);
    Tout *out = static_cast<Tout *>(a.out);

    float w[W][kConvCh], bias[kConvCh];
    load_weights<W>(a.weight, a.bias, c, w, bias);
    float win[W > 1 ? W - 1 : 1][kConvCh];   // the W - 1 inputs before the current token

    int n = seq_of(a.cu_seqlens, a.num_seqs, t0);
    int64_t bos, eos;
    clamp_range(T, a.cu_seqlens[n], a.cu_seqlens[n + 1], bos, eos);
    // window of position p of sequence n: an input, a carried tap, or zero
    auto fill = [&](int64_t t, const Tin *taps) {
#pragma unroll
        for (int j = 0; j < W - 1; ++j) {
            const int64_t p = t - (W - 1) + j;
            if (p >= bos) {
                load4(x + p * D + c, win[j]);
            } else if (taps) {
                load4(taps + (p - bos + (W - 1)) * D + c, win[j]);
            } else {
#pragma unroll
                for (int i = 0; i < kConvCh; ++i) win[j][i] = 0.f;
            }
        }
    };
    bool filled = false;   // the window holds the inputs before t of sequence n
    int64_t t = t0;
    while (t < t1) {
        while (t >= eos && n + 1 < a.num_seqs) {   // the sequence that holds t (empty ones skipped)
            ++n;
            clamp_range(T, a.cu_seqlens[n], a.cu_seqlens[n + 1], bos, eos);
            filled = false;
        }
        if (t >= eos) break;                     // past the last sequence: not written
        if (t < bos) { t = bos < t1 ? bos : t1; continue; }   // before it: not written
        if (!filled) {
            fill(t, tap_base<Tin>(a, n, W));
            filled = true;
        }
        const int64_t lim = eos < t1 ? eos : t1;
        constexpr int kConvBatch = conv_batch<Tin>();
        if (t + kConvBatch <= lim) {
            // a batch inside the sequence: inputs t .. t + kConvBatch - 1 (loaded raw, all in
            // flight at once), window before t; the window slides through the batch
            using R = typename Raw4<Tin>::type;
            R xr[kConvBatch];
#pragma unroll
            for (int u = 0; u < kConvBatch; ++u) xr[u] = *reinterpret_cast<const R *>(x + (t + u) * D + c);
#pragma unroll
            for (int u = 0; u < kConvBatch; ++u) {
                float xv[kConvCh], y[kConvCh];
                load4(reinterpret_cast<const Tin *>(&xr[u]), xv);
#pragma unroll
                for (int i = 0; i < kConvCh; ++i) {
                    float acc = bias[i];
#pragma unroll
                    for (int j = 0; j < W - 1; ++j) acc = fmaf(w[j][i], win[j][i], acc);
                    y[i] = act(fmaf(w[W - 1][i], xv[i], acc), a.activation);
                }
                store4(out + (t + u) * D + c, y);
#pragma unroll
                for (int j = 0; j + 1 < W - 1; ++j)
#pragma unroll
                    for (int i = 0; i < kConvCh; ++i) win[j][i] = win[j + 1][i];
                if (W > 1) {
#pragma unroll
                    for (int i = 0; i < kConvCh; ++i) win[W > 1 ? W - 2 : 0][i] = xv[i];
                }
            }
            t += kConvBatch;
            continue;
        }
        float xv[kConvCh], y[kConvCh];
        load4(x + t * D + c, xv);
#pragma unroll
        for (int i = 0; i < kConvCh; ++i) {
            float acc = bias[i];
#pragma unroll
            for (int j = 0; j < W - 1; ++j) acc = fmaf(w[j][i], win[j][i], acc);
            acc = fmaf(w[W - 1][i], xv[i], acc);
            y[i] = act(acc, a.activation);
        }
        store4(out + t * D + c, y);
#pragma unroll
        for (int j = 0; j + 1 < W - 1; ++j)
#pragma unroll
            for (int i = 0; i < kConvCh; ++i) win[j][i] = win[j + 1][i];
        if (W > 1) {
#pragma unroll
            for (int i = 0; i < kConvCh; ++i) win[W > 1 ? W - 2 : 0][i] = xv[i];
        }
        ++t;
    }
}

// New taps of each sequence with a slot: the last W - 1 entries of [old taps | inputs]
// (a thread reads and writes only its own channels, so the update is in place).
template <typename Tin, int W>
__global__ void __launch_bounds__(kConvThreads)
kda_conv_taps_kernel(const ConvArgs a)
{
    using R = typename Raw4<Tin>::type;
    const int c = (blockIdx.y * kConvThreads + threadIdx.x) * kConvCh;
    const int n = blockIdx.x;
    if (c >= a.dim) return;
    Tin *taps = const_cast<Tin *>(tap_base<Tin>(a, n, W));
    if (!taps) return;
    const int64_t D = a.dim;
    int64_t bos, eos;
    clamp_range(a.total_tokens, a.cu_seqlens[n], a.cu_seqlens[n + 1], bos, eos);
    const Tin *x = static_cast<const Tin *>(a.x);
    R nt[W > 1 ? W - 1 : 1];
#pragma unroll
    for (int i = 0; i < W - 1; ++i) {
        const int64_t p = eos - (W - 1) + i;
        nt[i] = p >= bos ? *reinterpret_cast<const R *>(x + p * D + c)
                         : *reinterpret_cast<const R *>(taps + (p - bos + (W - 1)) * D + c);
    }
#pragma unroll
    for (int i = 0; i < W - 1; ++i) *reinterpret_cast<R *>(taps + i * D + c) = nt[i];
}

// One token per sequence: output from the carried taps and the token, then the taps
// shift by one (in place, per thread).
template <typename Tin, typename Tout, int W>
__global__ void __launch_bounds__(kConvUpdThreads)
kda_conv_update_kernel(const ConvArgs a)
{
    using R = typename Raw4<Tin>::type;
    const int c = (blockIdx.y * kConvUpdThreads + threadIdx.x) * kConvCh;
    const int n = blockIdx.x;
    if (c >= a.dim) return;
    const int64_t D = a.dim;
    Tin *taps = const_cast<Tin *>(tap_base<Tin>(a, n, W));
    const Tin *xp = static_cast<const Tin *>(a.x) + n * D + c;
    R traw[W > 1 ? W - 1 : 1];
    float tv[W > 1 ? W - 1 : 1][kConvCh];
#pragma unroll
    for (int j = 0; j < W - 1; ++j) {
        if (taps) {
            traw[j] = *reinterpret_cast<const R *>(taps + j * D + c);
            load4(reinterpret_cast<const Tin *>(&traw[j]), tv[j]);
        } else {
#pragma unroll
            for (int i = 0; i < kConvCh; ++i) tv[j][i] = 0.f;
        }
    }
    const R xraw = *reinterpret_cast<const R *>(xp);
    float w[W][kConvCh], bias[kConvCh];
    load_weights<W>(a.weight, a.bias, c, w, bias);
    float xv[kConvCh], y[kConvCh];
    load4(reinterpret_cast<const Tin *>(&xraw), xv);
#pragma unroll
    for (int i = 0; i < kConvCh; ++i) {
        float acc = bias[i];
#pragma unroll
        for (int j = 0; j < W - 1; ++j) acc = fmaf(w[j][i], tv[j][i], acc);
        acc = fmaf(w[W - 1][i], xv[i], acc);
        y[i] = act(acc, a.activation);
    }
    store4(static_cast<Tout *>(a.out) + n * D + c, y);
    if (taps) {
#pragma unroll
        for (int j = 0; j + 1 < W - 1; ++j) *reinterpret_cast<R *>(taps + j * D + c) = traw[j + 1];
        if (W > 1) *reinterpret_cast<R *>(taps + (W > 1 ? W - 2 : 0) * D + c) = xraw;
    }
}

template <typename Tin, typename Tout, int W>
cudaError_t launch_fwd_w(const ConvArgs &a, cudaStream_t st)
{
    const dim3 chs((unsigned)((a.dim + kConvChPerCta - 1) / kConvChPerCta));
    if (a.total_tokens > 0) {
        const dim3 grid((unsigned)((a.total_tokens + kConvTile - 1) / kConvTile), chs.x);
        kda_conv_fwd_kernel<Tin, Tout, W><<<grid, kConvThreads, 0, st>>>(a);
    }
    if (W > 1 && a.state && a.num_seqs > 0)
        kda_conv_taps_kernel<Tin, W><<<dim3((unsigned)a.num_seqs, chs.x), kConvThreads, 0, st>>>(a);
    return cudaGetLastError();
}

template <typename Tin, typename Tout, int W>
cudaError_t launch_update_w(const ConvArgs &a, cudaStream_t st)
{
    const int per_cta = kConvUpdThreads * kConvCh;
    const dim3 grid((unsigned)a.num_seqs, (unsigned)((a.dim + per_cta - 1) / per_cta));
    kda_conv_update_kernel<Tin, Tout, W><<<grid, kConvUpdThreads, 0, st>>>(a);
    return cudaGetLastError();
}

template <template <typename, typename, int> class F, typename Tin, typename Tout>
cudaError_t by_width(const ConvArgs &a, cudaStream_t st)
{
    switch (a.width) {
    case 1: return F<Tin, Tout, 1>::run(a, st);
    case 2: return F<Tin, Tout, 2>::run(a, st);
    case 3: return F<Tin, Tout, 3>::run(a, st);
    default: return F<Tin, Tout, 4>::run(a, st);
    }
}
template <typename Tin, typename Tout, int W> struct Fwd {
    static cudaError_t run(const ConvArgs &a, cudaStream_t st) { return launch_fwd_w<Tin, Tout, W>(a, st); }
};
template <typename Tin, typename Tout, int W> struct Upd {
    static cudaError_t run(const ConvArgs &a, cudaStream_t st) { return launch_update_w<Tin, Tout, W>(a, st); }
};

template <template <typename, typename, int> class F>
cudaError_t dispatch(const ConvArgs &a, cudaStream_t st)
{
    if (a.dtype == kDtypeBF16)
        return a.out_dtype == kDtypeBF16 ? by_width<F, __nv_bfloat16, __nv_bfloat16>(a, st)
                                         : by_width<F, __nv_bfloat16, float>(a, st);
    return a.out_dtype == kDtypeBF16 ? by_width<F, float, __nv_bfloat16>(a, st)
                                     : by_width<F, float, float>(a, st);
}

}  // namespace

cudaError_t launch_conv_fwd(const ConvArgs &a, cudaStream_t stream)
{
    if (a.num_seqs == 0) return cudaSuccess;
    return dispatch<Fwd>(a, stream);
}

cudaError_t launch_conv_update(const ConvArgs &a, cudaStream_t stream)
{
    if (a.num_seqs == 0) return cudaSuccess;
    return dispatch<Upd>(a, stream);
}

}  // namespace kda
