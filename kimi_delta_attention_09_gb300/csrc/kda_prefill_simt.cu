// kda_prefill_simt.cu -- chunked KDA prefill on CUDA cores, fp32 throughout.
//
// This is the chunked prompt path of vllm.cpp PR #110 ("chunk_kda prefill AOT
// port", commit description: gate cumsum in exp2 space -> decayed intra-chunk
// k.k^T and q.k^T -> unit-lower-triangular solve -> w/u recompute -> inter-chunk
// state propagation -> output) fused into one kernel.  It keeps every exponential
// exact per element (no factorisation), so it is robust for any gate g <= 0 and
// serves the fp32-input path and as the GPU-side cross-check of the tensor-core
// kernel.  It is not the fast path for bf16 inputs.
//
// For one chunk of rows r = 0..63 (zero-padded past the sequence end, which makes
// padded rows inert: k = v = beta = g = 0) starting from state h (K x V):
//     G_r      = log2(e) * sum_{i<=r} g_i                     (per key channel)
//     A_kk[r,i]= beta_r sum_c k_rc k_ic 2^(G_rc - G_ic)       i < r
//     A_qk[r,i]=        sum_c q_rc k_ic 2^(G_rc - G_ic)       i <= r
//     T        = (I + A_kk)^-1                                (forward substitution)
//     X        = beta * (v - (k * 2^G) h)                      (= beta (V - K~ h))
//     D        = T X                                          (corrected values)
//     o        = scale ((q * 2^G) h + A_qk D)
//     h       <- Diag(2^G_last) h + (k * 2^(G_last - G))^T D
// (D = T(beta V) - T(beta K~) h = U - W h, the w/u of the WY form applied to h.)
//
// Mapping: one CTA (256 threads) per (sequence, head, 32-column tile of V); the
// CTA walks its sequence chunk by chunk with the state tile resident in shared
// memory.  Row strides are padded by one float so the column walks of the
// pairwise products are bank-conflict free.
#include "kda_internal.cuh"

namespace kda {
namespace {

constexpr int kSimtThreads = 256;
constexpr int kVT = 32;            // V columns per CTA
static_assert(kSimtThreads - 2 * kChunk >= 128, "the row-normalising threads follow the cumsum threads");

template <int K>
struct SimtSmem {
    static constexpr int C = kChunk, KP = K + 1, CP = kChunk + 1;
    static constexpr int h = 0;                    // [K][kVT]
    static constexpr int gam = h + K * kVT;        // [C][KP]   G, later k * 2^G
    static constexpr int qs = gam + C * KP;        // [C][KP]   q, later q * 2^G
    static constexpr int ks = qs + C * KP;         // [C][KP]   k, later k * 2^(G_last - G)
    static constexpr int vs = ks + C * KP;         // [C][kVT]
    static constexpr int xs = vs + C * kVT;        // [C][kVT]  beta * X
    static constexpr int ds = xs + C * kVT;        // [C][kVT]  D
    static constexpr int akk = ds + C * kVT;       // [C][CP]
    static constexpr int aqk = akk + C * CP;       // [C][CP]
    static constexpr int tm = aqk + C * CP;        // [C][CP]
    static constexpr int bs = tm + C * CP;         // [C]
    static constexpr int glast = bs + C;           // [K]
    static constexpr int total = glast + K;
    static constexpr size_t bytes = sizeof(float) * (size_t)total;
};

template <typename Tin, typename Tout, int K, int V>
__global__ void __launch_bounds__(kSimtThreads)
kda_prefill_simt_kernel(PrefillArgs a)
{
    using L = SimtSmem<K>;
    constexpr int C = kChunk, KP = L::KP, CP = L::CP;
    constexpr int kTiles = V / kVT;
    extern __shared__ float sm[];
    float *hS = sm + L::h, *gam = sm + L::gam, *qs = sm + L::qs, *ks = sm + L::ks;
    float *vs = sm + L::vs, *xs = sm + L::xs, *ds = sm + L::ds;
    float *akk = sm + L::akk, *aqk = sm + L::aqk, *tm = sm + L::tm;
    float *bs = sm + L::bs, *glast = sm + L::glast;

    const int tid = threadIdx.x;
    const int64_t n = blockIdx.x / kTiles;
    const int vt = blockIdx.x % kTiles;
    const int h = blockIdx.y;
    const int H = a.num_heads;
    const Tin *q = static_cast<const Tin *>(a.q);
    const Tin *k = static_cast<const Tin *>(a.k);
    const Tin *v = static_cast<const Tin *>(a.v);
    Tout *out = static_cast<Tout *>(a.out);

    int64_t bos, eos;
    clamp_range(a.total_tokens, a.cu_seqlens[n], a.cu_seqlens[n + 1], bos, eos);

    const float *init;
    float *fin;
    prefill_state_ptrs(a, n, h, init, fin);
    for (int i = tid; i < K * kVT; i += kSimtThreads) {
        const int c = i / kVT, j = i % kVT;
        hS[i] = init ? init[(int64_t)c * V + vt * kVT + j] : 0.f;
    }

    for (int64_t t0 = bos; t0 < eos; t0 += C) {
        const int len = (int)((eos - t0) < C ? (eos - t0) : C);
        __syncthreads();   // previous chunk finished with every buffer
        for (int i = tid; i < C * K; i += kSimtThreads) {
            const int r = i / K, c = i % K;
            float qv = 0.f, kv = 0.f, gv = 0.f;
            if (r < len) {
                const int64_t idx = ((t0 + r) * H + h) * K + c;
                qv = to_f32(q[idx]); kv = to_f32(k[idx]); gv = a.g[idx] * kLog2e;
            }
            qs[r * KP + c] = qv; ks[r * KP + c] = kv; gam[r * KP + c] = gv;
        }
        for (int i = tid; i < C * kVT; i += kSimtThreads) {
            const int r = i / kVT, j = i % kVT;
            vs[i] = r < len ? to_f32(v[((t0 + r) * H + h) * V + vt * kVT + j]) : 0.f;
        }
        for (int r = tid; r < C; r += kSimtThreads)
            bs[r] = r < len ? a.beta[(t0 + r) * H + h] : 0.f;
        __syncthreads();

        // in-chunk cumulative gate (exp2 space), one thread per key channel; meanwhile the
        // in-kernel L2 normalisation of the q and k rows, one thread per row
        if (tid < K) {
            float acc = 0.f;
            for (int r = 0; r < C; ++r) { acc += gam[r * KP + tid]; gam[r * KP + tid] = acc; }
            glast[tid] = acc;
        } else if (tid >= kSimtThreads - 2 * C && (a.flags & kFlagQkL2Norm)) {
            const int rr = tid - (kSimtThreads - 2 * C);
            float *row = (rr < C ? qs : ks) + (rr % C) * KP;
            float ss = 0.f;
            for (int c = 0; c < K; ++c) ss += row[c] * row[c];
            const float sc = rsqrtf(ss + kQkL2NormEps);
            for (int c = 0; c < K; ++c) row[c] *= sc;
        }
        // T starts as the identity
        for (int i = tid; i < C * C; i += kSimtThreads) {
            const int r = i / C, j = i % C;
            tm[r * CP + j] = (r == j) ? 1.f : 0.f;
        }
        __syncthreads();

        // decayed pairwise products, exact exponentials, lower triangle incl. diagonal
        for (int p = tid; p < C * (C + 1) / 2; p += kSimtThreads) {
            int r = (int)((sqrtf(8.f * p + 1.f) - 1.f) * 0.5f);
            while (r * (r + 1) / 2 > p) --r;
            while ((r + 1) * (r + 2) / 2 <= p) ++r;
            const int i = p - r * (r + 1) / 2;
            float sk = 0.f, sq = 0.f;
            for (int c = 0; c < K; ++c) {
                const float kic = ks[i * KP + c] * exp2f(gam[r * KP + c] - gam[i * KP + c]);
                sk += ks[r * KP + c] * kic;
                sq += qs[r * KP + c] * kic;
            }
            akk[r * CP + i] = (i < r) ? bs[r] * sk : 0.f;
            aqk[r * CP + i] = sq;
        }
        __syncthreads();

        // T = (I + A_kk)^-1: row r of T from rows < r (forward substitution)
        for (int r = 1; r < C; ++r) {
            if (tid < r) {
                float s = 0.f;
                for (int m = tid; m < r; ++m) s += akk[r * CP + m] * tm[m * CP + tid];
                tm[r * CP + tid] = -s;
            }
            __syncthreads();
        }

        // decayed operands: q~ = q 2^G, k~ = k 2^G (into gam), k^ = k 2^(G_last - G)
        for (int i = tid; i < C * K; i += kSimtThreads) {
            const int r = i / K, c = i % K;
            const float gm = gam[r * KP + c];
            const float e = exp2f(gm);
            const float kv = ks[r * KP + c];
            qs[r * KP + c] *= e;
            gam[r * KP + c] = kv * e;
            ks[r * KP + c] = kv * exp2f(glast[c] - gm);
        }
        __syncthreads();

        // X = beta (v - k~ h)
        for (int i = tid; i < C * kVT; i += kSimtThreads) {
            const int r = i / kVT, j = i % kVT;
            float s = vs[i];
            for (int c = 0; c < K; ++c) s -= gam[r * KP + c] * hS[c * kVT + j];
            xs[i] = bs[r] * s;
        }
        __syncthreads();
        // D = T X
        for (int i = tid; i < C * kVT; i += kSimtThreads) {
            const int r = i / kVT, j = i % kVT;
            float s = 0.f;
            for (int m = 0; m <= r; ++m) s += tm[r * CP + m] * xs[m * kVT + j];
            ds[i] = s;
        }
        __syncthreads();
        // o = scale (q~ h + A_qk D)
        for (int i = tid; i < C * kVT; i += kSimtThreads) {
            const int r = i / kVT, j = i % kVT;
            if (r < len) {
                float s = 0.f;
                for (int c = 0; c < K; ++c) s += qs[r * KP + c] * hS[c * kVT + j];
                for (int m = 0; m <= r; ++m) s += aqk[r * CP + m] * ds[m * kVT + j];
                out[((t0 + r) * H + h) * V + vt * kVT + j] = from_f32<Tout>(a.scale * s);
            }
        }
        __syncthreads();
        // h <- Diag(2^G_last) h + k^^T D
        for (int i = tid; i < K * kVT; i += kSimtThreads) {
            const int c = i / kVT, j = i % kVT;
            float s = exp2f(glast[c]) * hS[i];
            for (int m = 0; m < C; ++m) s += ks[m * KP + c] * ds[m * kVT + j];
            hS[i] = s;
        }
    }
    __syncthreads();
    if (fin) {
        for (int i = tid; i < K * kVT; i += kSimtThreads) {
            const int c = i / kVT, j = i % kVT;
            fin[(int64_t)c * V + vt * kVT + j] = hS[i];
        }
    }
}

template <typename Tin, typename Tout, int K, int V>
cudaError_t launch_simt_t(const PrefillArgs &a, cudaStream_t stream)
{
    const size_t smem = SimtSmem<K>::bytes;
    cudaError_t e = cudaFuncSetAttribute(kda_prefill_simt_kernel<Tin, Tout, K, V>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid((unsigned)((int64_t)a.num_seqs * (V / kVT)), (unsigned)a.num_heads);
    kda_prefill_simt_kernel<Tin, Tout, K, V><<<grid, kSimtThreads, smem, stream>>>(a);
    return cudaGetLastError();
}

template <typename Tin, typename Tout>
cudaError_t launch_simt_dims(const PrefillArgs &a, cudaStream_t stream)
{
    if (a.head_dim_k == 128 && a.head_dim_v == 128) return launch_simt_t<Tin, Tout, 128, 128>(a, stream);
    if (a.head_dim_k == 128 && a.head_dim_v == 64) return launch_simt_t<Tin, Tout, 128, 64>(a, stream);
    if (a.head_dim_k == 64 && a.head_dim_v == 128) return launch_simt_t<Tin, Tout, 64, 128>(a, stream);
    return launch_simt_t<Tin, Tout, 64, 64>(a, stream);
}

}  // namespace

cudaError_t launch_prefill_simt(const PrefillArgs &a, cudaStream_t stream)
{
    if (a.num_seqs == 0) return cudaSuccess;
    if (a.dtype == kDtypeBF16)
        return a.out_dtype == kDtypeBF16 ? launch_simt_dims<__nv_bfloat16, __nv_bfloat16>(a, stream)
                                         : launch_simt_dims<__nv_bfloat16, float>(a, stream);
    return a.out_dtype == kDtypeBF16 ? launch_simt_dims<float, __nv_bfloat16>(a, stream)
                                     : launch_simt_dims<float, float>(a, stream);
}

}  // namespace kda
