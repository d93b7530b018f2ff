// kda_decode.cu -- one-token KDA decode over paged fp32 states, in place.
//
// The decode side of the prefill=chunk / decode=recurrent split (vllm.cpp PR #113
// "paged-incremental decode", commit body: one token advanced per step from the
// carried state) over paged state slots selected per sequence (vllm.cpp PR #122
// "fold Kimi-Linear onto the shared paged runner", block B2: gather / scatter by the
// per-sequence state indices).  The gather, the update and the scatter are fused:
// every selected state is read from HBM once and written back once.
//
// Per (sequence n, head h), with S = pool[state_idx[n], h] (K x V, row = key channel) and,
// with the in-kernel L2 normalisation, k and q first scaled to unit norm over K (the
// norms reduce beside S^T k and S^T q, and every product is linear in k and in q):
//     S <- Diag(exp g) S;   u = S^T k;   d = beta (v - u);   S <- S + k d^T;
//     o  = scale S^T q = scale ((Diag(exp g) S_old)^T q + (k.q) d)
// so S is read once, both reductions (against k and q) run on the decayed state,
// and the write-back happens once d is known.
//
// Mapping: one CTA of 128 threads per (n, h, 32-column slice of V).  Thread t owns
// columns [4*(t%8), +4) of the slice (one float4) on rows t/8 + 16*j, j < K/16, so
// a warp reads four 128-byte row segments per instruction (fully coalesced) and
// every thread has K/16 independent 16-byte loads in flight before it computes.
// The work is HBM-bound (K*V*8 bytes of state per (n, h) against ~7 K*V flops).
//
// State storage: fp32, or bf16 (the pool's element type as a configuration of the
// state dtype, vllm.cpp PR #122 "fold Kimi-Linear onto the shared paged runner",
// block B3, kda_state_dtype).  A bf16 pool is read into fp32, the step runs in fp32
// exactly as for an fp32 pool, the output is read from the fp32 updated state, and
// the state is rounded to nearest-even bf16 only where it is stored: half the bytes
// per step, one rounding of the carried state per step.  Its kernel takes 64 columns
// per CTA (8 per thread, one 16-byte load and store per row), so that a CTA moves as
// many bytes as on an fp32 pool.
#include "kda_internal.cuh"

namespace kda {
namespace {

constexpr int kDecThreads = 128;
constexpr int kDecCols = 32;   // V columns per CTA

template <typename Tin, typename Tout, int K, int V, bool kL2>
__global__ void __launch_bounds__(kDecThreads)
kda_decode_kernel(DecodeArgs a)
{
    constexpr int kSlices = V / kDecCols;
    constexpr int kRowsPerThread = K / 16;
    const int tid = threadIdx.x;
    const int cg = tid & 7;          // column group (float4)
    const int rg = tid >> 3;         // row group 0..15
    const int64_t n = blockIdx.x / kSlices;
    const int slice = blockIdx.x % kSlices;
    const int h = blockIdx.y;
    const int H = a.num_heads;
    const int col0 = slice * kDecCols + cg * 4;

    const int32_t slot = a.state_idx[n];
    Tout *out = static_cast<Tout *>(a.out) + (n * H + h) * V + col0;
    if (slot < 0 || slot >= a.num_slots) {           // bounds check: touch no slot
        if (rg == 0) {
#pragma unroll
            for (int i = 0; i < 4; ++i) out[i] = from_f32<Tout>(0.f);
        }
        return;
    }

    float4 *S = reinterpret_cast<float4 *>(
        static_cast<float *>(a.pool) + ((int64_t)slot * H + h) * (int64_t)(K * V) + col0);
    const Tin *kp = static_cast<const Tin *>(a.k) + (n * H + h) * K;
    const Tin *qp = static_cast<const Tin *>(a.q) + (n * H + h) * K;
    const float *gp = a.g + (n * H + h) * K;

    // issue every state load first
    float4 s[kRowsPerThread];
#pragma unroll
    for (int j = 0; j < kRowsPerThread; ++j)
        s[j] = __ldcs(S + (int64_t)(rg + 16 * j) * (V / 4));

    float kr[kRowsPerThread], qr[kRowsPerThread], dr[kRowsPerThread];
#pragma unroll
    for (int j = 0; j < kRowsPerThread; ++j) {
        const int c = rg + 16 * j;
        kr[j] = to_f32(kp[c]);
        qr[j] = to_f32(qp[c]);
        dr[j] = expf(gp[c]);
    }

    // decay, then partial reductions against k and q (and k.q, |k|^2, |q|^2) over this
    // thread's rows
    float pk[4] = {0.f, 0.f, 0.f, 0.f}, pq[4] = {0.f, 0.f, 0.f, 0.f}, kq = 0.f, kk = 0.f, qq = 0.f;
#pragma unroll
    for (int j = 0; j < kRowsPerThread; ++j) {
        s[j].x *= dr[j]; s[j].y *= dr[j]; s[j].z *= dr[j]; s[j].w *= dr[j];
        pk[0] += s[j].x * kr[j]; pk[1] += s[j].y * kr[j];
        pk[2] += s[j].z * kr[j]; pk[3] += s[j].w * kr[j];
        pq[0] += s[j].x * qr[j]; pq[1] += s[j].y * qr[j];
        pq[2] += s[j].z * qr[j]; pq[3] += s[j].w * qr[j];
        kq += kr[j] * qr[j];
        if (kL2) {
            kk += kr[j] * kr[j];
            qq += qr[j] * qr[j];
        }
    }
    // reduce over the 4 row groups of this warp (lanes differing in bits 3, 4)
#pragma unroll
    for (int off = 8; off <= 16; off <<= 1) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            pk[i] += __shfl_xor_sync(0xffffffffu, pk[i], off);
            pq[i] += __shfl_xor_sync(0xffffffffu, pq[i], off);
        }
        kq += __shfl_xor_sync(0xffffffffu, kq, off);
        if (kL2) {
            kk += __shfl_xor_sync(0xffffffffu, kk, off);
            qq += __shfl_xor_sync(0xffffffffu, qq, off);
        }
    }
    // ... and over the 4 warps
    __shared__ float red[kDecThreads / 32][8][kL2 ? 11 : 9];
    const int warp = tid >> 5, lane = tid & 31;
    if (lane < 8) {
#pragma unroll
        for (int i = 0; i < 4; ++i) { red[warp][lane][i] = pk[i]; red[warp][lane][4 + i] = pq[i]; }
        red[warp][lane][8] = kq;
        if (kL2) {
            red[warp][lane][9] = kk;
            red[warp][lane][10] = qq;
        }
    }
    __syncthreads();
    float u[4] = {0.f, 0.f, 0.f, 0.f}, qs[4] = {0.f, 0.f, 0.f, 0.f};
    kq = kk = qq = 0.f;
#pragma unroll
    for (int w = 0; w < kDecThreads / 32; ++w) {
#pragma unroll
        for (int i = 0; i < 4; ++i) { u[i] += red[w][cg][i]; qs[i] += red[w][cg][4 + i]; }
        kq += red[w][cg][8];
        if (kL2) {
            kk += red[w][cg][9];
            qq += red[w][cg][10];
        }
    }
    if (kL2) {   // in-kernel L2 normalisation: every product above is linear in k and in q
        const float rk = rsqrtf(kk + kQkL2NormEps), rq = rsqrtf(qq + kQkL2NormEps);
#pragma unroll
        for (int i = 0; i < 4; ++i) { u[i] *= rk; qs[i] *= rq; }
        kq *= rk * rq;
#pragma unroll
        for (int j = 0; j < kRowsPerThread; ++j) kr[j] *= rk;
    }

    const float beta = a.beta[n * H + h];
    const Tin *vp = static_cast<const Tin *>(a.v) + (n * H + h) * V + col0;
    float d[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) d[i] = beta * (to_f32(vp[i]) - u[i]);

    // write back S + k d^T
#pragma unroll
    for (int j = 0; j < kRowsPerThread; ++j) {
        float4 w = s[j];
        w.x += kr[j] * d[0]; w.y += kr[j] * d[1]; w.z += kr[j] * d[2]; w.w += kr[j] * d[3];
        __stcs(S + (int64_t)(rg + 16 * j) * (V / 4), w);
    }
    if (rg == 0) {
#pragma unroll
        for (int i = 0; i < 4; ++i) out[i] = from_f32<Tout>(a.scale * (qs[i] + kq * d[i]));
    }
}

constexpr int kDecCols16 = 64;   // V columns per CTA on a bf16 pool

// The same step on a bf16 pool: thread t owns columns [8 (t % 8), +8) of the CTA's
// 64 on rows t / 8 + 16 j; the state is widened to fp32 where it is used and rounded to
// nearest-even bf16 on store.  The CTA's 16 KB slice of the slot comes in by cp.async into
// shared memory (each thread reads back only its own rows): the loads in flight then do
// not hold registers, and 8 CTAs fit on an SM instead of 5.
template <typename Tin, typename Tout, int K, int V, bool kL2>
__global__ void __launch_bounds__(kDecThreads, 8)
kda_decode_bf16_state_kernel(DecodeArgs a)
{
    constexpr int kSlices = V / kDecCols16;
    constexpr int kRowsPerThread = K / 16;
    const int tid = threadIdx.x;
    const int cg = tid & 7;          // column group (8 columns)
    const int rg = tid >> 3;         // row group 0..15
    const int64_t n = blockIdx.x / kSlices;
    const int slice = blockIdx.x % kSlices;
    const int h = blockIdx.y;
    const int H = a.num_heads;
    const int col0 = slice * kDecCols16 + cg * 8;

    const int32_t slot = a.state_idx[n];
    Tout *out = static_cast<Tout *>(a.out) + (n * H + h) * V + col0;
    if (slot < 0 || slot >= a.num_slots) {           // bounds check: touch no slot
        if (rg == 0) {
#pragma unroll
            for (int i = 0; i < 8; ++i) out[i] = from_f32<Tout>(0.f);
        }
        return;
    }

    __nv_bfloat16 *S = static_cast<__nv_bfloat16 *>(a.pool) + ((int64_t)slot * H + h) * (int64_t)(K * V) + col0;
    const Tin *kp = static_cast<const Tin *>(a.k) + (n * H + h) * K;
    const Tin *qp = static_cast<const Tin *>(a.q) + (n * H + h) * K;
    const float *gp = a.g + (n * H + h) * K;

    __shared__ __align__(16) uint4 stile[K][8];
#pragma unroll
    for (int j = 0; j < kRowsPerThread; ++j) {
        const uint32_t dst = (uint32_t)__cvta_generic_to_shared(&stile[rg + 16 * j][cg]);
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" :: "r"(dst), "l"(S + (int64_t)(rg + 16 * j) * V) : "memory");
    }
    asm volatile("cp.async.commit_group;\n" ::: "memory");

    float kr[kRowsPerThread], qr[kRowsPerThread], dr[kRowsPerThread];
#pragma unroll
    for (int j = 0; j < kRowsPerThread; ++j) {
        const int c = rg + 16 * j;
        kr[j] = to_f32(kp[c]);
        qr[j] = to_f32(qp[c]);
        dr[j] = expf(gp[c]);
    }

    asm volatile("cp.async.wait_group 0;\n" ::: "memory");   // this thread's own rows
    // the decayed row, widened where it is needed
    auto decayed = [&](int j, float (&x)[8]) {
        const uint4 rw = stile[rg + 16 * j][cg];
        const __nv_bfloat162 *w = reinterpret_cast<const __nv_bfloat162 *>(&rw);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float2 f = __bfloat1622float2(w[e]);
            x[2 * e] = f.x * dr[j];
            x[2 * e + 1] = f.y * dr[j];
        }
    };
    float pk[8], pq[8], kq = 0.f, kk = 0.f, qq = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) pk[i] = pq[i] = 0.f;
#pragma unroll
    for (int j = 0; j < kRowsPerThread; ++j) {
        float x[8];
        decayed(j, x);
#pragma unroll
        for (int i = 0; i < 8; ++i) { pk[i] += x[i] * kr[j]; pq[i] += x[i] * qr[j]; }
        kq += kr[j] * qr[j];
        if (kL2) {
            kk += kr[j] * kr[j];
            qq += qr[j] * qr[j];
        }
    }
#pragma unroll
    for (int off = 8; off <= 16; off <<= 1) {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            pk[i] += __shfl_xor_sync(0xffffffffu, pk[i], off);
            pq[i] += __shfl_xor_sync(0xffffffffu, pq[i], off);
        }
        kq += __shfl_xor_sync(0xffffffffu, kq, off);
        if (kL2) {
            kk += __shfl_xor_sync(0xffffffffu, kk, off);
            qq += __shfl_xor_sync(0xffffffffu, qq, off);
        }
    }
    __shared__ float red[kDecThreads / 32][8][kL2 ? 19 : 17];
    const int warp = tid >> 5, lane = tid & 31;
    if (lane < 8) {
#pragma unroll
        for (int i = 0; i < 8; ++i) { red[warp][lane][i] = pk[i]; red[warp][lane][8 + i] = pq[i]; }
        red[warp][lane][16] = kq;
        if (kL2) {
            red[warp][lane][17] = kk;
            red[warp][lane][18] = qq;
        }
    }
    __syncthreads();
    float u[8], qs[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) u[i] = qs[i] = 0.f;
    kq = kk = qq = 0.f;
#pragma unroll
    for (int w = 0; w < kDecThreads / 32; ++w) {
#pragma unroll
        for (int i = 0; i < 8; ++i) { u[i] += red[w][cg][i]; qs[i] += red[w][cg][8 + i]; }
        kq += red[w][cg][16];
        if (kL2) {
            kk += red[w][cg][17];
            qq += red[w][cg][18];
        }
    }
    if (kL2) {   // in-kernel L2 normalisation: every product above is linear in k and in q
        const float rk = rsqrtf(kk + kQkL2NormEps), rq = rsqrtf(qq + kQkL2NormEps);
#pragma unroll
        for (int i = 0; i < 8; ++i) { u[i] *= rk; qs[i] *= rq; }
        kq *= rk * rq;
#pragma unroll
        for (int j = 0; j < kRowsPerThread; ++j) kr[j] *= rk;
    }

    const float beta = a.beta[n * H + h];
    const Tin *vp = static_cast<const Tin *>(a.v) + (n * H + h) * V + col0;
    float d[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) d[i] = beta * (to_f32(vp[i]) - u[i]);

#pragma unroll
    for (int j = 0; j < kRowsPerThread; ++j) {
        float x[8];
        decayed(j, x);
        uint4 w;
        uint32_t *pw = reinterpret_cast<uint32_t *>(&w);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            __nv_bfloat162 b2 = __floats2bfloat162_rn(x[2 * e] + kr[j] * d[2 * e],
                                                      x[2 * e + 1] + kr[j] * d[2 * e + 1]);
            pw[e] = *reinterpret_cast<uint32_t *>(&b2);
        }
        __stcs(reinterpret_cast<uint4 *>(S + (int64_t)(rg + 16 * j) * V), w);
    }
    if (rg == 0) {
#pragma unroll
        for (int i = 0; i < 8; ++i) out[i] = from_f32<Tout>(a.scale * (qs[i] + kq * d[i]));
    }
}

template <typename Tin, typename Tout, int K, int V, bool kL2>
void launch_decode_l2(const DecodeArgs &a, cudaStream_t stream)
{
    if (a.state_dtype == kDtypeBF16) {
        dim3 grid((unsigned)((int64_t)a.num_seqs * (V / kDecCols16)), (unsigned)a.num_heads);
        kda_decode_bf16_state_kernel<Tin, Tout, K, V, kL2><<<grid, kDecThreads, 0, stream>>>(a);
    } else {
        dim3 grid((unsigned)((int64_t)a.num_seqs * (V / kDecCols)), (unsigned)a.num_heads);
        kda_decode_kernel<Tin, Tout, K, V, kL2><<<grid, kDecThreads, 0, stream>>>(a);
    }
}

template <typename Tin, typename Tout, int K, int V>
cudaError_t launch_decode_t(const DecodeArgs &a, cudaStream_t stream)
{
    if (a.flags & kFlagQkL2Norm) launch_decode_l2<Tin, Tout, K, V, true>(a, stream);
    else launch_decode_l2<Tin, Tout, K, V, false>(a, stream);
    return cudaGetLastError();
}

template <typename Tin, typename Tout>
cudaError_t launch_decode_dims(const DecodeArgs &a, cudaStream_t stream)
{
    if (a.head_dim_k == 128 && a.head_dim_v == 128) return launch_decode_t<Tin, Tout, 128, 128>(a, stream);
    if (a.head_dim_k == 128 && a.head_dim_v == 64) return launch_decode_t<Tin, Tout, 128, 64>(a, stream);
    if (a.head_dim_k == 64 && a.head_dim_v == 128) return launch_decode_t<Tin, Tout, 64, 128>(a, stream);
    return launch_decode_t<Tin, Tout, 64, 64>(a, stream);
}

}  // namespace

cudaError_t launch_decode(const DecodeArgs &a, cudaStream_t stream)
{
    if (a.num_seqs == 0) return cudaSuccess;
    if (a.dtype == kDtypeBF16)
        return a.out_dtype == kDtypeBF16 ? launch_decode_dims<__nv_bfloat16, __nv_bfloat16>(a, stream)
                                         : launch_decode_dims<__nv_bfloat16, float>(a, stream);
    return a.out_dtype == kDtypeBF16 ? launch_decode_dims<float, __nv_bfloat16>(a, stream)
                                     : launch_decode_dims<float, float>(a, stream);
}

}  // namespace kda
