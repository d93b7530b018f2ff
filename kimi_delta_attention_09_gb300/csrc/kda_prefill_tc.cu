// kda_prefill_tc.cu -- chunked KDA prefill on tensor cores (bf16 inputs, K = V = 128).
//
// The chunked prompt path of vllm.cpp PR #110 ("chunk_kda prefill AOT port",
// commit description: in-chunk gate cumsum in exp2 space, the decayed intra-chunk
// k.k^T, the unit-lower-triangular solve, the w/u recompute, the inter-chunk state
// propagation and the output), fused into ONE kernel so that every input byte is
// read from HBM once and only the output and the final state are written.
//
// Algebra per chunk of rows r = 0..63 (padded rows past the sequence end are zero,
// which makes them inert), with state h (K x V, fp32) on entry:
//     G       = log2(e) * cumsum(g)                        (per key channel)
//     A_kk    = beta * strict_lower( sum_c k_r k_i 2^(G_r - G_i) )
//     A_qk    = lower( sum_c q_r k_i 2^(G_r - G_i) )
//     T       = (I + A_kk)^-1
//     X       = beta * (v - K~ h),  K~ = k 2^G               (beta-scaled residual)
//     D       = T X                                          (corrected values, = U - W h)
//     o       = scale * (Q~ h + A_qk D),  Q~ = q 2^G
//     h      <- Diag(2^G_last) h + K^T D,  K^ = k 2^(G_last - G)
//
// Numerics (checked against the fp64 oracle before this kernel was written):
// * All tensor-core operands are fp16 (10-bit mantissa), accumulation fp32; the state
//   and the triangular solve are fp32.  bf16 operands miss a 2e-3 relative bar by
//   2-3x; fp16 operands meet it with ~3x margin.
// * fp16 range is handled by factoring 2^(G_r - G_i) around a per-channel reference
//   m_R = G at row 16R+8 of each 16-row block R:  a_r = x_r 2^(G_r - m_R(r)),
//   b_i = k_i 2^(m_R(i) - G_i), and for an off-diagonal block pair the factor
//   2^(m_R - m_I) <= 1 is applied to b in registers.  Every stored factor spans at
//   most 8 steps of the gate.  A chunk whose factors leave [2^-8, 2^8] (gates below
//   about -0.7 per step sustained over 8 steps) takes an exact-exponential CUDA-core
//   path for its intra-chunk matrices instead; its result is the same algebra.
//
// Mapping: one CTA (8 warps) per (sequence, head, 32-column tile of V); it walks its
// sequence chunk by chunk.  Per chunk, all warps first build the intra-chunk
// operands (gate cumsum, factors, A_kk / A_qk with mma.sync, blocked solve), then
// run the state step on tensor cores; the state tile lives in registers (fp32),
// mirrored to shared memory in fp16 as the next chunk's MMA operand.  The raw
// inputs of chunk j+1 are fetched with cp.async while chunk j's solve and state
// step run.
#include <cstring>

#include <cuda.h>
#include <cuda_fp16.h>
#include <cudaTypedefs.h>

#include "kda_internal.cuh"

namespace kda {
namespace {

constexpr int kThreads = 256;
constexpr int C = kChunk;        // 64 rows per chunk
constexpr int KD = 128;          // key dim
constexpr int VD = 128;          // value dim
constexpr int VT = 32;           // value columns per CTA
constexpr int kVTiles = VD / VT;
constexpr int LD128 = KD + 8;    // f16 row stride (halves) of 128-column tiles: 272 B
constexpr int LD64 = C + 8;      // f16 row stride of 64-column tiles: 144 B
constexpr int LDV = VT + 1;      // fp32 V tile stride
constexpr int LDA = C + 1;       // fp32 A_kk / T stride
constexpr float kFactorMax = 256.f;   // fp16 factor bound (2^8) of the fast path

// Shared memory map (byte offsets).
struct Smem {
    static constexpr int q_raw = 0;                          // bf16 [64][128]
    static constexpr int k_raw = q_raw + C * KD * 2;         // bf16 [64][128]
    static constexpr int g_raw = k_raw + C * KD * 2;         // f32  [64][128] -> G
    static constexpr int v_raw = g_raw + C * KD * 4;         // bf16 [64][32]
    static constexpr int b_raw = v_raw + C * VT * 2;         // f32  [64]
    static constexpr int a_k = b_raw + C * 4;                // f16 [64][LD128]; later A_kk/T f32 [64][LDA]
    static constexpr int a_q = a_k + C * LD128 * 2;          // f16 [64][LD128]
    static constexpr int b_k = a_q + C * LD128 * 2;          // f16 [64][LD128]
    static constexpr int nkt = b_k + C * LD128 * 2;          // f16 -K~ [64][LD128]
    static constexpr int qt = nkt + C * LD128 * 2;           // f16  Q~ [64][LD128]
    static constexpr int kh = qt + C * LD128 * 2;            // f16  K^ [64][LD128] (row i, col c)
    static constexpr int tm = kh + C * LD128 * 2;            // f16  T  [64][LD64]
    static constexpr int aqk = tm + C * LD64 * 2;            // f16  A_qk [64][LD64]
    static constexpr int ht = aqk + C * LD64 * 2;            // f16  h^T [32][LD128]
    static constexpr int xt = ht + VT * LD128 * 2;           // f16  (beta X)^T [32][LD64]; xt+dt hold fp16 A_kk in the solve
    static constexpr int dt = xt + VT * LD64 * 2;            // f16  D^T [32][LD64]
    static constexpr int vs = dt + VT * LD64 * 2;            // f32  V [64][LDV]
    static constexpr int beta = vs + C * LDV * 4;            // f32  [64]
    static constexpr int dec = beta + C * 4;                 // f32  [128] 2^G_last
    static constexpr int mref = dec + KD * 4;                // f32  [4][128] m_R
    static constexpr int pm = mref + 4 * KD * 4;             // f32  [4][128] 2^m_R
    static constexpr int fm = pm + 4 * KD * 4;               // f32  [4][128] 2^(G_last - m_R)
    static constexpr int rho = fm + 4 * KD * 4;              // f16  [6][128] 2^(m_R - m_I), I < R
    static constexpr int flag = rho + 6 * KD * 2;            // int
    static constexpr int mbar = flag + 8;                    // u64 mbarrier of the chunk loads
    static constexpr int total = mbar + 8;
};
static_assert(Smem::total <= 232448, "shared memory budget");
static_assert(C * LDA * 4 <= C * LD128 * 2, "A_kk must fit in the a_k region");
static_assert(Smem::dt == Smem::xt + VT * LD64 * 2 && 2 * VT == C, "fp16 A_kk spans xt and dt");

// ------------------------------------------------------------------ PTX helpers
__device__ __forceinline__ uint32_t smem_u32(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                        uint32_t &r3)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];\n"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                          uint32_t &r3)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];\n"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}

// D += A * B, m16n8k16, fp16 operands, fp32 accumulators
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1)
{
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
        "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void cp_async4(uint32_t dst, const void *src, int src_bytes)
{
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;\n"
                 :: "r"(dst), "l"(src), "r"(src_bytes));
}

__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n"); }

// 3-D tiled TMA load (tensor map in kernel-parameter space) completing on an mbarrier
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap *map, int x, int y, int z,
                                            uint32_t mbar)
{
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
        "[%0], [%1, {%2, %3, %4}], [%5];\n"
        :: "r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(mbar)
        : "memory");
}

__device__ __forceinline__ void mbar_init(uint32_t mbar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" :: "r"(mbar), "r"(count) : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t mbar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n"
                 :: "r"(mbar), "r"(bytes) : "memory");
}

// Bounded wait for the phase with parity `parity` to complete; false on timeout.
__device__ __forceinline__ bool mbar_wait(uint32_t mbar, uint32_t parity)
{
    for (int i = 0; i < (1 << 22); ++i) {
        uint32_t done;
        asm volatile("{\n.reg .pred p;\nmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
                     "selp.u32 %0, 1, 0, p;\n}\n"
                     : "=r"(done) : "r"(mbar), "r"(parity) : "memory");
        if (done) return true;
    }
    return false;
}

__device__ __forceinline__ void fence_proxy_async_smem()
{
    asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
}
__device__ __forceinline__ void cp_async_wait_all()
{
    asm volatile("cp.async.wait_group 0;\n" ::: "memory");
}

__device__ __forceinline__ uint32_t pack_h2(float lo, float hi)
{
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&h);
}

__device__ __forceinline__ uint32_t hmul2_u32(uint32_t a, uint32_t b)
{
    __half2 r = __hmul2(*reinterpret_cast<__half2 *>(&a), *reinterpret_cast<__half2 *>(&b));
    return *reinterpret_cast<uint32_t *>(&r);
}

// ldmatrix lane addresses (element offsets) -----------------------------------
// A operand, 16x16 at (row0, col0) of a row-major tile with leading dimension ld.
__device__ __forceinline__ int a_off(int lane, int row0, int col0, int ld)
{
    return (row0 + (lane & 15)) * ld + col0 + ((lane >> 4) << 3);
}
// B operand stored [n][k] (k contiguous): two n-tiles (n0, n0+8) x k16 at k0.
__device__ __forceinline__ int bnk_off(int lane, int n0, int k0, int ld)
{
    return (n0 + (lane & 7) + ((lane >> 4) << 3)) * ld + k0 + (((lane >> 3) & 1) << 3);
}
// B operand stored [k][n] (n contiguous), read transposed: two n-tiles at (k0, n0).
__device__ __forceinline__ int bkn_off(int lane, int k0, int n0, int ld)
{
    return (k0 + (lane & 7) + (((lane >> 3) & 1) << 3)) * ld + n0 + ((lane >> 4) << 3);
}

// Tensor maps of q, k, g (box 128 channels x 1 head x 64 tokens) and v (box 32
// columns x 1 head x 64 tokens), built on the host for each call.
struct TmaMaps {
    CUtensorMap q, k, g, v;
};

// ------------------------------------------------------------------ loads
// Tokens [t0, t0+64) of q, k, g and of this CTA's 32 v columns arrive as four TMA
// tiles that complete on the chunk mbarrier (rows past the end of the tensor are
// zero-filled by the TMA unit; rows past the end of the SEQUENCE are zeroed after
// arrival, see zero_tail_rows).  beta (strided by H) uses 4-byte cp.async.  Called
// by all threads after a barrier that ends every read of the raw buffers.
__device__ __forceinline__ void issue_chunk_loads(unsigned char *sm, const PrefillArgs &a,
                                                  const TmaMaps &maps, int64_t t0, int len,
                                                  int h, int vt, int tid)
{
    if (tid < C) {
        const int valid = tid < len;
        const int64_t row = t0 + (valid ? tid : 0);
        cp_async4(smem_u32(sm + Smem::b_raw + tid * 4), a.beta + row * a.num_heads + h, valid ? 4 : 0);
    }
    cp_async_commit();
    if (tid == 0) {
        const uint32_t mbar = smem_u32(sm + Smem::mbar);
        fence_proxy_async_smem();   // earlier generic reads of the raw buffers come first
        mbar_arrive_expect_tx(mbar, C * (2 * KD * 2 + KD * 4 + VT * 2));
        const int z = (int)t0;
        tma_load_3d(smem_u32(sm + Smem::q_raw), &maps.q, 0, h, z, mbar);
        tma_load_3d(smem_u32(sm + Smem::k_raw), &maps.k, 0, h, z, mbar);
        tma_load_3d(smem_u32(sm + Smem::g_raw), &maps.g, 0, h, z, mbar);
        tma_load_3d(smem_u32(sm + Smem::v_raw), &maps.v, vt * VT, h, z, mbar);
    }
}

// Zero the rows [len, 64) of the raw tiles (tokens of the next sequence).
__device__ __forceinline__ void zero_tail_rows(unsigned char *sm, int len, int tid)
{
    for (int e = tid; e < (C - len) * KD / 8; e += kThreads) {   // 16 B per store
        const int r = len + e / (KD / 8), piece = e % (KD / 8);
        const uint4 z = make_uint4(0, 0, 0, 0);
        *reinterpret_cast<uint4 *>(sm + Smem::q_raw + (r * KD + piece * 8) * 2) = z;
        *reinterpret_cast<uint4 *>(sm + Smem::k_raw + (r * KD + piece * 8) * 2) = z;
        *reinterpret_cast<uint4 *>(sm + Smem::g_raw + (r * KD + piece * 8) * 4) = z;
        *reinterpret_cast<uint4 *>(sm + Smem::g_raw + (r * KD + piece * 8 + 4) * 4) = z;
        if (piece < VT / 8)
            *reinterpret_cast<uint4 *>(sm + Smem::v_raw + (r * VT + piece * 8) * 2) = z;
    }
}

// Exact-exponential intra-chunk matrices for chunks outside the fp16 factor range:
// A_kk (fp32, into the a_k region) and A_qk (fp16), and the decayed operands
// -K~, Q~, K^ recomputed with one exponential per element.
__device__ void exact_intra_chunk(unsigned char *sm, int tid)
{
    const __nv_bfloat16 *qr = reinterpret_cast<const __nv_bfloat16 *>(sm + Smem::q_raw);
    const __nv_bfloat16 *kr = reinterpret_cast<const __nv_bfloat16 *>(sm + Smem::k_raw);
    const float *G = reinterpret_cast<const float *>(sm + Smem::g_raw);
    const float *beta = reinterpret_cast<const float *>(sm + Smem::beta);
    float *akk = reinterpret_cast<float *>(sm + Smem::a_k);
    __half *aqk = reinterpret_cast<__half *>(sm + Smem::aqk);
    __half *nkt = reinterpret_cast<__half *>(sm + Smem::nkt);
    __half *qt = reinterpret_cast<__half *>(sm + Smem::qt);
    __half *kh = reinterpret_cast<__half *>(sm + Smem::kh);
    for (int p = tid; p < C * (C + 1) / 2; p += kThreads) {
        int r = (int)((sqrtf(8.f * p + 1.f) - 1.f) * 0.5f);
        while (r * (r + 1) / 2 > p) --r;
        while ((r + 1) * (r + 2) / 2 <= p) ++r;
        const int i = p - r * (r + 1) / 2;
        float sk = 0.f, sq = 0.f;
        for (int c = 0; c < KD; ++c) {
            const float kic = __bfloat162float(kr[i * KD + c]) * exp2f(G[r * KD + c] - G[i * KD + c]);
            sk += __bfloat162float(kr[r * KD + c]) * kic;
            sq += __bfloat162float(qr[r * KD + c]) * kic;
        }
        akk[r * LDA + i] = (i < r) ? beta[r] * sk : 0.f;
        aqk[r * LD64 + i] = __float2half_rn(sq);
        if (i < r) aqk[i * LD64 + r] = __float2half_rn(0.f);
    }
    for (int e = tid; e < C * KD; e += kThreads) {
        const int r = e >> 7, c = e & 127;
        const float gr = G[r * KD + c], gl = G[(C - 1) * KD + c];
        const float kv = __bfloat162float(kr[r * KD + c]);
        const float qv = __bfloat162float(qr[r * KD + c]);
        const float eg = exp2f(gr);
        nkt[r * LD128 + c] = __float2half_rn(-kv * eg);
        qt[r * LD128 + c] = __float2half_rn(qv * eg);
        kh[r * LD128 + c] = __float2half_rn(kv * exp2f(gl - gr));
    }
}

template <typename Tout>
__global__ void __launch_bounds__(kThreads, 1)
kda_prefill_tc_kernel(const PrefillArgs a, const __grid_constant__ TmaMaps maps)
{
    extern __shared__ __align__(128) unsigned char sm[];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g8 = lane >> 2, tig = lane & 3;
    const int64_t n = blockIdx.x / kVTiles;
    const int vt = blockIdx.x % kVTiles;
    const int h = blockIdx.y;
    const int H = a.num_heads;

    float *G = reinterpret_cast<float *>(sm + Smem::g_raw);
    const __nv_bfloat16 *qraw = reinterpret_cast<const __nv_bfloat16 *>(sm + Smem::q_raw);
    const __nv_bfloat16 *kraw = reinterpret_cast<const __nv_bfloat16 *>(sm + Smem::k_raw);
    const __nv_bfloat16 *vraw = reinterpret_cast<const __nv_bfloat16 *>(sm + Smem::v_raw);
    const float *braw = reinterpret_cast<const float *>(sm + Smem::b_raw);
    __half *ak = reinterpret_cast<__half *>(sm + Smem::a_k);
    __half *aq = reinterpret_cast<__half *>(sm + Smem::a_q);
    __half *bk = reinterpret_cast<__half *>(sm + Smem::b_k);
    __half *nkt = reinterpret_cast<__half *>(sm + Smem::nkt);
    __half *qt = reinterpret_cast<__half *>(sm + Smem::qt);
    __half *kh = reinterpret_cast<__half *>(sm + Smem::kh);
    __half *tmh = reinterpret_cast<__half *>(sm + Smem::tm);
    __half *aqk = reinterpret_cast<__half *>(sm + Smem::aqk);
    __half *ht = reinterpret_cast<__half *>(sm + Smem::ht);
    __half *xt = reinterpret_cast<__half *>(sm + Smem::xt);
    __half *dt = reinterpret_cast<__half *>(sm + Smem::dt);
    float *vs = reinterpret_cast<float *>(sm + Smem::vs);
    float *beta_s = reinterpret_cast<float *>(sm + Smem::beta);
    float *dec = reinterpret_cast<float *>(sm + Smem::dec);
    float *mref = reinterpret_cast<float *>(sm + Smem::mref);
    float *pm = reinterpret_cast<float *>(sm + Smem::pm);
    float *fm = reinterpret_cast<float *>(sm + Smem::fm);
    __half *rho = reinterpret_cast<__half *>(sm + Smem::rho);
    volatile int *flag = reinterpret_cast<volatile int *>(sm + Smem::flag);
    float *akk = reinterpret_cast<float *>(sm + Smem::a_k);       // aliases a_k after P3

    int64_t bos, eos;
    clamp_range(a.total_tokens, a.cu_seqlens[n], a.cu_seqlens[n + 1], bos, eos);

    // state-step roles: warp -> (16 value rows mt, quarter qw of chunk rows / key channels)
    const int mt = warp & 1, qw = warp >> 1;

    // the state tile h^T [v][c] for v in 16mt.., c in 32qw.. : 4 n8-tiles of fp32 accumulators
    float hreg[4][4];
    const int64_t state_base = (n * H + h) * (int64_t)(KD * VD) + vt * VT;
#pragma unroll
    for (int nt = 0; nt < 4; ++nt) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int v = 16 * mt + g8 + ((e >> 1) << 3);
            const int c = 32 * qw + 8 * nt + 2 * tig + (e & 1);
            hreg[nt][e] = a.init_state ? a.init_state[state_base + (int64_t)c * VD + v] : 0.f;
        }
    }
    // fp16 mirror of h^T for the MMAs of the first chunk
#pragma unroll
    for (int nt = 0; nt < 4; ++nt) {
        const int c = 32 * qw + 8 * nt + 2 * tig;
        const int v0 = 16 * mt + g8;
        *reinterpret_cast<uint32_t *>(ht + v0 * LD128 + c) = pack_h2(hreg[nt][0], hreg[nt][1]);
        *reinterpret_cast<uint32_t *>(ht + (v0 + 8) * LD128 + c) = pack_h2(hreg[nt][2], hreg[nt][3]);
    }

    const uint32_t mbar = smem_u32(sm + Smem::mbar);
    if (tid == 0) mbar_init(mbar, 1);
    __syncthreads();
    if (bos < eos) issue_chunk_loads(sm, a, maps, bos, (int)((eos - bos) < C ? (eos - bos) : C), h, vt, tid);

    Tout *out = static_cast<Tout *>(a.out);
    uint32_t load_parity = 0;
    bool failed = false;

    for (int64_t t0 = bos; t0 < eos; t0 += C) {
        const int len = (int)((eos - t0) < C ? (eos - t0) : C);
        cp_async_wait_all();
        if (!mbar_wait(mbar, load_parity)) {
            // the chunk's copies did not land within the wait bound: stop, and mark
            // this CTA's outputs as invalid (NaN) below instead of hanging
            failed = true;
        }
        load_parity ^= 1u;
        if (!failed && len < C) zero_tail_rows(sm, len, tid);
        if (__syncthreads_or(failed)) { failed = true; break; }
        if (tid == 0) *flag = 0;

        // ---------------- P1: in-chunk gate cumsum, exp2 space (two halves of 32 rows)
        {
            const int c = tid & 127, half = tid >> 7;
            float acc = 0.f;
#pragma unroll
            for (int r0 = 32 * half; r0 < 32 * half + 32; r0 += 8) {
                float x[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) x[u] = G[(r0 + u) * KD + c];
#pragma unroll
                for (int u = 0; u < 8; ++u) { acc += x[u] * kLog2e; G[(r0 + u) * KD + c] = acc; }
            }
        }
        __syncthreads();
        if (tid >= 128) {
            const int c = tid & 127;
            const float base = G[31 * KD + c];
#pragma unroll 8
            for (int r = 32; r < 64; ++r) G[r * KD + c] += base;
        }
        __syncthreads();
        // per-channel scalars
        if (tid < 128) {
            const int c = tid;
            const float gl = G[(C - 1) * KD + c];
            dec[c] = exp2f(gl);
            float m[4];
#pragma unroll
            for (int R = 0; R < 4; ++R) {
                m[R] = G[(16 * R + 8) * KD + c];
                mref[R * KD + c] = m[R];
                pm[R * KD + c] = exp2f(m[R]);
                fm[R * KD + c] = exp2f(gl - m[R]);
            }
            int p = 0;
#pragma unroll
            for (int R = 1; R < 4; ++R)
#pragma unroll
                for (int I = 0; I < R; ++I, ++p) rho[p * KD + c] = __float2half_rn(exp2f(m[R] - m[I]));
        } else if (tid < 128 + C) {
            beta_s[tid - 128] = braw[tid - 128];
        }
        for (int e = tid; e < C * VT; e += kThreads) {
            const int r = e >> 5, j = e & 31;
            vs[r * LDV + j] = __bfloat162float(vraw[r * VT + j]);
        }
        __syncthreads();

        // ---------------- P2: factors and fp16 operands, four channels per thread
        {
            bool bad = false;
#pragma unroll 2
            for (int e = tid; e < C * KD / 4; e += kThreads) {
                const int r = e >> 5, c = (e & 31) * 4, R = r >> 4;
                const float4 gv = *reinterpret_cast<const float4 *>(G + r * KD + c);
                const float4 mv = *reinterpret_cast<const float4 *>(mref + R * KD + c);
                const float4 pv = *reinterpret_cast<const float4 *>(pm + R * KD + c);
                const float4 fv = *reinterpret_cast<const float4 *>(fm + R * KD + c);
                const uint2 kb = *reinterpret_cast<const uint2 *>(kraw + r * KD + c);
                const uint2 qb = *reinterpret_cast<const uint2 *>(qraw + r * KD + c);
                const float g4[4] = {gv.x, gv.y, gv.z, gv.w}, m4[4] = {mv.x, mv.y, mv.z, mv.w};
                const float p4[4] = {pv.x, pv.y, pv.z, pv.w}, f4[4] = {fv.x, fv.y, fv.z, fv.w};
                const float2 k01 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&kb.x));
                const float2 k23 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&kb.y));
                const float2 q01 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&qb.x));
                const float2 q23 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&qb.y));
                const float k4[4] = {k01.x, k01.y, k23.x, k23.y}, q4[4] = {q01.x, q01.y, q23.x, q23.y};
                float ok[4], oq[4], ob[4], ot[4], oqt[4], okh[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const float x = g4[u] - m4[u];
                    const float em = exp2f(x), ep = exp2f(-x);
                    bad |= !(em <= kFactorMax && ep <= kFactorMax);
                    ok[u] = k4[u] * em;
                    oq[u] = q4[u] * em;
                    ob[u] = k4[u] * ep;
                    ot[u] = -ok[u] * p4[u];
                    oqt[u] = oq[u] * p4[u];
                    okh[u] = ob[u] * f4[u];
                }
                const int o = r * LD128 + c;
                *reinterpret_cast<uint2 *>(ak + o) = make_uint2(pack_h2(ok[0], ok[1]), pack_h2(ok[2], ok[3]));
                *reinterpret_cast<uint2 *>(aq + o) = make_uint2(pack_h2(oq[0], oq[1]), pack_h2(oq[2], oq[3]));
                *reinterpret_cast<uint2 *>(bk + o) = make_uint2(pack_h2(ob[0], ob[1]), pack_h2(ob[2], ob[3]));
                *reinterpret_cast<uint2 *>(nkt + o) = make_uint2(pack_h2(ot[0], ot[1]), pack_h2(ot[2], ot[3]));
                *reinterpret_cast<uint2 *>(qt + o) = make_uint2(pack_h2(oqt[0], oqt[1]), pack_h2(oqt[2], oqt[3]));
                *reinterpret_cast<uint2 *>(kh + o) = make_uint2(pack_h2(okh[0], okh[1]), pack_h2(okh[2], okh[3]));
            }
            if (__any_sync(0xffffffffu, bad) && lane == 0) *flag = 1;
        }
        __syncthreads();
        const bool exact_path = *flag != 0;

        // ---------------- P3: A_kk and A_qk (lower block triangle) on tensor cores
        if (!exact_path) {
            // warp -> (matrix, row block R, up to three 16-column blocks I <= R); the A
            // fragments of a row block are loaded once per k-step and reused.
            const int mat = warp >> 2, sub = warp & 3;
            const __half *A = mat == 0 ? ak : aq;
            // (R, I) of this warp's column blocks; sub 3 also takes row block 0
            const int nblk = sub == 2 ? 3 : 2 + (sub == 3);
            int Rb[3], Ib[3];
            if (sub == 0)      { Rb[0] = 3; Ib[0] = 0; Rb[1] = 3; Ib[1] = 1; Rb[2] = 3; Ib[2] = 1; }
            else if (sub == 1) { Rb[0] = 3; Ib[0] = 2; Rb[1] = 3; Ib[1] = 3; Rb[2] = 3; Ib[2] = 3; }
            else if (sub == 2) { Rb[0] = 2; Ib[0] = 0; Rb[1] = 2; Ib[1] = 1; Rb[2] = 2; Ib[2] = 2; }
            else               { Rb[0] = 1; Ib[0] = 0; Rb[1] = 1; Ib[1] = 1; Rb[2] = 0; Ib[2] = 0; }
            float acc[3][2][4];
#pragma unroll
            for (int b = 0; b < 3; ++b)
#pragma unroll
                for (int t = 0; t < 2; ++t) acc[b][t][0] = acc[b][t][1] = acc[b][t][2] = acc[b][t][3] = 0.f;
#pragma unroll
            for (int ks = 0; ks < KD / 16; ++ks) {
                uint32_t afr[2][4];
                ldsm_x4(smem_u32(A + a_off(lane, 16 * Rb[0], 16 * ks, LD128)),
                        afr[0][0], afr[0][1], afr[0][2], afr[0][3]);
                if (sub == 3)
                    ldsm_x4(smem_u32(A + a_off(lane, 0, 16 * ks, LD128)),
                            afr[1][0], afr[1][1], afr[1][2], afr[1][3]);
#pragma unroll
                for (int b = 0; b < 3; ++b) {
                    if (b < nblk) {
                        const int R = Rb[b], I = Ib[b];
                        uint32_t bf[4];
                        ldsm_x4(smem_u32(bk + bnk_off(lane, 16 * I, 16 * ks, LD128)),
                                bf[0], bf[1], bf[2], bf[3]);
                        if (I < R) {
                            const int pair = R * (R - 1) / 2 + I;
                            const __half *rp = rho + pair * KD + 16 * ks + 2 * tig;
                            const uint32_t s0 = *reinterpret_cast<const uint32_t *>(rp);
                            const uint32_t s1 = *reinterpret_cast<const uint32_t *>(rp + 8);
                            bf[0] = hmul2_u32(bf[0], s0); bf[1] = hmul2_u32(bf[1], s1);
                            bf[2] = hmul2_u32(bf[2], s0); bf[3] = hmul2_u32(bf[3], s1);
                        }
                        const bool alt = (sub == 3 && b == 2);   // row block 0 of warp sub 3
                        const uint32_t af[4] = {alt ? afr[1][0] : afr[0][0], alt ? afr[1][1] : afr[0][1],
                                                alt ? afr[1][2] : afr[0][2], alt ? afr[1][3] : afr[0][3]};
                        mma16816(acc[b][0], af, bf[0], bf[1]);
                        mma16816(acc[b][1], af, bf[2], bf[3]);
                    }
                }
            }
            __syncthreads();   // every read of a_k / a_q / b_k is done; a_k becomes A_kk (fp32)
#pragma unroll
            for (int b = 0; b < 3; ++b) {
                if (b < nblk) {
                    const int R = Rb[b], I = Ib[b];
#pragma unroll
                    for (int t = 0; t < 2; ++t) {
#pragma unroll
                        for (int hh = 0; hh < 2; ++hh) {
                            const int r = 16 * R + g8 + 8 * hh;
                            const int i = 16 * I + 8 * t + 2 * tig;
                            const float v0 = acc[b][t][2 * hh], v1 = acc[b][t][2 * hh + 1];
                            if (mat == 0) {
                                akk[r * LDA + i] = (i < r) ? beta_s[r] * v0 : 0.f;
                                akk[r * LDA + i + 1] = (i + 1 < r) ? beta_s[r] * v1 : 0.f;
                            } else {
                                *reinterpret_cast<uint32_t *>(aqk + r * LD64 + i) =
                                    pack_h2(i <= r ? v0 : 0.f, i + 1 <= r ? v1 : 0.f);
                            }
                        }
                    }
                }
            }
        } else {
            exact_intra_chunk(sm, tid);
        }
        __syncthreads();

        // raw buffers are free: fetch the next chunk while the solve and state step run
        if (t0 + C < eos) {
            const int64_t t1 = t0 + C;
            issue_chunk_loads(sm, a, maps, t1, (int)((eos - t1) < C ? (eos - t1) : C), h, vt, tid);
        }

        // ---------------- P4: T = (I + A_kk)^-1 in 16x16 blocks
        // Diagonal blocks: fp32 forward substitution, one warp per block (lane j owns
        // column j).  Below-diagonal blocks, by distance from the diagonal:
        //     T_RI = -T_RR sum_{J=I}^{R-1} A_RJ T_JI
        // on tensor cores, evaluated transposed (X^T = sum T_JI^T A_RJ^T, then
        // T_RI^T = -X^T T_RR^T) so X^T passes from accumulator to operand in registers.
        {
            __half *akh = reinterpret_cast<__half *>(sm + Smem::xt);   // A_kk fp16 [64][LD64]
            for (int e = tid; e < 6 * 128; e += kThreads) {            // 6 blocks x 16 rows x 8 pairs
                const int blk = e >> 7, rem = e & 127, rr = rem >> 3, pp = (rem & 7) * 2;
                const int R = blk == 0 ? 1 : blk < 3 ? 2 : 3;
                const int J = blk - (R == 1 ? 0 : R == 2 ? 1 : 3);
                const int r = 16 * R + rr, m = 16 * J + pp;
                *reinterpret_cast<uint32_t *>(akh + r * LD64 + m) =
                    pack_h2(akk[r * LDA + m], akk[r * LDA + m + 1]);
            }
            if (warp < 4) {
                const int R = warp, j = lane & 15;
                float col[16];
#pragma unroll
                for (int m = 0; m < 16; ++m) col[m] = (m == j) ? 1.f : 0.f;
                const float *Ab = akk + (16 * R) * LDA + 16 * R;
#pragma unroll
                for (int r = 1; r < 16; ++r) {
                    float s4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                    for (int m = 0; m < r; ++m) s4[m & 3] += Ab[r * LDA + m] * col[m];
                    if (j < r) col[r] = -((s4[0] + s4[1]) + (s4[2] + s4[3]));
                }
                if (lane < 16) {
#pragma unroll
                    for (int r = 0; r < 16; ++r) tmh[(16 * R + r) * LD64 + 16 * R + j] = __float2half_rn(col[r]);
                }
            }
            __syncthreads();
            for (int lvl = 1; lvl < 4; ++lvl) {
                if (warp < 4 - lvl) {
                    const int I = warp, R = warp + lvl;
                    float xa[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
                    for (int J = I; J < R; ++J) {
                        uint32_t af[4], bf[4];
                        // A = T_JI^T (rows i, cols m) from T_JI stored [m][i]
                        ldsm_x4_t(smem_u32(tmh + (16 * J + (lane & 7) + ((lane >> 4) << 3)) * LD64 +
                                           16 * I + (((lane >> 3) & 1) << 3)),
                                  af[0], af[1], af[2], af[3]);
                        // B = A_RJ^T as [k=m][n=r] from A_RJ stored [r][m]
                        ldsm_x4(smem_u32(akh + bnk_off(lane, 16 * R, 16 * J, LD64)), bf[0], bf[1], bf[2], bf[3]);
                        mma16816(xa[0], af, bf[0], bf[1]);
                        mma16816(xa[1], af, bf[2], bf[3]);
                    }
                    const uint32_t xf[4] = {pack_h2(-xa[0][0], -xa[0][1]), pack_h2(-xa[0][2], -xa[0][3]),
                                            pack_h2(-xa[1][0], -xa[1][1]), pack_h2(-xa[1][2], -xa[1][3])};
                    uint32_t tb[4];
                    ldsm_x4(smem_u32(tmh + bnk_off(lane, 16 * R, 16 * R, LD64)), tb[0], tb[1], tb[2], tb[3]);
                    float ta[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
                    mma16816(ta[0], xf, tb[0], tb[1]);
                    mma16816(ta[1], xf, tb[2], tb[3]);
#pragma unroll
                    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int i = 16 * I + g8 + ((e >> 1) << 3);
                            const int r = 16 * R + 8 * nt + 2 * tig + (e & 1);
                            tmh[r * LD64 + i] = __float2half_rn(ta[nt][e]);
                        }
                }
                __syncthreads();
            }
        }

        // ---------------- S1: X^T = V^T - h^T K~^T,  O1^T = h^T Q~^T   (rows v of mt, cols r of qw)
        float xacc[2][4], oacc[2][4];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int v = 16 * mt + g8 + ((e >> 1) << 3);
                const int r = 16 * qw + 8 * nt + 2 * tig + (e & 1);
                xacc[nt][e] = vs[r * LDV + v];
                oacc[nt][e] = 0.f;
            }
        }
#pragma unroll
        for (int ks = 0; ks < KD / 16; ++ks) {
            uint32_t af[4], bx[4], bq[4];
            ldsm_x4(smem_u32(ht + a_off(lane, 16 * mt, 16 * ks, LD128)), af[0], af[1], af[2], af[3]);
            ldsm_x4(smem_u32(nkt + bnk_off(lane, 16 * qw, 16 * ks, LD128)), bx[0], bx[1], bx[2], bx[3]);
            ldsm_x4(smem_u32(qt + bnk_off(lane, 16 * qw, 16 * ks, LD128)), bq[0], bq[1], bq[2], bq[3]);
            mma16816(xacc[0], af, bx[0], bx[1]);
            mma16816(xacc[1], af, bx[2], bx[3]);
            mma16816(oacc[0], af, bq[0], bq[1]);
            mma16816(oacc[1], af, bq[2], bq[3]);
        }
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
            const int r = 16 * qw + 8 * nt + 2 * tig;
            const int v0 = 16 * mt + g8;
            const float b0 = beta_s[r], b1 = beta_s[r + 1];
            *reinterpret_cast<uint32_t *>(xt + v0 * LD64 + r) = pack_h2(b0 * xacc[nt][0], b1 * xacc[nt][1]);
            *reinterpret_cast<uint32_t *>(xt + (v0 + 8) * LD64 + r) =
                pack_h2(b0 * xacc[nt][2], b1 * xacc[nt][3]);
        }
        __syncthreads();

        // ---------------- S2: D^T = (beta X)^T T^T  (T lower triangular: k-steps <= qw)
        float dacc[2][4];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) dacc[nt][0] = dacc[nt][1] = dacc[nt][2] = dacc[nt][3] = 0.f;
        for (int ks = 0; ks <= qw; ++ks) {
            uint32_t af[4], bt[4];
            ldsm_x4(smem_u32(xt + a_off(lane, 16 * mt, 16 * ks, LD64)), af[0], af[1], af[2], af[3]);
            ldsm_x4(smem_u32(tmh + bnk_off(lane, 16 * qw, 16 * ks, LD64)), bt[0], bt[1], bt[2], bt[3]);
            mma16816(dacc[0], af, bt[0], bt[1]);
            mma16816(dacc[1], af, bt[2], bt[3]);
        }
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
            const int r = 16 * qw + 8 * nt + 2 * tig;
            const int v0 = 16 * mt + g8;
            *reinterpret_cast<uint32_t *>(dt + v0 * LD64 + r) = pack_h2(dacc[nt][0], dacc[nt][1]);
            *reinterpret_cast<uint32_t *>(dt + (v0 + 8) * LD64 + r) = pack_h2(dacc[nt][2], dacc[nt][3]);
        }
        __syncthreads();

        // ---------------- S3: O^T += D^T A_qk^T ; h^T <- h^T Diag(2^G_last) + D^T K^
#pragma unroll
        for (int nt = 0; nt < 4; ++nt) {
            const int c = 32 * qw + 8 * nt + 2 * tig;
            const float d0 = dec[c], d1 = dec[c + 1];
            hreg[nt][0] *= d0; hreg[nt][1] *= d1; hreg[nt][2] *= d0; hreg[nt][3] *= d1;
        }
#pragma unroll
        for (int ks = 0; ks < C / 16; ++ks) {
            uint32_t af[4], bk0[4], bk1[4];
            ldsm_x4(smem_u32(dt + a_off(lane, 16 * mt, 16 * ks, LD64)), af[0], af[1], af[2], af[3]);
            if (ks <= qw) {
                uint32_t ba[4];
                ldsm_x4(smem_u32(aqk + bnk_off(lane, 16 * qw, 16 * ks, LD64)), ba[0], ba[1], ba[2], ba[3]);
                mma16816(oacc[0], af, ba[0], ba[1]);
                mma16816(oacc[1], af, ba[2], ba[3]);
            }
            ldsm_x4_t(smem_u32(kh + bkn_off(lane, 16 * ks, 32 * qw, LD128)), bk0[0], bk0[1], bk0[2], bk0[3]);
            ldsm_x4_t(smem_u32(kh + bkn_off(lane, 16 * ks, 32 * qw + 16, LD128)), bk1[0], bk1[1], bk1[2], bk1[3]);
            mma16816(hreg[0], af, bk0[0], bk0[1]);
            mma16816(hreg[1], af, bk0[2], bk0[3]);
            mma16816(hreg[2], af, bk1[0], bk1[1]);
            mma16816(hreg[3], af, bk1[2], bk1[3]);
        }
        // output rows of this chunk
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int v = 16 * mt + g8 + ((e >> 1) << 3);
                const int r = 16 * qw + 8 * nt + 2 * tig + (e & 1);
                if (r < len)
                    out[((t0 + r) * H + h) * VD + vt * VT + v] = from_f32<Tout>(a.scale * oacc[nt][e]);
            }
        }
        // fp16 mirror of the new state for the next chunk
#pragma unroll
        for (int nt = 0; nt < 4; ++nt) {
            const int c = 32 * qw + 8 * nt + 2 * tig;
            const int v0 = 16 * mt + g8;
            *reinterpret_cast<uint32_t *>(ht + v0 * LD128 + c) = pack_h2(hreg[nt][0], hreg[nt][1]);
            *reinterpret_cast<uint32_t *>(ht + (v0 + 8) * LD128 + c) = pack_h2(hreg[nt][2], hreg[nt][3]);
        }
        // the next iteration's first barrier orders these writes before their reads
    }

    if (failed) {
        // error marker: NaN state; the copies still in flight get one more bounded wait
        mbar_wait(mbar, load_parity);
#pragma unroll
        for (int nt = 0; nt < 4; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) hreg[nt][e] = __int_as_float(0x7fc00000);
    }
    if (a.final_state) {
#pragma unroll
        for (int nt = 0; nt < 4; ++nt) {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int v = 16 * mt + g8 + ((e >> 1) << 3);
                const int c = 32 * qw + 8 * nt + 2 * tig + (e & 1);
                a.final_state[state_base + (int64_t)c * VD + v] = hreg[nt][e];
            }
        }
    }
}

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) != cudaSuccess || q != cudaDriverEntryPointSuccess)
            p = nullptr;
        return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }();
    return fn;
}

// [T, H, inner] row-major tensor, box (box_inner x 1 x 64)
bool encode_map(CUtensorMap *m, const void *base, CUtensorMapDataType type, int esize, int64_t T,
                int H, int inner, int box_inner)
{
    auto enc = tensor_map_encoder();
    if (!enc) return false;
    const cuuint64_t dims[3] = {(cuuint64_t)inner, (cuuint64_t)H, (cuuint64_t)(T > 0 ? T : 1)};
    const cuuint64_t strides[2] = {(cuuint64_t)inner * esize, (cuuint64_t)inner * esize * H};
    const cuuint32_t box[3] = {(cuuint32_t)box_inner, 1u, (cuuint32_t)C};
    const cuuint32_t estr[3] = {1u, 1u, 1u};
    return enc(m, type, 3, const_cast<void *>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <typename Tout>
cudaError_t launch_tc_t(const PrefillArgs &a, cudaStream_t stream)
{
    TmaMaps maps;
    memset(&maps, 0, sizeof(maps));
    const int H = a.num_heads;
    if (a.total_tokens > 0) {   // with no tokens no tile is ever loaded
        const int64_t T = a.total_tokens;
        if (!encode_map(&maps.q, a.q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, T, H, KD, KD) ||
            !encode_map(&maps.k, a.k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, T, H, KD, KD) ||
            !encode_map(&maps.g, a.g, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, T, H, KD, KD) ||
            !encode_map(&maps.v, a.v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, T, H, VD, VT))
            return cudaErrorInvalidValue;
    }
    const int smem = Smem::total;
    cudaError_t e = cudaFuncSetAttribute(kda_prefill_tc_kernel<Tout>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    dim3 grid((unsigned)((int64_t)a.num_seqs * kVTiles), (unsigned)a.num_heads);
    kda_prefill_tc_kernel<Tout><<<grid, kThreads, smem, stream>>>(a, maps);
    return cudaGetLastError();
}

}  // namespace

bool prefill_tc_supported(const PrefillArgs &a)
{
    return a.dtype == kDtypeBF16 && a.head_dim_k == KD && a.head_dim_v == VD;
}

cudaError_t launch_prefill_tc(const PrefillArgs &a, cudaStream_t stream)
{
    if (a.num_seqs == 0) return cudaSuccess;
    return a.out_dtype == kDtypeBF16 ? launch_tc_t<__nv_bfloat16>(a, stream)
                                     : launch_tc_t<float>(a, stream);
}

}  // namespace kda
