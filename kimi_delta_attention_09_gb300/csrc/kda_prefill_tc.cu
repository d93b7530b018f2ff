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
// Mapping: one CTA (16 warps) per (sequence, head, 32-column tile of V); it walks its
// sequence chunk by chunk.  The raw inputs of a chunk arrive as TMA tiles (issued one
// chunk ahead by a dedicated warp).  Per chunk, the warps build the intra-chunk
// operands (gate cumsum, factors, A_kk / A_qk with mma.sync, blocked solve), then run
// the state step: the state tile h^T (fp32, 128 key channels x 32 values) lives in
// tensor memory, and the two big contractions of the step are tcgen05 MMAs issued by
// one thread -- [-K~; Q~] h (X and the inter-chunk part of o) and K^^T D accumulated
// into the state, with A_qk D accumulated into o.  The small D = T (beta X) product
// stays on mma.sync.  tcgen05 operands use the 128-byte-swizzled K-major layout.
#include <cstring>

#include <cuda.h>
#include <cuda_fp16.h>
#include <cudaTypedefs.h>

#include "kda_internal.cuh"

namespace kda {
namespace {

constexpr int kThreads = 512;   // 16 warps
constexpr int C = kChunk;        // 64 rows per chunk
constexpr int KD = 128;          // key dim
constexpr int VD = 128;          // value dim
constexpr int VT = 32;           // value columns per CTA
constexpr int kVTiles = VD / VT;
constexpr int LD128 = KD + 8;    // f16 row stride (halves) of 128-column tiles: 272 B
constexpr int LD64 = C + 8;      // f16 row stride of 64-column tiles: 144 B
constexpr float kFactorMax = 256.f;   // fp16 factor bound (2^8) of the fast path

// Shared memory map (byte offsets).  SW128 tiles: 128-byte-swizzled K-major tcgen05
// operands (1024-byte aligned); the others are padded row-major mma.sync operands.
struct Smem {
    static constexpr int q_raw = 0;                          // bf16 [64][128]
    static constexpr int k_raw = q_raw + C * KD * 2;         // bf16 [64][128]
    static constexpr int g_raw = k_raw + C * KD * 2;         // f32  [64][128] raw natural-log gate
    static constexpr int v_raw = g_raw + C * KD * 4;         // bf16 [64][32]
    static constexpr int b_raw = v_raw + C * VT * 2;         // f32  [64][4] beta of heads 4*(h/4)..
    static constexpr int a_k = b_raw + C * 4 * 4;            // f16 k 2^(G - m_R)  [64][LD128]
    static constexpr int a_q = a_k + C * LD128 * 2;          // f16 q 2^(G - m_R)  [64][LD128]
    static constexpr int b_k = a_q + C * LD128 * 2;          // f16 k 2^(m_R - G)  [64][LD128]
    static constexpr int tm = b_k + C * LD128 * 2;           // f16  T  [64][LD64]
    static constexpr int a1 = (tm + C * LD64 * 2 + 1023) / 1024 * 1024;   // SW128 [-K~; Q~] 128 x 128
    static constexpr int kht = a1 + 2 * C * KD * 2;          // SW128 K^^T: 128 (channel) x 64 (row)
    static constexpr int akh = kht + KD * C * 2;             // SW128 A_kk fp16 64 x 64
    static constexpr int aqk = akh + C * C * 2;              // SW128 A_qk fp16 64 x 64 (follows akh:
                                                             // [akh; aqk] is the 128-row A of o += A_qk D)
    static constexpr int ht = aqk + C * C * 2;               // SW128 h^T fp16 32 (value) x 128 (channel)
    static constexpr int dt = ht + VT * KD * 2;              // SW128 D^T fp16 32 (value) x 64 (row)
    static constexpr int xt = dt + VT * C * 2;               // f16 (beta X)^T [32][LD64]
    static constexpr int tot8 = dt;                          // f32 [8][128] group sums (P1/P2 only)
    static constexpr int first8 = xt;                        // f32 [8][128] group firsts (P1/P2 only)
    static constexpr int vs = xt + VT * LD64 * 2;            // bf16 V [64][32]
    static constexpr int beta = vs + C * VT * 2;             // f32  [64]
    static constexpr int dec = beta + C * 4;                 // f32  [128] 2^G_last
    static constexpr int rho = dec + KD * 4;                 // f16  [6][128] 2^(m_R - m_I), I < R
    static constexpr int flag = rho + 6 * KD * 2;            // int
    static constexpr int mbar = flag + 8;                    // u64 mbarrier of the chunk loads
    static constexpr int mbar_mma = mbar + 8;                // u64 mbarrier of the tcgen05 MMAs
    static constexpr int tmem = mbar_mma + 8;                // u32 tensor-memory base
    static constexpr int total = tmem + 8;
};
static_assert(Smem::total <= 232448, "shared memory budget");
static_assert(Smem::a1 % 1024 == 0 && Smem::kht % 1024 == 0 && Smem::akh % 1024 == 0 &&
              Smem::aqk % 1024 == 0 && Smem::ht % 1024 == 0 && Smem::dt % 1024 == 0,
              "SW128 tiles need 1024-byte alignment");
static_assert(Smem::first8 + 8 * KD * 4 <= Smem::vs + C * VT * 2 && Smem::tot8 + 8 * KD * 4 <= Smem::xt,
              "gate group sums fit in the D^T / (beta X)^T space");

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

__device__ __forceinline__ void ldsm_x2(uint32_t addr, uint32_t &r0, uint32_t &r1)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0, %1}, [%2];\n"
                 : "=r"(r0), "=r"(r1) : "r"(addr));
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

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, int x, int y,
                                            uint32_t mbar)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
        "[%0], [%1, {%2, %3}], [%4];\n"
        :: "r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(mbar)
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

// 1/x for x in [2^-8, 2^8] on the FMA pipe: exponent-negating seed, then three
// Newton-Raphson steps y <- y (2 - x y) (relative error ~1e-7, below fp16 rounding).
__device__ __forceinline__ float recip_nr(float x)
{
    float y = __int_as_float(0x7EF311C3 - __float_as_int(x));
    y = y * (2.f - x * y);
    y = y * (2.f - x * y);
    y = y * (2.f - x * y);
    return y;
}

__device__ __forceinline__ void named_bar_sync(int id, int count)
{
    asm volatile("bar.sync %0, %1;\n" :: "r"(id), "r"(count) : "memory");
}
__device__ __forceinline__ void named_bar_arrive(int id, int count)
{
    asm volatile("bar.arrive %0, %1;\n" :: "r"(id), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem()
{
    asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
}
__device__ __forceinline__ void cp_async_wait_all()
{
    asm volatile("cp.async.wait_group 0;\n" ::: "memory");
}

// ------------------------------------------------------------------ tcgen05 helpers
// Element (row, k) of a 128-byte-swizzled K-major tile of `rows` rows, in halves:
// 64-element column blocks stacked after all rows; within a block, row r is 128 B
// and its 16-byte chunk j sits at chunk j ^ (r % 8).
__device__ __forceinline__ int sw128(int row, int k, int rows)
{
    return ((k >> 6) * rows + row) * 64 + ((((k >> 3) & 7) ^ (row & 7)) << 3) + (k & 7);
}

// Shared-memory matrix descriptor of a SW128 K-major operand starting at `saddr`:
// 8-row groups 1024 B apart, descriptor version 1, layout SWIZZLE_128B.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr)
{
    return (uint64_t)((saddr >> 4) & 0x3FFF) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
           ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

// descriptor of k16-step ks of a SW128 tile with `rows` rows at `base`
__device__ __forceinline__ uint64_t sw128_kdesc(uint32_t base, int ks, int rows)
{
    return sw128_desc(base + (uint32_t)((ks >> 2) * rows * 128 + (ks & 3) * 32));
}

// instruction descriptor: fp16 A and B (K-major), fp32 D, M = 128, N = 32
constexpr uint32_t kIdescM128N32 = (1u << 4) | ((32u >> 3) << 17) | ((128u >> 4) << 24);

__device__ __forceinline__ void umma_f16(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc,
                                         uint32_t idesc, uint32_t accumulate)
{
    asm volatile("{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\n"
                 "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n"
                 :: "r"(tmem_d), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate));
}

__device__ __forceinline__ void umma_commit(uint32_t mbar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n"
                 :: "r"(mbar) : "memory");
}

__device__ __forceinline__ void tc_fence_before()
{
    asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after()
{
    asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory");
}

// 32 lanes x 16 columns of fp32 from / to tensor memory
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16])
{
    uint32_t r[16];
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x16.b32 "
                 "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];\n"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
                   "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]),
                   "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
                 : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory");
#pragma unroll
    for (int j = 0; j < 16; ++j) v[j] = __uint_as_float(r[j]);
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const float (&v)[16])
{
    asm volatile("tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
                 "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};\n"
                 :: "r"(taddr), "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])),
                    "r"(__float_as_uint(v[2])), "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])),
                    "r"(__float_as_uint(v[5])), "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])),
                    "r"(__float_as_uint(v[8])), "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])),
                    "r"(__float_as_uint(v[11])), "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])),
                    "r"(__float_as_uint(v[14])), "r"(__float_as_uint(v[15]))
                 : "memory");
    asm volatile("tcgen05.wait::st.sync.aligned;\n" ::: "memory");
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

// Tensor maps of q, k, g (box 128 channels x 1 head x 64 tokens) and v (box 32
// columns x 1 head x 64 tokens), built on the host for each call.
struct TmaMaps {
    CUtensorMap q, k, g, v, beta;   // beta: [T, H] fp32, box 4 heads x 64 tokens (H % 4 == 0)
    int beta_tma;                   // 0: beta comes by 4-byte cp.async instead
};

// ------------------------------------------------------------------ loads
// Tokens [t0, t0+64) of q, k, g, of this CTA's 32 v columns and of beta arrive as
// TMA tiles that complete on the chunk mbarrier (rows past the end of the tensor are
// zero-filled by the TMA unit; rows past the end of the SEQUENCE are zeroed after
// arrival, see zero_tail_rows).  When H is not a multiple of 4, beta (strided by H)
// comes by 4-byte cp.async instead.  Called by ONE warp after a barrier that ends
// every read of the raw buffers.
__device__ __forceinline__ void issue_chunk_loads(unsigned char *sm, const PrefillArgs &a,
                                                  const TmaMaps &maps, int64_t t0, int len,
                                                  int h, int vt, int lane)
{
    float *braw = reinterpret_cast<float *>(sm + Smem::b_raw);
    if (!maps.beta_tma) {
        for (int r = lane; r < C; r += 32) {
            const int valid = r < len;
            const int64_t row = t0 + (valid ? r : 0);
            cp_async4(smem_u32(braw + r * 4), a.beta + row * a.num_heads + h, valid ? 4 : 0);
        }
    }
    cp_async_commit();
    if (lane == 0) {
        const uint32_t mbar = smem_u32(sm + Smem::mbar);
        fence_proxy_async_smem();   // earlier generic reads of the raw buffers come first
        const uint32_t bytes = C * (2 * KD * 2 + KD * 4 + VT * 2) + (maps.beta_tma ? C * 16 : 0);
        mbar_arrive_expect_tx(mbar, bytes);
        const int z = (int)t0;
        tma_load_3d(smem_u32(sm + Smem::q_raw), &maps.q, 0, h, z, mbar);
        tma_load_3d(smem_u32(sm + Smem::k_raw), &maps.k, 0, h, z, mbar);
        tma_load_3d(smem_u32(sm + Smem::g_raw), &maps.g, 0, h, z, mbar);
        tma_load_3d(smem_u32(sm + Smem::v_raw), &maps.v, vt * VT, h, z, mbar);
        if (maps.beta_tma) tma_load_2d(smem_u32(braw), &maps.beta, h & ~3, z, mbar);
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

// scale * v[0..16) to 16 contiguous outputs (16-byte stores)
__device__ __forceinline__ void store_row16(float *dst, const float (&v)[16], float scale)
{
#pragma unroll
    for (int j = 0; j < 4; ++j)
        reinterpret_cast<float4 *>(dst)[j] =
            make_float4(scale * v[4 * j], scale * v[4 * j + 1], scale * v[4 * j + 2], scale * v[4 * j + 3]);
}
__device__ __forceinline__ void store_row16(__nv_bfloat16 *dst, const float (&v)[16], float scale)
{
#pragma unroll
    for (int j = 0; j < 2; ++j) {
        uint4 w;
        __nv_bfloat162 *p = reinterpret_cast<__nv_bfloat162 *>(&w);
#pragma unroll
        for (int u = 0; u < 4; ++u)
            p[u] = __floats2bfloat162_rn(scale * v[8 * j + 2 * u], scale * v[8 * j + 2 * u + 1]);
        reinterpret_cast<uint4 *>(dst)[j] = w;
    }
}

// Exact-exponential intra-chunk matrices for chunks outside the fp16 factor range.
// Recomputes the exp2-space cumsum G in place in g_raw, then writes A_kk and A_qk
// (fp16) with one exponential per pair and channel, and the state-step operands
// -K~, Q~ and K^^T with one exponential per element.
__device__ void exact_intra_chunk(unsigned char *sm, int tid)
{
    const __nv_bfloat16 *qr = reinterpret_cast<const __nv_bfloat16 *>(sm + Smem::q_raw);
    const __nv_bfloat16 *kr = reinterpret_cast<const __nv_bfloat16 *>(sm + Smem::k_raw);
    float *G = reinterpret_cast<float *>(sm + Smem::g_raw);
    const float *beta = reinterpret_cast<const float *>(sm + Smem::beta);
    __half *akh = reinterpret_cast<__half *>(sm + Smem::akh);
    __half *aqk = reinterpret_cast<__half *>(sm + Smem::aqk);
    __half *a1 = reinterpret_cast<__half *>(sm + Smem::a1);
    __half *kht = reinterpret_cast<__half *>(sm + Smem::kht);
    if (tid < KD) {
        float acc = 0.f;
        for (int r = 0; r < C; ++r) { acc += G[r * KD + tid] * kLog2e; G[r * KD + tid] = acc; }
    }
    __syncthreads();
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
        akh[sw128(r, i, C)] = __float2half_rn((i < r) ? beta[r] * sk : 0.f);
        aqk[sw128(r, i, C)] = __float2half_rn(sq);
        if (i < r) {
            akh[sw128(i, r, C)] = __float2half_rn(0.f);
            aqk[sw128(i, r, C)] = __float2half_rn(0.f);
        }
    }
    for (int e = tid; e < C * KD; e += kThreads) {
        const int r = e >> 7, c = e & 127;
        const float gr = G[r * KD + c], gl = G[(C - 1) * KD + c];
        const float kv = __bfloat162float(kr[r * KD + c]);
        const float qv = __bfloat162float(qr[r * KD + c]);
        const float eg = exp2f(gr);
        a1[sw128(r, c, 2 * C)] = __float2half_rn(-kv * eg);
        a1[sw128(C + r, c, 2 * C)] = __float2half_rn(qv * eg);
        kht[sw128(c, r, KD)] = __float2half_rn(kv * exp2f(gl - gr));
    }
}

// T_RR = (I + A_RR)^-1 of one 16x16 diagonal block (fp32 forward substitution on the
// fp16 A_kk, lane j owns column j), written to T (fp16) with its zeros and unit diagonal.
__device__ __forceinline__ void invert_diag_block(const __half *akh, __half *tmh, int R, int lane)
{
    const int j = lane & 15;
    float col[16];
#pragma unroll
    for (int m = 0; m < 16; ++m) col[m] = (m == j) ? 1.f : 0.f;
#pragma unroll
    for (int r = 1; r < 16; ++r) {
        float s4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int m = 0; m < r; ++m)
            s4[m & 3] += __half2float(akh[sw128(16 * R + r, 16 * R + m, C)]) * col[m];
        if (j < r) col[r] = -((s4[0] + s4[1]) + (s4[2] + s4[3]));
    }
    if (lane < 16) {
#pragma unroll
        for (int r = 0; r < 16; ++r) tmh[(16 * R + r) * LD64 + 16 * R + j] = __float2half_rn(col[r]);
    }
}

template <typename Tout>
__global__ void __launch_bounds__(kThreads, 1)
kda_prefill_tc_kernel(const PrefillArgs a, const __grid_constant__ TmaMaps maps)
{
    extern __shared__ __align__(1024) unsigned char sm[];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g8 = lane >> 2, tig = lane & 3;
    const int64_t n = blockIdx.x / kVTiles;
    const int vt = blockIdx.x % kVTiles;
    const int h = blockIdx.y;
    const int H = a.num_heads;

    const float *graw = reinterpret_cast<const float *>(sm + Smem::g_raw);
    const __nv_bfloat16 *qraw = reinterpret_cast<const __nv_bfloat16 *>(sm + Smem::q_raw);
    const __nv_bfloat16 *kraw = reinterpret_cast<const __nv_bfloat16 *>(sm + Smem::k_raw);
    const float *braw = reinterpret_cast<const float *>(sm + Smem::b_raw);
    __half *ak = reinterpret_cast<__half *>(sm + Smem::a_k);
    __half *aq = reinterpret_cast<__half *>(sm + Smem::a_q);
    __half *bk = reinterpret_cast<__half *>(sm + Smem::b_k);
    __half *tmh = reinterpret_cast<__half *>(sm + Smem::tm);
    __half *a1 = reinterpret_cast<__half *>(sm + Smem::a1);
    __half *kht = reinterpret_cast<__half *>(sm + Smem::kht);
    __half *akh = reinterpret_cast<__half *>(sm + Smem::akh);
    __half *aqk = reinterpret_cast<__half *>(sm + Smem::aqk);
    __half *ht = reinterpret_cast<__half *>(sm + Smem::ht);
    __half *dt = reinterpret_cast<__half *>(sm + Smem::dt);
    __half *xt = reinterpret_cast<__half *>(sm + Smem::xt);
    __nv_bfloat16 *vs = reinterpret_cast<__nv_bfloat16 *>(sm + Smem::vs);
    float *beta_s = reinterpret_cast<float *>(sm + Smem::beta);
    float *dec = reinterpret_cast<float *>(sm + Smem::dec);
    __half *rho = reinterpret_cast<__half *>(sm + Smem::rho);
    float *tot8 = reinterpret_cast<float *>(sm + Smem::tot8);
    float *first8 = reinterpret_cast<float *>(sm + Smem::first8);
    volatile int *flag = reinterpret_cast<volatile int *>(sm + Smem::flag);

    int64_t bos, eos;
    clamp_range(a.total_tokens, a.cu_seqlens[n], a.cu_seqlens[n + 1], bos, eos);
    const float *init;
    float *fin;
    prefill_state_ptrs(a, n, h, init, fin);

    // ---- tensor memory (64 columns: [0, 32) the step accumulator D1, [32, 64) the state
    //      h^T with lane = key channel, column = value) and the two mbarriers
    const uint32_t mbar = smem_u32(sm + Smem::mbar);
    const uint32_t mbar_mma = smem_u32(sm + Smem::mbar_mma);
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n"
                     :: "r"(smem_u32(sm + Smem::tmem)), "r"(64) : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n" ::: "memory");
    }
    if (tid == 0) {
        mbar_init(mbar, 1);
        mbar_init(mbar_mma, 1);
    }
    // A_qk blocks above the diagonal are never written by the fast path; zero them once
    for (int e = tid; e < C * C; e += kThreads) {
        const int r = e >> 6, i = e & 63;
        if ((i >> 4) > (r >> 4)) aqk[sw128(r, i, C)] = __float2half_rn(0.f);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(sm + Smem::tmem);
    const uint32_t tD1 = tmem, tH = tmem + 32;

    // TMEM epilogue roles (warp w reaches lanes 32 (w % 4) .. +31):
    //   state warps 8..15: key channels sc = 32 (w % 4) + lane, value columns [16 hc, 16 hc + 16)
    //   X rows (lanes 0..63): warps 0, 1 (columns 0..15) and 4, 5 (columns 16..31)
    //   o rows (lanes 64..127): warps 2, 3 (columns 0..15) and 6, 7 (columns 16..31)
    const bool state_warp = warp >= 8;
    const int sc = 32 * (warp & 3) + lane;                       // key channel of a state warp
    const int hc = (warp >> 2) & 1;                              // its half of the value columns
    const uint32_t lane_off = (uint32_t)(32 * (warp & 3)) << 16;  // TMEM lane quadrant
    if (state_warp) {   // initial state -> tensor memory and its fp16 mirror
        float hv[16];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float4 x = init ? *reinterpret_cast<const float4 *>(init + (int64_t)sc * VD + vt * VT + 16 * hc + 4 * j)
                                  : make_float4(0.f, 0.f, 0.f, 0.f);
            hv[4 * j] = x.x; hv[4 * j + 1] = x.y; hv[4 * j + 2] = x.z; hv[4 * j + 3] = x.w;
        }
        tmem_st16(tH + lane_off + 16 * hc, hv);
#pragma unroll
        for (int v = 0; v < 16; ++v) ht[sw128(16 * hc + v, sc, VT)] = __float2half_rn(hv[v]);
        fence_proxy_async_smem();
        tc_fence_before();
    }

    constexpr int kLoadWarp = kThreads / 32 - 1;   // issues every chunk's loads
    if (bos < eos && warp == kLoadWarp)
        issue_chunk_loads(sm, a, maps, bos, (int)((eos - bos) < C ? (eos - bos) : C), h, vt, lane);

    Tout *out = static_cast<Tout *>(a.out);
    uint32_t load_parity = 0, mma_parity = 0;
    bool failed = false;

    for (int64_t t0 = bos; t0 < eos; t0 += C) {
        const int len = (int)((eos - t0) < C ? (eos - t0) : C);
        cp_async_wait_all();
        if (!mbar_wait(mbar, load_parity)) failed = true;   // loads did not land: stop
        load_parity ^= 1u;
        if (!failed && len < C) zero_tail_rows(sm, len, tid);
        if (__syncthreads_or(failed)) { failed = true; break; }
        tc_fence_after();
        if (tid == 0) *flag = 0;

        // ---------------- P1: in-chunk gate cumsum, exp2 space; thread = (channel pair, 8-row group E)
        const int pcp = tid & 63, pE = tid >> 6, pc0 = 2 * pcp;
        float2 gx[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const float2 g2 = *reinterpret_cast<const float2 *>(graw + (8 * pE + u) * KD + pc0);
            gx[u] = make_float2(g2.x * kLog2e, g2.y * kLog2e);
        }
#pragma unroll
        for (int u = 1; u < 8; ++u) { gx[u].x += gx[u - 1].x; gx[u].y += gx[u - 1].y; }
        *reinterpret_cast<float2 *>(tot8 + pE * KD + pc0) = gx[7];
        *reinterpret_cast<float2 *>(first8 + pE * KD + pc0) = gx[0];
        if (tid < C * VT * 2 / 16)   // copy v (4 KB) out of the raw buffer, 16 B per thread
            reinterpret_cast<uint4 *>(vs)[tid] = reinterpret_cast<const uint4 *>(sm + Smem::v_raw)[tid];
        if (tid < C) beta_s[tid] = tid < len ? braw[tid * 4 + (maps.beta_tma ? (h & 3) : 0)] : 0.f;
        __syncthreads();

        // ---------------- P2: per-block references, scalars, factors and fp16 operands
        {
            // prefix sums over the 8-row groups; block references m_R = G(row 16R+8)
            float2 pre = make_float2(0.f, 0.f), run = make_float2(0.f, 0.f), mAll[4];
#pragma unroll
            for (int E = 0; E < 8; ++E) {
                const float2 t = *reinterpret_cast<const float2 *>(tot8 + E * KD + pc0);
                if (E & 1) {
                    const float2 f = *reinterpret_cast<const float2 *>(first8 + E * KD + pc0);
                    mAll[E >> 1] = make_float2(run.x + f.x, run.y + f.y);
                }
                if (E == pE) pre = run;
                run.x += t.x; run.y += t.y;
            }
            const float2 glast = run;
            float2 mR = mAll[0];
#pragma unroll
            for (int R = 1; R < 4; ++R) if (R == (pE >> 1)) mR = mAll[R];
            if (pE >= 4) {   // pair factors of block R = pE - 4, two channels
                const int R = pE & 3;
                float2 m = mAll[0];
#pragma unroll
                for (int RR = 1; RR < 4; ++RR) if (RR == R) m = mAll[RR];
#pragma unroll
                for (int I = 0; I < 3; ++I)
                    if (I < R)
                        *reinterpret_cast<uint32_t *>(rho + (R * (R - 1) / 2 + I) * KD + pc0) =
                            pack_h2(exp2f(m.x - mAll[I].x), exp2f(m.y - mAll[I].y));
            } else if (pE == 0) {
                *reinterpret_cast<float2 *>(dec + pc0) = make_float2(exp2f(glast.x), exp2f(glast.y));
            }
            // this block's scales 2^m_R (for K~, Q~) and 2^(G_last - m_R) (for K^)
            const float pmx = exp2f(mR.x), pmy = exp2f(mR.y);
            const float fmx = exp2f(glast.x - mR.x), fmy = exp2f(glast.y - mR.y);
            const float bx = pre.x - mR.x, by = pre.y - mR.y;   // G_r - m_R = gx + b
            bool bad = false;
            float khx[8], khy[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int r = 8 * pE + u;
                const float emx = exp2f(gx[u].x + bx), emy = exp2f(gx[u].y + by);
                bad |= !(emx <= kFactorMax && emx >= 1.f / kFactorMax &&
                         emy <= kFactorMax && emy >= 1.f / kFactorMax);
                const float epx = recip_nr(emx), epy = recip_nr(emy);
                const float2 kv = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(kraw + r * KD + pc0));
                const float2 qv = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(qraw + r * KD + pc0));
                const float akx = kv.x * emx, aky = kv.y * emy, aqx = qv.x * emx, aqy = qv.y * emy;
                const float bkx = kv.x * epx, bky = kv.y * epy;
                *reinterpret_cast<uint32_t *>(ak + r * LD128 + pc0) = pack_h2(akx, aky);
                *reinterpret_cast<uint32_t *>(aq + r * LD128 + pc0) = pack_h2(aqx, aqy);
                *reinterpret_cast<uint32_t *>(bk + r * LD128 + pc0) = pack_h2(bkx, bky);
                *reinterpret_cast<uint32_t *>(a1 + sw128(r, pc0, 2 * C)) = pack_h2(-akx * pmx, -aky * pmy);
                *reinterpret_cast<uint32_t *>(a1 + sw128(C + r, pc0, 2 * C)) = pack_h2(aqx * pmx, aqy * pmy);
                khx[u] = bkx * fmx;
                khy[u] = bky * fmy;
            }
            // K^^T: the eight rows of this group are one 16-byte chunk of key-channel row c
            *reinterpret_cast<uint4 *>(kht + sw128(pc0, 8 * pE, KD)) =
                make_uint4(pack_h2(khx[0], khx[1]), pack_h2(khx[2], khx[3]),
                           pack_h2(khx[4], khx[5]), pack_h2(khx[6], khx[7]));
            *reinterpret_cast<uint4 *>(kht + sw128(pc0 + 1, 8 * pE, KD)) =
                make_uint4(pack_h2(khy[0], khy[1]), pack_h2(khy[2], khy[3]),
                           pack_h2(khy[4], khy[5]), pack_h2(khy[6], khy[7]));
            if (__any_sync(0xffffffffu, bad) && lane == 0) *flag = 1;
        }
        __syncthreads();
        const bool exact_path = *flag != 0;

        // The raw buffers are free once P2 has read them, except on the exact path,
        // which reads them during P3: the load warp fetches the next chunk now (or,
        // on the exact path, after P3) so the copies overlap the rest of this chunk.
        if (warp == kLoadWarp && !exact_path && t0 + C < eos) {
            const int64_t t1 = t0 + C;
            issue_chunk_loads(sm, a, maps, t1, (int)((eos - t1) < C ? (eos - t1) : C), h, vt, lane);
        }

        // ---------------- P3: A_kk and A_qk (lower block triangle) on tensor cores
        // Ten tasks, one 16x16 block (R, I <= R) each, both matrices per task (the B
        // fragments of block I serve A_kk and A_qk); warp w % 4 picks the scheduler, so
        // the tasks are placed three, three, two and two per scheduler.  Warps 10..13
        // invert the diagonal blocks as soon as the task that owns them has stored them.
        if (!exact_path) {
            if (warp < 10) {
                const int R = warp < 4 ? 3 : warp < 7 ? 2 : warp < 9 ? 1 : 0;
                const int I = warp < 4 ? warp : warp < 7 ? warp - 4 : warp < 9 ? warp - 7 : 0;
                float acc[2][2][4];   // [matrix][n8 tile][frag]
#pragma unroll
                for (int m = 0; m < 2; ++m)
#pragma unroll
                    for (int t = 0; t < 2; ++t) acc[m][t][0] = acc[m][t][1] = acc[m][t][2] = acc[m][t][3] = 0.f;
                const __half *rp = rho + (I < R ? R * (R - 1) / 2 + I : 0) * KD + 2 * tig;
#pragma unroll
                for (int ks = 0; ks < KD / 16; ++ks) {
                    uint32_t fk[4], fq[4], bf[4];
                    ldsm_x4(smem_u32(ak + a_off(lane, 16 * R, 16 * ks, LD128)), fk[0], fk[1], fk[2], fk[3]);
                    ldsm_x4(smem_u32(aq + a_off(lane, 16 * R, 16 * ks, LD128)), fq[0], fq[1], fq[2], fq[3]);
                    ldsm_x4(smem_u32(bk + bnk_off(lane, 16 * I, 16 * ks, LD128)), bf[0], bf[1], bf[2], bf[3]);
                    if (I < R) {
                        const uint32_t s0 = *reinterpret_cast<const uint32_t *>(rp + 16 * ks);
                        const uint32_t s1 = *reinterpret_cast<const uint32_t *>(rp + 16 * ks + 8);
                        bf[0] = hmul2_u32(bf[0], s0); bf[1] = hmul2_u32(bf[1], s1);
                        bf[2] = hmul2_u32(bf[2], s0); bf[3] = hmul2_u32(bf[3], s1);
                    }
                    mma16816(acc[0][0], fk, bf[0], bf[1]);
                    mma16816(acc[0][1], fk, bf[2], bf[3]);
                    mma16816(acc[1][0], fq, bf[0], bf[1]);
                    mma16816(acc[1][1], fq, bf[2], bf[3]);
                }
#pragma unroll
                for (int t = 0; t < 2; ++t) {
#pragma unroll
                    for (int hh = 0; hh < 2; ++hh) {
                        const int r = 16 * R + g8 + 8 * hh;
                        const int i = 16 * I + 8 * t + 2 * tig;
                        const float k0 = acc[0][t][2 * hh], k1 = acc[0][t][2 * hh + 1];
                        *reinterpret_cast<uint32_t *>(akh + sw128(r, i, C)) =
                            pack_h2(i < r ? beta_s[r] * k0 : 0.f, i + 1 < r ? beta_s[r] * k1 : 0.f);
                        const float q0 = acc[1][t][2 * hh], q1 = acc[1][t][2 * hh + 1];
                        *reinterpret_cast<uint32_t *>(aqk + sw128(r, i, C)) =
                            pack_h2(i <= r ? q0 : 0.f, i + 1 <= r ? q1 : 0.f);
                    }
                }
                if (I == R) named_bar_arrive(1 + R, 64);   // diagonal block stored
            } else if (warp < 14) {
                const int R = warp - 10;
                named_bar_sync(1 + R, 64);
                invert_diag_block(akh, tmh, R, lane);
            }
        } else {
            exact_intra_chunk(sm, tid);
            __syncthreads();
            if (warp >= 10 && warp < 14) invert_diag_block(akh, tmh, warp - 10, lane);
        }
        fence_proxy_async_smem();   // A_qk, -K~/Q~ and K^^T are read by tcgen05 below
        __syncthreads();

        // exact path: the raw buffers are free now (the solve's barriers below are
        // named, without the load warp)
        if (warp == kLoadWarp && exact_path && t0 + C < eos) {
            const int64_t t1 = t0 + C;
            issue_chunk_loads(sm, a, maps, t1, (int)((eos - t1) < C ? (eos - t1) : C), h, vt, lane);
        }

        // ---------------- S1 issue: D1 = [-K~; Q~] h  (X part in rows 0..63, o part in 64..127)
        if (tid == 0) {
            tc_fence_after();
#pragma unroll
            for (int ks = 0; ks < KD / 16; ++ks)
                umma_f16(tD1, sw128_kdesc(smem_u32(a1), ks, 2 * C), sw128_kdesc(smem_u32(ht), ks, VT),
                         kIdescM128N32, ks > 0);
            umma_commit(mbar_mma);
        }

        // ---------------- P4: T = (I + A_kk)^-1 in 16x16 blocks
        // Diagonal blocks were inverted during P3.  Below-diagonal blocks, by distance
        // from the diagonal:
        //     T_RI = -T_RR sum_{J=I}^{R-1} A_RJ T_JI
        // on tensor cores, evaluated transposed (X^T = sum T_JI^T A_RJ^T, then
        // T_RI^T = -X^T T_RR^T) so X^T passes from accumulator to operand in registers.
        {
            constexpr int kSolveThreads = kThreads - 32;   // all warps but the load warp
            for (int lvl = 1; lvl < 4 && warp != kLoadWarp; ++lvl) {
                if (warp < 4 - lvl) {
                    const int I = warp, R = warp + lvl;
                    float xa[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
                    for (int J = I; J < R; ++J) {
                        uint32_t af[4], bf[4];
                        // A = T_JI^T (rows i, cols m) from T_JI stored [m][i]
                        ldsm_x4_t(smem_u32(tmh + (16 * J + (lane & 7) + ((lane >> 4) << 3)) * LD64 +
                                           16 * I + (((lane >> 3) & 1) << 3)),
                                  af[0], af[1], af[2], af[3]);
                        // B = A_RJ^T as [k=m][n=r] from A_RJ stored (swizzled) [r][m]
                        const int bn = 16 * R + (lane & 7) + ((lane >> 4) << 3);
                        const int bkk = 16 * J + (((lane >> 3) & 1) << 3);
                        ldsm_x4(smem_u32(akh + sw128(bn, bkk, C)), bf[0], bf[1], bf[2], bf[3]);
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
                named_bar_sync(5, kSolveThreads);
            }
        }

        // ---------------- S1: decay the state for this chunk, then X = V - K~ h from D1
        if (state_warp) {   // h <- Diag(2^G_last) h  (before K^^T D is accumulated into it)
            tc_fence_after();
            float hv[16];
            tmem_ld16(tH + lane_off + 16 * hc, hv);
            const float d = dec[sc];
#pragma unroll
            for (int v = 0; v < 16; ++v) hv[v] *= d;
            tmem_st16(tH + lane_off + 16 * hc, hv);
            tc_fence_before();
        }
        if (!mbar_wait(mbar_mma, mma_parity)) failed = true;
        mma_parity ^= 1u;
        tc_fence_after();
        if (warp == 0 || warp == 1 || warp == 4 || warp == 5) {   // rows 0..63 of D1: -K~ h
            const int r = 32 * (warp & 1) + lane, half = warp >> 2;
            float xv[16];
            tmem_ld16(tD1 + ((uint32_t)(32 * (warp & 3)) << 16) + 16 * half, xv);
            const float b = beta_s[r];
            const uint4 *vrow = reinterpret_cast<const uint4 *>(vs + r * VT + 16 * half);
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const uint4 w = vrow[j];
                const __nv_bfloat162 *p2 = reinterpret_cast<const __nv_bfloat162 *>(&w);
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const float2 vv = __bfloat1622float2(p2[u]);
                    const int v = 8 * j + 2 * u;
                    xt[(16 * half + v) * LD64 + r] = __float2half_rn(b * (vv.x + xv[v]));
                    xt[(16 * half + v + 1) * LD64 + r] = __float2half_rn(b * (vv.y + xv[v + 1]));
                }
            }
            tc_fence_before();
        }
        __syncthreads();

        // ---------------- S2: D^T = (beta X)^T T^T  (mma.sync; T lower triangular: k-blocks <= qw/2)
        {
            const int mt = warp & 1, qw = warp >> 1, rblk = qw >> 1;
            float dacc[4] = {0.f, 0.f, 0.f, 0.f};
            const int brow = (8 * qw + (lane & 7)) * LD64 + (((lane >> 3) & 1) << 3);
            for (int ks = 0; ks <= rblk; ++ks) {
                uint32_t af[4], bt[2];
                ldsm_x4(smem_u32(xt + a_off(lane, 16 * mt, 16 * ks, LD64)), af[0], af[1], af[2], af[3]);
                ldsm_x2(smem_u32(tmh + brow + 16 * ks), bt[0], bt[1]);
                mma16816(dacc, af, bt[0], bt[1]);
            }
            const int r = 8 * qw + 2 * tig;
            const int v0 = 16 * mt + g8;
            *reinterpret_cast<uint32_t *>(dt + sw128(v0, r, VT)) = pack_h2(dacc[0], dacc[1]);
            *reinterpret_cast<uint32_t *>(dt + sw128(v0 + 8, r, VT)) = pack_h2(dacc[2], dacc[3]);
        }
        fence_proxy_async_smem();
        __syncthreads();

        // ---------------- S3: h += K^^T D ; D1[64..127] += A_qk D  (one tcgen05 batch)
        if (tid == 0) {
            tc_fence_after();
#pragma unroll
            for (int ks = 0; ks < C / 16; ++ks)
                umma_f16(tH, sw128_kdesc(smem_u32(kht), ks, KD), sw128_kdesc(smem_u32(dt), ks, VT),
                         kIdescM128N32, 1u);
            // A = [A_kk (rows 0..63, lands in the consumed X rows); A_qk (rows 64..127)]
#pragma unroll
            for (int ks = 0; ks < C / 16; ++ks)
                umma_f16(tD1, sw128_kdesc(smem_u32(akh), ks, 2 * C), sw128_kdesc(smem_u32(dt), ks, VT),
                         kIdescM128N32, 1u);
            umma_commit(mbar_mma);
        }
        if (!mbar_wait(mbar_mma, mma_parity)) failed = true;
        mma_parity ^= 1u;
        tc_fence_after();
        if (warp == 2 || warp == 3 || warp == 6 || warp == 7) {   // rows 64..127 of D1: o
            const int r = 32 * (warp & 1) + lane, half = warp >> 2;
            float ov[16];
            tmem_ld16(tD1 + ((uint32_t)(32 * (warp & 3)) << 16) + 16 * half, ov);
            if (r < len) store_row16(out + ((t0 + r) * H + h) * VD + vt * VT + 16 * half, ov, a.scale);
        }
        if (state_warp) {   // fp16 mirror of the new state for the next chunk's S1
            float hv[16];
            tmem_ld16(tH + lane_off + 16 * hc, hv);
#pragma unroll
            for (int v = 0; v < 16; ++v) ht[sw128(16 * hc + v, sc, VT)] = __float2half_rn(hv[v]);
            fence_proxy_async_smem();
        }
        tc_fence_before();
        if (__syncthreads_or(failed)) { failed = true; break; }
    }

    if (failed) {
        // error marker: NaN state; copies or MMAs still in flight get one more bounded wait
        mbar_wait(mbar, load_parity);
        mbar_wait(mbar_mma, mma_parity);
    }
    if (fin && state_warp) {
        tc_fence_after();
        float hv[16];
        tmem_ld16(tH + lane_off + 16 * hc, hv);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            float4 x = make_float4(hv[4 * j], hv[4 * j + 1], hv[4 * j + 2], hv[4 * j + 3]);
            if (failed) x = make_float4(__int_as_float(0x7fc00000), __int_as_float(0x7fc00000),
                                        __int_as_float(0x7fc00000), __int_as_float(0x7fc00000));
            *reinterpret_cast<float4 *>(fin + (int64_t)sc * VD + vt * VT + 16 * hc + 4 * j) = x;
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" :: "r"(tmem), "r"(64) : "memory");
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

// beta [T, H] fp32 as a 2-D map, box 4 heads x 64 tokens (needs H % 4 == 0 for the
// 16-byte row pitch)
bool encode_map_2d(CUtensorMap *m, const float *base, int64_t T, int H)
{
    auto enc = tensor_map_encoder();
    if (!enc) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)H, (cuuint64_t)T};
    const cuuint64_t strides[1] = {(cuuint64_t)H * 4};
    const cuuint32_t box[2] = {4u, (cuuint32_t)C};
    const cuuint32_t estr[2] = {1u, 1u};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float *>(base), dims, strides, box,
               estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
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
        maps.beta_tma = (H % 4 == 0) && encode_map_2d(&maps.beta, a.beta, T, H);
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
