// kda_tc_common.cuh -- constants, PTX wrappers (mma.sync, ldmatrix, TMA, mbarrier,
// tcgen05) and the blocked triangular inverse shared by the tensor-core prefill
// kernels.  Internal; every definition has internal linkage.
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>
#include <cudaTypedefs.h>

#include "kda_internal.cuh"

namespace kda {
namespace {

constexpr int C = kChunk;        // 64 rows per chunk
constexpr int KD = 128;          // key dim
constexpr int VD = 128;          // value dim
constexpr int VT = 32;           // value columns per CTA
constexpr int kVTiles = VD / VT;
constexpr int LD64 = C + 8;      // f16 row stride of 64-column tiles: 144 B
constexpr float kSpanMax = 16.f; // widest in-chunk gate span (log2) of the fp16 fast path

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

// four 8x8 b16 matrices from registers to shared memory, transposed: register i of
// thread (g, t) holds elements (g, 2t), (g, 2t + 1) of matrix i, which land in rows 2t,
// 2t + 1, column g of the stored matrix; lane 8 i + j gives the address of row j of
// stored matrix i (16 bytes)
__device__ __forceinline__ void stsm_x4_t(uint32_t addr, uint32_t r0, uint32_t r1, uint32_t r2,
                                          uint32_t r3)
{
    asm volatile("stmatrix.sync.aligned.m8n8.x4.trans.shared.b16 [%0], {%1, %2, %3, %4};\n"
                 :: "r"(addr), "r"(r0), "r"(r1), "r"(r2), "r"(r3) : "memory");
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

// 1/x on the special-function unit (approximate reciprocal, relative error ~2^-23,
// far below the fp16 rounding of every operand it feeds)
__device__ __forceinline__ float rcp_approx(float x)
{
    float y;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// 2^x on the special-function unit (ex2.approx.ftz, relative error ~2^-22; results below
// the normal range flush to zero, which the fast path's factors in [2^-8, 2^8] never are)
__device__ __forceinline__ float ex2_approx(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ void named_bar_sync(int id, int count)
{
    asm volatile("bar.sync %0, %1;\n" :: "r"(id), "r"(count) : "memory");
}
// named barrier over `count` threads that also ORs `pred` across them
__device__ __forceinline__ bool bar_red_or(int id, int count, bool pred)
{
    int r;
    asm volatile("{\n.reg .pred p, q;\nsetp.ne.b32 p, %1, 0;\nbar.red.or.pred q, %2, %3, p;\n"
                 "selp.b32 %0, 1, 0, q;\n}\n"
                 : "=r"(r) : "r"((int)pred), "r"(id), "r"(count) : "memory");
    return r != 0;
}

__device__ __forceinline__ void mbar_arrive(uint32_t mbar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" :: "r"(mbar) : "memory");
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

// instruction descriptors: fp16 A and B (K-major), fp32 D, M = 128, N = 32 / 64
constexpr uint32_t kIdescM128N32 = (1u << 4) | ((32u >> 3) << 17) | ((128u >> 4) << 24);
// the same with N = 64
constexpr uint32_t kIdescM128N64 = (1u << 4) | ((64u >> 3) << 17) | ((128u >> 4) << 24);

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

// T_RR = (I + A_RR)^-1 of the 16x16 diagonal blocks R = 2 P and 2 P + 1 by fp32
// forward substitution on the fp16 A_kk, right-looking: half-warp R % 2, lane j owns
// column j of block R; once T[m][j] is final, every row below it is updated,
//     T[r][j] -= A[r][m] T[m][j]    (r > m),
// so the dependent chain is one multiply-add per step.  Columns m, m + 1 of A are
// read as one 4-byte broadcast per row.  Written to T (fp16) with its zeros and unit
// diagonal.
__device__ __forceinline__ void invert_diag_blocks(const __half *akh, __half *tmh, int P, int lane)
{
    const int j = lane & 15, R = 2 * P + (lane >> 4);
    float col[16];
#pragma unroll
    for (int m = 0; m < 16; ++m) col[m] = (m == j) ? 1.f : 0.f;
#pragma unroll
    for (int mp = 0; mp < 8; ++mp) {
        const int m = 2 * mp;
        float2 am[16];   // (A[r][m], A[r][m + 1]) for r > m
#pragma unroll
        for (int r = m + 1; r < 16; ++r)
            am[r] = __half22float2(*reinterpret_cast<const __half2 *>(akh + sw128(16 * R + r, 16 * R + m, C)));
#pragma unroll
        for (int r = m + 1; r < 16; ++r) col[r] -= am[r].x * col[m];
#pragma unroll
        for (int r = m + 2; r < 16; ++r) col[r] -= am[r].y * col[m + 1];
    }
#pragma unroll
    for (int rr = 0; rr < 16; ++rr) tmh[(16 * R + rr) * LD64 + 16 * R + j] = __float2half_rn(col[rr]);
}

// T_RI (R > I) of column block I, top to bottom, by ONE warp (no barrier between the
// blocks of a column: each needs only T_JI, I <= J < R, of the same column):
//     T_RI = -T_RR sum_{J=I}^{R-1} A_RJ T_JI
// on tensor cores, evaluated transposed (X^T = sum T_JI^T A_RJ^T, then
// T_RI^T = -X^T T_RR^T) so X^T passes from accumulator to operand in registers.
__device__ __forceinline__ void solve_column_block(const __half *akh, __half *tmh, int I, int lane)
{
    const int g8 = lane >> 2, tig = lane & 3;
#pragma unroll
    for (int R = I + 1; R < 4; ++R) {
        float xj[3][2][4];   // one accumulator per J, summed afterwards (no chained mma)
#pragma unroll
        for (int J = I; J < R; ++J) {
            float (&xa)[2][4] = xj[J - I];
#pragma unroll
            for (int t = 0; t < 2; ++t) xa[t][0] = xa[t][1] = xa[t][2] = xa[t][3] = 0.f;
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
        float xa[2][4];
#pragma unroll
        for (int t = 0; t < 2; ++t)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                float acc = xj[0][t][e];
#pragma unroll
                for (int J = I + 1; J < R; ++J) acc += xj[J - I][t][e];
                xa[t][e] = acc;
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
                const int rr = 16 * R + 8 * nt + 2 * tig + (e & 1);
                tmh[rr * LD64 + i] = __float2half_rn(ta[nt][e]);
            }
        __syncwarp();   // T_RI is read (ldmatrix, other lanes) by the next block of the column
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

}  // namespace
}  // namespace kda
