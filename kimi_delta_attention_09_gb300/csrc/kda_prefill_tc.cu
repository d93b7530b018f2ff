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
//   and the diagonal blocks of the triangular solve are fp32.  bf16 operands miss a
//   2e-3 relative bar by 2-3x; fp16 operands meet it with ~3x margin.
// * fp16 range is handled by factoring 2^(G_r - G_i) around one per-channel reference
//   m = (max_r G_r + min_r G_r) / 2 of the chunk:  a_r = x_r 2^(G_r - m) and
//   b_i = k_i 2^(m - G_i), so every stored factor lies in [2^-8, 2^8] while the gate
//   spans at most 16 (log2 units) over the chunk -- about 11 per 64 rows at the
//   gate strength of the synthetic workloads.  A chunk with a wider span (gates below
//   about -0.17 per step sustained over the chunk) takes an exact-exponential
//   CUDA-core path for A_kk and A_qk instead; its result is the same algebra.
// * The state-step product [K~; Q~] h is evaluated as [a_k; a_q] (2^m h), with the
//   fp16 copy of the state scaled by 2^m per key channel (m capped at max G - 8, so
//   a_r stays below 2^8 on either path).
//
// Mapping: one CTA (16 warps) per (sequence, head, 32-column tile of V); it walks its
// sequence chunk by chunk.  The raw inputs of a chunk arrive as TMA tiles (issued one
// chunk ahead by a dedicated warp).  Per chunk:
//   P1/P2  gate cumsum, reference, factors; fp16 operands [a_k; a_q] (128 x 128),
//          b (64 x 128) and K^^T (128 x 64) in 128-byte-swizzled K-major layout
//   MMA A  [A_kk'; A_qk'] = [a_k; a_q] b^T on tcgen05 (M 128, N 64, K 128) into TMEM
//   MMA S1 [K~ h; Q~ h] = [a_k; a_q] (2^m h) on tcgen05 (N 32), issued once the state
//          warps have refreshed the scaled fp16 state copy and decayed the TMEM state
//   epilogues: masked, beta-scaled A_kk and A_qk to fp16; X = beta (v - K~ h)
//   solve  T = (I + A_kk)^-1: 16x16 diagonal blocks by fp32 forward substitution,
//          the rest blockwise on mma.sync;  D = T X on mma.sync
//   MMA S3 h += K^^T D and o-rows += A_qk D on tcgen05; o epilogue to global.
#include <cstring>

#include "kda_tc_common.cuh"

namespace kda {
namespace {

constexpr int kThreads = 512;   // 16 warps: two groups of 8
constexpr int kGroup = 256;     // threads per group
constexpr int kBarPrep = 1;     // named barrier of the operand group (warps 8..15)
constexpr int kBarStep = 2;     // named barrier of the state-step group (warps 0..7)

// Shared memory map (byte offsets).  SW128 tiles: 128-byte-swizzled K-major tcgen05
// operands (1024-byte aligned); the others are padded row-major mma.sync operands.
// "x2" buffers are double-buffered by chunk parity: the operand group fills slot
// n % 2 for chunk n while the state-step group still reads slot (n - 1) % 2.
struct Smem {
    static constexpr int q_raw = 0;                          // bf16 [64][128]
    static constexpr int k_raw = q_raw + C * KD * 2;         // bf16 [64][128]
    static constexpr int g_raw = k_raw + C * KD * 2;         // f32  [64][128] raw natural-log gate
    static constexpr int v_raw = g_raw + C * KD * 4;         // bf16 [64][32]
    static constexpr int b_raw = v_raw + C * VT * 2;         // f32  [64][4] beta of heads 4*(h/4)..
    static constexpr int tm = b_raw + C * 4 * 4;             // f16 T [64][LD64]
    static constexpr int vs = tm + C * LD64 * 2;             // x2 bf16 V [64][32]
    static constexpr int beta = vs + 2 * C * VT * 2;         // x2 f32 [64]
    static constexpr int dec = beta + 2 * C * 4;             // x2 f32 [128] 2^G_last
    static constexpr int pm = dec + 2 * KD * 4;              // x2 f32 [128] 2^m
    static constexpr int bars = pm + 2 * KD * 4;              // u64 mbarriers (see Bar)
    static constexpr int tmem = bars + 8 * 8;                // u32 tensor-memory base
    static constexpr int flag = tmem + 4;                    // int: exact path for this chunk
    static constexpr int aop = (flag + 4 + 1023) / 1024 * 1024;   // SW128 [a_k; a_q] 128 x 128
    static constexpr int bk = aop + 2 * C * KD * 2;          // SW128 b: 64 (row) x 128 (channel)
    static constexpr int kht = bk + C * KD * 2;              // x2 SW128 K^^T: 128 (channel) x 64 (row)
    static constexpr int akh = kht + 2 * KD * C * 2;         // x2 [SW128 A_kk 64 x 64; SW128 A_qk 64 x 64]
                                                             // ([A_kk; A_qk] is the 128-row A of o += A_qk D)
    static constexpr int ht = akh + 2 * 2 * C * C * 2;       // SW128 (2^m h)^T fp16 32 (value) x 128 (channel)
    static constexpr int xt = ht;                            // f16 (beta X)^T [32][LD64]: written once S1
                                                             // (the only reader of ht) has completed
    static constexpr int dt = ht + VT * KD * 2;              // SW128 D^T fp16 32 (value) x 64 (row)
    static constexpr int tot = bk;                           // f32 [4][128] 16-row group sums } P1/P2
    static constexpr int first = bk + 4 * KD * 4;            // f32 [128] G of row 0           } only
    static constexpr int total = dt + VT * C * 2;
};
// mbarriers: chunk loads, A MMA, S1 MMA, S3 MMA, operands ready, slot 0 / 1 released
struct Bar { enum { load = 0, a = 1, s1 = 2, s3 = 3, ready = 4, free0 = 5 }; };
static_assert(Smem::total <= 232448, "shared memory budget");
static_assert(Smem::aop % 1024 == 0 && Smem::bk % 1024 == 0 && Smem::kht % 1024 == 0 &&
              Smem::akh % 1024 == 0 && Smem::ht % 1024 == 0 && Smem::dt % 1024 == 0,
              "SW128 tiles need 1024-byte alignment");
static_assert(VT * LD64 * 2 <= VT * KD * 2, "(beta X)^T fits in the h^T space");
static_assert(Smem::first + KD * 4 <= Smem::kht, "gate group sums fit in the b space");

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
        const uint32_t mbar = smem_u32(sm + Smem::bars + 8 * Bar::load);
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

// Zero the rows [len, 64) of the raw tiles (tokens of the next sequence); one group.
__device__ __forceinline__ void zero_tail_rows(unsigned char *sm, int len, int gtid)
{
    for (int e = gtid; e < (C - len) * KD / 8; e += kGroup) {   // 16 B per store
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

// Exact-exponential intra-chunk matrices for chunks whose gate span leaves the fp16
// fast path (run by the operand group).  Recomputes the exp2-space cumsum G in place
// in g_raw, then writes A_kk
// and A_qk (fp16, zeros above the diagonal) with one exponential per pair and
// channel, and K^^T with one exponential per element (its fast-path values can
// overflow at such spans).
__device__ __noinline__ void exact_intra_chunk(unsigned char *sm, int gtid, const float *beta,
                                               __half *akh, __half *aqk, __half *kht)
{
    const __nv_bfloat16 *qr = reinterpret_cast<const __nv_bfloat16 *>(sm + Smem::q_raw);
    const __nv_bfloat16 *kr = reinterpret_cast<const __nv_bfloat16 *>(sm + Smem::k_raw);
    float *G = reinterpret_cast<float *>(sm + Smem::g_raw);
    if (gtid < KD) {
        float acc = 0.f;
        for (int r = 0; r < C; ++r) { acc += G[r * KD + gtid] * kLog2e; G[r * KD + gtid] = acc; }
    }
    named_bar_sync(kBarPrep, kGroup);
    for (int p = gtid; p < C * (C + 1) / 2; p += kGroup) {
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
    for (int e = gtid; e < C * KD; e += kGroup) {
        const int r = e >> 7, c = e & 127;
        const float gr = G[r * KD + c], gl = G[(C - 1) * KD + c];
        kht[sw128(c, r, KD)] = __float2half_rn(__bfloat162float(kr[r * KD + c]) * exp2f(gl - gr));
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

    __half *aop = reinterpret_cast<__half *>(sm + Smem::aop);
    __half *ht = reinterpret_cast<__half *>(sm + Smem::ht);
    __half *dt = reinterpret_cast<__half *>(sm + Smem::dt);
    __half *xt = reinterpret_cast<__half *>(sm + Smem::xt);
    // slot buffers of chunk parity s
    auto vs_s = [&](int s) { return reinterpret_cast<__nv_bfloat16 *>(sm + Smem::vs) + s * C * VT; };
    auto beta_s = [&](int s) { return reinterpret_cast<float *>(sm + Smem::beta) + s * C; };
    auto dec_s = [&](int s) { return reinterpret_cast<float *>(sm + Smem::dec) + s * KD; };
    auto pm_s = [&](int s) { return reinterpret_cast<float *>(sm + Smem::pm) + s * KD; };
    auto kht_s = [&](int s) { return reinterpret_cast<__half *>(sm + Smem::kht) + s * KD * C; };
    auto akh_s = [&](int s) { return reinterpret_cast<__half *>(sm + Smem::akh) + s * 2 * C * C; };
    auto bar = [&](int b) { return smem_u32(sm + Smem::bars + 8 * b); };

    int64_t bos, eos;
    clamp_range(a.total_tokens, a.cu_seqlens[n], a.cu_seqlens[n + 1], bos, eos);
    const float *init;
    float *fin;
    prefill_state_ptrs(a, n, h, init, fin);

    // ---- tensor memory (128 columns: [0, 32) the step accumulator D1, [32, 64) the
    //      state h^T with lane = key channel, column = value, [64, 128) the A matrices)
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n"
                     :: "r"(smem_u32(sm + Smem::tmem)), "r"(128) : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n" ::: "memory");
    }
    if (tid == 0)
        for (int b = 0; b <= Bar::free0 + 1; ++b) mbar_init(bar(b), 1);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(sm + Smem::tmem);
    const uint32_t tD1 = tmem, tH = tmem + 32, tDA = tmem + 64;
    const uint32_t lane_off = (uint32_t)(32 * (warp & 3)) << 16;   // TMEM lane quadrant of this warp
    bool failed = false;

    if (warp >= 8) {
        // =====================================================================
        // Operand group (warps 8..15): for chunk n, the gate cumsum, reference and
        // factors, the fp16 operands and A_kk / A_qk (tcgen05 + epilogue), into
        // slot n % 2; it runs one chunk ahead of the state-step group.
        // =====================================================================
        const int gtid = tid - kGroup;
        constexpr int kLoadWarp = 15;   // issues every chunk's loads
        if (bos < eos && warp == kLoadWarp)
            issue_chunk_loads(sm, a, maps, bos, (int)((eos - bos) < C ? (eos - bos) : C), h, vt, lane);
        const float *graw = reinterpret_cast<const float *>(sm + Smem::g_raw);
        const __nv_bfloat16 *qraw = reinterpret_cast<const __nv_bfloat16 *>(sm + Smem::q_raw);
        const __nv_bfloat16 *kraw = reinterpret_cast<const __nv_bfloat16 *>(sm + Smem::k_raw);
        const float *braw = reinterpret_cast<const float *>(sm + Smem::b_raw);
        __half *bop = reinterpret_cast<__half *>(sm + Smem::bk);
        float *tot = reinterpret_cast<float *>(sm + Smem::tot);
        float *first = reinterpret_cast<float *>(sm + Smem::first);
        volatile int *flag = reinterpret_cast<volatile int *>(sm + Smem::flag);
        uint32_t load_parity = 0, a_parity = 0;

        int ci = 0;
        for (int64_t t0 = bos; t0 < eos; t0 += C, ++ci) {
            const int len = (int)((eos - t0) < C ? (eos - t0) : C);
            const int s = ci & 1;
            __half *kht = kht_s(s), *akh = akh_s(s), *aqk = akh + C * C;
            float *bs = beta_s(s);
            // slot s is free once the step of chunk ci - 2 has ended
            if (ci >= 2 && !mbar_wait(bar(Bar::free0 + s), ((ci - 2) >> 1) & 1)) failed = true;
            cp_async_wait_all();
            if (!mbar_wait(bar(Bar::load), load_parity)) failed = true;   // loads did not land: stop
            load_parity ^= 1u;
            if (!failed && len < C) zero_tail_rows(sm, len, gtid);
            if (bar_red_or(kBarPrep, kGroup, failed)) { failed = true; break; }
            if (gtid == 0) *flag = 0;

            // ---------------- P1: in-chunk gate cumsum, exp2 space; thread = (channel pair, 16-row group E)
            const int pcp = gtid & 63, pE = gtid >> 6, pc0 = 2 * pcp;
            float2 gx[16];
#pragma unroll
            for (int u = 0; u < 16; ++u) {
                const float2 g2 = *reinterpret_cast<const float2 *>(graw + (16 * pE + u) * KD + pc0);
                gx[u] = make_float2(g2.x * kLog2e, g2.y * kLog2e);
            }
#pragma unroll
            for (int u = 1; u < 16; ++u) { gx[u].x += gx[u - 1].x; gx[u].y += gx[u - 1].y; }
            *reinterpret_cast<float2 *>(tot + pE * KD + pc0) = gx[15];
            if (pE == 0) *reinterpret_cast<float2 *>(first + pc0) = gx[0];
            // v (4 KB) and beta of this chunk into slot s
            reinterpret_cast<uint4 *>(vs_s(s))[gtid] = reinterpret_cast<const uint4 *>(sm + Smem::v_raw)[gtid];
            if (gtid < C) bs[gtid] = gtid < len ? braw[gtid * 4 + (maps.beta_tma ? (h & 3) : 0)] : 0.f;
            named_bar_sync(kBarPrep, kGroup);

            // ---------------- P2: reference, factors and the fp16 tcgen05 operands
            float2 pre = make_float2(0.f, 0.f), run = make_float2(0.f, 0.f);
#pragma unroll
            for (int E = 0; E < 4; ++E) {
                const float2 t = *reinterpret_cast<const float2 *>(tot + E * KD + pc0);
                if (E == pE) pre = run;
                run.x += t.x; run.y += t.y;
            }
            const float2 glast = run, g0 = *reinterpret_cast<const float2 *>(first + pc0);
            // reference: the midpoint of the first and last row's G (the midrange when
            // the gate is a decay), capped so that no factor 2^(G - m) exceeds 2^8 then
            const float mx_ = fmaxf(0.5f * (g0.x + glast.x), g0.x - 0.5f * kSpanMax);
            const float my_ = fmaxf(0.5f * (g0.y + glast.y), g0.y - 0.5f * kSpanMax);
            if (pE == 0) {
                *reinterpret_cast<float2 *>(pm_s(s) + pc0) = make_float2(exp2f(mx_), exp2f(my_));
                *reinterpret_cast<float2 *>(dec_s(s) + pc0) = make_float2(exp2f(glast.x), exp2f(glast.y));
            }
            const float fx = exp2f(glast.x - mx_), fy = exp2f(glast.y - my_);   // K^ = b 2^(G_last - m)
            const float bx = pre.x - mx_, by = pre.y - my_;                    // G_r - m = gx + b
            named_bar_sync(kBarPrep, kGroup);   // the group sums (in the b space) are read
            // [a_k; a_q] of the previous chunk is read by its S1 MMA: wait for it
            if (ci >= 1 && !mbar_wait(bar(Bar::s1), (ci - 1) & 1)) failed = true;
            float amax = 0.f;
#pragma unroll
            for (int hb = 0; hb < 2; ++hb) {
                float khx[8], khy[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const int r = 16 * pE + 8 * hb + u;
                    const float xx = gx[8 * hb + u].x + bx, xy = gx[8 * hb + u].y + by;   // G_r - m
                    amax = fmaxf(amax, fmaxf(fabsf(xx), fabsf(xy)));
                    const float ex = exp2f(xx), ey = exp2f(xy);
                    const float ix = rcp_approx(ex), iy = rcp_approx(ey);
                    const float2 kv = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(kraw + r * KD + pc0));
                    const float2 qv = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(qraw + r * KD + pc0));
                    *reinterpret_cast<uint32_t *>(aop + sw128(r, pc0, 2 * C)) = pack_h2(kv.x * ex, kv.y * ey);
                    *reinterpret_cast<uint32_t *>(aop + sw128(C + r, pc0, 2 * C)) = pack_h2(qv.x * ex, qv.y * ey);
                    const float b0 = kv.x * ix, b1 = kv.y * iy;
                    *reinterpret_cast<uint32_t *>(bop + sw128(r, pc0, C)) = pack_h2(b0, b1);
                    khx[u] = b0 * fx;
                    khy[u] = b1 * fy;
                }
                // K^^T: these eight rows are one 16-byte chunk of key-channel row c
                const int r0 = 16 * pE + 8 * hb;
                *reinterpret_cast<uint4 *>(kht + sw128(pc0, r0, KD)) =
                    make_uint4(pack_h2(khx[0], khx[1]), pack_h2(khx[2], khx[3]),
                               pack_h2(khx[4], khx[5]), pack_h2(khx[6], khx[7]));
                *reinterpret_cast<uint4 *>(kht + sw128(pc0 + 1, r0, KD)) =
                    make_uint4(pack_h2(khy[0], khy[1]), pack_h2(khy[2], khy[3]),
                               pack_h2(khy[4], khy[5]), pack_h2(khy[6], khy[7]));
            }
            // fast path: every factor 2^(G_r - m) within [2^-8, 2^8]
            if (__any_sync(0xffffffffu, !(amax <= 0.5f * kSpanMax)) && lane == 0) *flag = 1;
            fence_proxy_async_smem();   // the operands are read by tcgen05
            named_bar_sync(kBarPrep, kGroup);
            const bool exact_path = *flag != 0;

            if (!exact_path) {
                // ---------------- MMA A: [A_kk'; A_qk'] = [a_k; a_q] b^T
                if (gtid == 0) {
                    tc_fence_after();
#pragma unroll
                    for (int ks = 0; ks < KD / 16; ++ks)
                        umma_f16(tDA, sw128_kdesc(smem_u32(aop), ks, 2 * C), sw128_kdesc(smem_u32(bop), ks, C),
                                 kIdescM128N64, ks > 0);
                    umma_commit(bar(Bar::a));
                }
                // the raw buffers are free: fetch the next chunk
                if (warp == kLoadWarp && t0 + C < eos) {
                    const int64_t t1 = t0 + C;
                    issue_chunk_loads(sm, a, maps, t1, (int)((eos - t1) < C ? (eos - t1) : C), h, vt, lane);
                }
                // ---------------- A epilogue: masked, beta-scaled fp16 A_kk and A_qk
                //   lanes 0..63 A_kk, 64..127 A_qk; warp w: lane quadrant w % 4, columns [32 ((w / 4) % 2), +32)
                if (!mbar_wait(bar(Bar::a), a_parity)) failed = true;
                a_parity ^= 1u;
                tc_fence_after();
                const int c0 = 32 * ((warp >> 2) & 1), rg = 32 * (warp & 3) + lane;
                float av[2][16];
                tmem_ld16(tDA + lane_off + c0, av[0]);
                tmem_ld16(tDA + lane_off + c0 + 16, av[1]);
                const bool kk = rg < C;
                const int r = kk ? rg : rg - C;
                const float sb = kk ? bs[r] : 1.f;
                const int lim = kk ? r : r + 1;   // columns i < lim are kept
                __half *dst = kk ? akh : aqk;
#pragma unroll
                for (int t = 0; t < 4; ++t) {
                    uint32_t w[4];
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const int e = 8 * t + 2 * u, i = c0 + e;
                        const float x0 = i < lim ? sb * av[e >> 4][e & 15] : 0.f;
                        const float x1 = i + 1 < lim ? sb * av[(e + 1) >> 4][(e + 1) & 15] : 0.f;
                        w[u] = pack_h2(x0, x1);
                    }
                    *reinterpret_cast<uint4 *>(dst + sw128(r, c0 + 8 * t, C)) = make_uint4(w[0], w[1], w[2], w[3]);
                }
                tc_fence_before();
            } else {
                exact_intra_chunk(sm, gtid, bs, akh, aqk, kht);
                named_bar_sync(kBarPrep, kGroup);
                if (warp == kLoadWarp && t0 + C < eos) {
                    const int64_t t1 = t0 + C;
                    issue_chunk_loads(sm, a, maps, t1, (int)((eos - t1) < C ? (eos - t1) : C), h, vt, lane);
                }
            }
            fence_proxy_async_smem();   // A_kk, A_qk and K^^T are read by tcgen05 in the state step
            named_bar_sync(kBarPrep, kGroup);

            // operands of chunk ci are complete: hand slot s to the state step
            if (bar_red_or(kBarPrep, kGroup, failed)) { failed = true; break; }
            if (gtid == 0) mbar_arrive(bar(Bar::ready));
        }
        if (failed) {   // copies or MMAs still in flight get one more bounded wait
            mbar_wait(bar(Bar::load), load_parity);
            mbar_wait(bar(Bar::a), a_parity);
        }
    } else {
        // =====================================================================
        // State-step group (warps 0..7): per chunk, once its operands are ready,
        //   the scaled fp16 copy of h and the decay of h, S1, then T = (I + A_kk)^-1
        //   (warps 2, 3, 6) while warps 0, 1, 4, 5 form X = beta (v - K~ h), then
        //   D = T X, S3 and the output.  Warp w reaches TMEM lanes 32 (w % 4) ..;
        //   state roles: key channel sc = 32 (w % 4) + lane, value columns [16 hc, +16).
        // =====================================================================
        const int sc = 32 * (warp & 3) + lane;
        const int hc = (warp >> 2) & 1;
        {   // initial state -> tensor memory
            float hv[16];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float4 x = init ? *reinterpret_cast<const float4 *>(init + (int64_t)sc * VD + vt * VT + 16 * hc + 4 * j)
                                      : make_float4(0.f, 0.f, 0.f, 0.f);
                hv[4 * j] = x.x; hv[4 * j + 1] = x.y; hv[4 * j + 2] = x.z; hv[4 * j + 3] = x.w;
            }
            tmem_st16(tH + lane_off + 16 * hc, hv);
            tc_fence_before();
        }
        Tout *out = static_cast<Tout *>(a.out);
        int ci = 0;
        for (int64_t t0 = bos; t0 < eos; t0 += C, ++ci) {
            const int len = (int)((eos - t0) < C ? (eos - t0) : C);
            const int s = ci & 1, par = ci & 1;
            if (!mbar_wait(bar(Bar::ready), par)) failed = true;
            if (bar_red_or(kBarStep, kGroup, failed)) { failed = true; break; }
            tc_fence_after();

            // ---------------- fp16 copy (2^m h)^T for S1, then h <- Diag(2^G_last) h
            {
                float hv[16];
                tmem_ld16(tH + lane_off + 16 * hc, hv);
                const float p = pm_s(s)[sc], d = dec_s(s)[sc];
#pragma unroll
                for (int v = 0; v < 16; ++v) {
                    ht[sw128(16 * hc + v, sc, VT)] = __float2half_rn(p * hv[v]);
                    hv[v] *= d;
                }
                tmem_st16(tH + lane_off + 16 * hc, hv);
                fence_proxy_async_smem();
                tc_fence_before();
            }
            named_bar_sync(kBarStep, kGroup);

            // ---------------- MMA S1: D1 = [a_k; a_q] (2^m h) = [K~ h; Q~ h]
            if (tid == 0) {
                tc_fence_after();
#pragma unroll
                for (int ks = 0; ks < KD / 16; ++ks)
                    umma_f16(tD1, sw128_kdesc(smem_u32(aop), ks, 2 * C), sw128_kdesc(smem_u32(ht), ks, VT),
                             kIdescM128N32, ks > 0);
                umma_commit(bar(Bar::s1));
            }
            __half *tmh = reinterpret_cast<__half *>(sm + Smem::tm);
            const __half *akh = akh_s(s);
            // ---------------- T = (I + A_kk)^-1: the diagonal blocks (warps 2, 3, while S1 runs
            //                  and warps 0, 1, 4, 5 form X), then the column blocks 0, 1, 2
            //                  below them (warps 2, 3, 6)
            if (warp == 2 || warp == 3) invert_diag_blocks(akh, tmh, warp - 2, lane);
            // ---------------- X = beta (v - K~ h) from rows 0..63 of D1 (warps 0, 1, 4, 5)
            if ((warp & 2) == 0) {
                if (!mbar_wait(bar(Bar::s1), par)) failed = true;
                tc_fence_after();
                const int r = 32 * (warp & 1) + lane, half = warp >> 2;
                float xv[16];
                tmem_ld16(tD1 + lane_off + 16 * half, xv);
                const float b = beta_s(s)[r];
                const uint4 *vrow = reinterpret_cast<const uint4 *>(vs_s(s) + r * VT + 16 * half);
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    const uint4 w = vrow[j];
                    const __nv_bfloat162 *p2 = reinterpret_cast<const __nv_bfloat162 *>(&w);
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const float2 vv = __bfloat1622float2(p2[u]);
                        const int v = 8 * j + 2 * u;
                        xt[(16 * half + v) * LD64 + r] = __float2half_rn(b * (vv.x - xv[v]));
                        xt[(16 * half + v + 1) * LD64 + r] = __float2half_rn(b * (vv.y - xv[v + 1]));
                    }
                }
                tc_fence_before();
            }
            named_bar_sync(kBarStep, kGroup);
            if (warp == 2 || warp == 3 || warp == 6) solve_column_block(akh, tmh, warp == 6 ? 2 : warp - 2, lane);
            named_bar_sync(kBarStep, kGroup);

            // ---------------- S2: D^T = (beta X)^T T^T  (mma.sync; T lower triangular: k-blocks <= qw/2)
            {
                const int mt = warp & 1;
#pragma unroll
                for (int jq = 0; jq < 2; ++jq) {
                    const int qw = (warp >> 1) + 4 * jq, rblk = qw >> 1;
                    float dk[4][4];   // one accumulator per k-block (no chained mma)
                    const int brow = (8 * qw + (lane & 7)) * LD64 + (((lane >> 3) & 1) << 3);
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks) {
                        dk[ks][0] = dk[ks][1] = dk[ks][2] = dk[ks][3] = 0.f;
                        if (ks <= rblk) {
                            uint32_t af[4], bt[2];
                            ldsm_x4(smem_u32(xt + a_off(lane, 16 * mt, 16 * ks, LD64)), af[0], af[1], af[2], af[3]);
                            ldsm_x2(smem_u32(tmh + brow + 16 * ks), bt[0], bt[1]);
                            mma16816(dk[ks], af, bt[0], bt[1]);
                        }
                    }
                    float dacc[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) dacc[e] = (dk[0][e] + dk[1][e]) + (dk[2][e] + dk[3][e]);
                    const int r = 8 * qw + 2 * tig;
                    const int v0 = 16 * mt + g8;
                    *reinterpret_cast<uint32_t *>(dt + sw128(v0, r, VT)) = pack_h2(dacc[0], dacc[1]);
                    *reinterpret_cast<uint32_t *>(dt + sw128(v0 + 8, r, VT)) = pack_h2(dacc[2], dacc[3]);
                }
            }
            fence_proxy_async_smem();
            named_bar_sync(kBarStep, kGroup);

            // ---------------- MMA S3: h += K^^T D ; D1[64..127] += A_qk D  (one tcgen05 batch)
            if (tid == 0) {
                tc_fence_after();
#pragma unroll
                for (int ks = 0; ks < C / 16; ++ks)
                    umma_f16(tH, sw128_kdesc(smem_u32(kht_s(s)), ks, KD), sw128_kdesc(smem_u32(dt), ks, VT),
                             kIdescM128N32, 1u);
                // A = [A_kk (rows 0..63, lands in the consumed X rows); A_qk (rows 64..127)]
#pragma unroll
                for (int ks = 0; ks < C / 16; ++ks)
                    umma_f16(tD1, sw128_kdesc(smem_u32(akh_s(s)), ks, 2 * C), sw128_kdesc(smem_u32(dt), ks, VT),
                             kIdescM128N32, 1u);
                umma_commit(bar(Bar::s3));
            }
            if (!mbar_wait(bar(Bar::s3), par)) failed = true;
            tc_fence_after();
            if (warp & 2) {   // rows 64..127 of D1: o (warps 2, 3, 6, 7)
                const int r = 32 * (warp & 1) + lane, half = warp >> 2;
                float ov[16];
                tmem_ld16(tD1 + lane_off + 16 * half, ov);
                if (r < len) store_row16(out + ((t0 + r) * H + h) * VD + vt * VT + 16 * half, ov, a.scale);
            }
            tc_fence_before();
            // slot s and the step buffers are consumed
            if (bar_red_or(kBarStep, kGroup, failed)) { failed = true; break; }
            if (tid == 0) mbar_arrive(bar(Bar::free0 + s));
        }
        if (failed) {   // MMAs still in flight get one more bounded wait
            mbar_wait(bar(Bar::s1), ci & 1);
            mbar_wait(bar(Bar::s3), ci & 1);
        }
        if (fin) {   // error marker: NaN state
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
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" :: "r"(tmem), "r"(128) : "memory");
    }
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
