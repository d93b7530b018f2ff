// kda_prefill_rr.cu -- chunked KDA prefill with the per-chunk operands built once per
// head and shared by the four value-tile CTAs of a thread-block cluster.
//
// The computation is the chunked prompt path of vllm.cpp PR #110 ("chunk_kda prefill
// AOT port", commit description) in the same algebra and precision as the fused
// kernel of kda_prefill_tc.cu (see its header):
//     G = log2(e) cumsum(g);  [A_kk'; A_qk'] = [a_k; a_q] b^T;  T = (I + A_kk)^-1
//     X = beta (v - K~ h);  D = T X;  o = scale (Q~ h + A_qk D);  h <- Diag(2^G_last) h + K^^T D
// What differs is who builds the operands.  Everything except v and the state is the
// same for the four 32-column value tiles of a (sequence, head), so:
//
//   * one cluster of 4 CTAs (rank j = value tile j) walks the chunks of a (sequence,
//     head) work item; rank j BUILDS the operand record of chunks n = j (mod 4) --
//     gate cumsum, reference, fp16 factors [a_k; a_q] and K^^T, the A matrices
//     (tcgen05) and the whole triangular inverse T -- and writes it to a ring of 8
//     records per cluster in global memory (it stays in L2);
//   * every CTA receives each record in one of two shared-memory slots (one multicast
//     bulk copy from the builder to all four) and runs the serial state step of its
//     value tile on it (S1, X, S2 = T X, S3; a chunk's output rows are stored during the
//     next chunk's S1 / X phase, by warps that are otherwise idle then).
//
// Hand-offs (all waits bounded in time; a wait that runs out records KDA timeout status in
// the workspace header, drains this CTA's copies and MMAs in flight and ends the work):
//   slot_free[n % 8] (builder's CTA, count 4): each CTA arms its slot n % 2 for chunk n
//                    (expected bytes, its own v tile on TMA) and arrives remotely;
//   slot_full[s]     (each CTA): completed by the v tile and by the builder's ONE
//                    multicast bulk copy of record n from global memory into slot
//                    n % 2 of all four CTAs, issued once the record is written and
//                    every slot is armed;
//   the builder reuses ring entry n % 8 for chunk n + 8 once its own CTA has received
//   record n (the multicast read is then complete), seen through a shared counter.
// The clusters are persistent: cluster c takes work items c, c + G, ... (item = n H + h),
// so the ring needs G x 8 records whatever the number of sequences.
#include <atomic>
#include <cstring>

#include "kda_tc_common.cuh"

namespace kda {
namespace {

constexpr int kThreads = 512;   // 16 warps: state-step group (0..7), builder group (8..15)
constexpr int kGroup = 256;
constexpr int kBarBuild = 1;    // named barrier of the builder group
constexpr int kBarStep = 2;     // named barrier of the state-step group
constexpr int kRanks = kVTiles; // CTAs per cluster; rank j builds the chunks n = j (mod 4)
constexpr int kRing = 8;        // records per cluster in the global ring
constexpr int LDX = VT + 8;     // f16 row stride of beta X [64][32]: 80 B (conflict-free ldmatrix)

// Operand record of one chunk: the byte image of the shared-memory tiles the state step
// reads (SW128 tiles keep their swizzle at any 1024-byte aligned base).
struct Rec {
    static constexpr int aop = 0;                     // SW128 [a_k; a_q] 128 x 128 f16
    static constexpr int kht = aop + 2 * C * KD * 2;  // SW128 K^^T 128 (channel) x 64 (row)
    static constexpr int ta = kht + KD * C * 2;       // SW128 [T; A_qk] 128 x 64: the A of o += A_qk D
    static constexpr int beta = ta + 2 * C * C * 2;   // f32 [64] (0 past the sequence end)
    static constexpr int dec = beta + C * 4;          // f32 [128] 2^G_last
    static constexpr int pm = dec + KD * 4;           // f32 [128] 2^m
    static constexpr int bytes = pm + KD * 4;
};
static_assert(Rec::bytes % 16 == 0, "bulk copies move multiples of 16 bytes");
static_assert(Rec::bytes == kPrefillRrRecordBytes && kRing == kPrefillRrRing, "record ring size");
constexpr int kWsHeader = kPrefillRrHeaderBytes;   // workspace header: the device status word

// Failure reporting: every wait whose completion depends on another CTA or on the
// tensor pipe is bounded by the launch's wait limit; the clean-up waits after a failure
// have a fixed bound of their own (they wait only for work this CTA has started).
struct RrWait {
    int *status;
    unsigned long long wait_ns;
};
__device__ __forceinline__ uint64_t gtimer()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
__device__ __noinline__ void raise_timeout(const RrWait &w) { atomicExch(w.status, kStatusTimeout); }
__device__ __forceinline__ bool mbar_try_cta(uint32_t mbar, uint32_t parity)
{
    uint32_t done;
    asm volatile("{\n.reg .pred p;\nmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
                 "selp.u32 %0, 1, 0, p;\n}\n"
                 : "=r"(done) : "r"(mbar), "r"(parity) : "memory");
    return done != 0;
}
// one probe that suspends the thread for at most `hint_ns` while the phase is incomplete
__device__ __forceinline__ bool mbar_try_hint(uint32_t mbar, uint32_t parity, uint32_t hint_ns, bool cluster_scope)
{
    uint32_t done;
    if (cluster_scope)
        asm volatile("{\n.reg .pred p;\nmbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2, %3;\n"
                     "selp.u32 %0, 1, 0, p;\n}\n"
                     : "=r"(done) : "r"(mbar), "r"(parity), "r"(hint_ns) : "memory");
    else
        asm volatile("{\n.reg .pred p;\nmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n"
                     "selp.u32 %0, 1, 0, p;\n}\n"
                     : "=r"(done) : "r"(mbar), "r"(parity), "r"(hint_ns) : "memory");
    return done != 0;
}
// bounded by the wait limit (time); each probe suspends for at most the limit
__device__ bool wait_t(uint32_t mbar, uint32_t parity, const RrWait &w, bool cluster_scope = false)
{
    const uint32_t hint = w.wait_ns < 1000000ull ? (uint32_t)w.wait_ns : 1000000u;
    const uint64_t t0 = gtimer();
    for (;;) {
        if (mbar_try_hint(mbar, parity, hint, cluster_scope)) return true;
        if (gtimer() - t0 > w.wait_ns) { raise_timeout(w); return false; }
    }
}
// clean-up after a failure: a fixed bound
__device__ bool mbar_drain(uint32_t mbar, uint32_t parity)
{
    for (int i = 0; i < (1 << 22); ++i)
        if (mbar_try_cta(mbar, parity)) return true;
    return false;
}

// mbarriers
struct Bar { enum { slot_full = 0, slot_free = 2, a = slot_free + kRing, s1 = a + 1, s3 = s1 + 1,
                    raw = s3 + 1, count = raw + 1 }; };

// Shared memory map (byte offsets)
struct Smem {
    static constexpr int slot_v = (Rec::bytes + 1023) / 1024 * 1024;   // v tile bf16 [64][32]
    static constexpr int slot_bytes = slot_v + C * VT * 2;            // record + v tile
    static constexpr int ht = 2 * slot_bytes;                // SW128 (2^m h)^T f16 32 x 128
    static constexpr int xs = ht;                            // f16 beta X [64][LDX] once S1 is done
    static constexpr int dt = ht + VT * KD * 2;              // SW128 D^T f16 32 x 64
    static constexpr int st_aop = dt + VT * C * 2;           // builder: SW128 [a_k; a_q]; until P2
                                                             // the chunk's raw g tile (TMA)
    static constexpr int st_bk = st_aop + 2 * C * KD * 2;    // builder: SW128 b 64 x 128; until P2
                                                             // the chunk's raw k tile (TMA)
    static constexpr int tm = st_bk;                         // builder: f16 T [64][LD64] (b is dead)
    static constexpr int st_tw = st_bk + C * KD * 2;         // builder: SW128 T 64 x 64 (record ta rows 0..63);
                                                             // with st_akk, until P2 the raw q tile (TMA)
    static constexpr int st_akk = st_tw + C * C * 2;         // builder: SW128 A_kk 64 x 64
    static constexpr int st_vec = st_akk + C * C * 2;        // builder: beta, dec, pm (record layout)
    static constexpr int st_kht = st_tw;                     // builder: SW128 K^^T 128 x 64 over T and
                                                             // A_kk, from P2 until its bulk store read it
    static constexpr int st_aqk = st_tw;                     // builder: SW128 A_qk 64 x 64 from the A
                                                             // epilogue until its bulk store read it
    static constexpr int bars = st_vec + (Rec::bytes - Rec::beta);
    static constexpr int consumed = bars + Bar::count * 8;   // i64: chunks whose record this CTA has
    static constexpr int tmem = consumed + 8;                // u32
    static constexpr int flag = tmem + 4;
    static constexpr int nred = (flag + 4 + 15) / 16 * 16;  // builder: f32 [8 warps][32] row |x|^2 sums
    static constexpr int nscl = nred + 8 * 32 * 4;           // builder: f32 [4][q 16 | k 16] 1/|x| per row
    static constexpr int tot = nscl + 4 * 32 * 4;            // builder: f32 [4][128] group sums
    static constexpr int first = tot + 4 * KD * 4;           // builder: f32 [128] G of row 0
    static constexpr int total = first + KD * 4;
};
static_assert(Smem::total <= 232448, "shared memory budget");
static_assert(Smem::slot_bytes % 1024 == 0 && Smem::ht % 1024 == 0 && Smem::dt % 1024 == 0 &&
              Smem::st_aop % 1024 == 0 && Smem::st_bk % 1024 == 0 && Smem::st_tw % 1024 == 0 &&
              Smem::st_akk % 1024 == 0, "SW128 tiles need 1024-byte alignment");
static_assert(C * LD64 * 2 <= C * KD * 2, "the padded T fits in the b space");
static_assert(Smem::st_akk == Smem::st_tw + C * C * 2 && 2 * C * C * 2 == C * KD * 2,
              "the raw q tile spans the T and A_kk staging");
static_assert(C * LDX * 2 <= VT * KD * 2, "beta X fits in the h^T space");

struct RrMaps {
    CUtensorMap q, k, g;   // box 128 channels x 1 head x 64 tokens (L2 prefetch of a builder's next chunk)
    CUtensorMap beta;      // [T, H] fp32, box 4 heads x 64 tokens (L2 prefetch; H % 4 == 0 only)
    CUtensorMap v;         // box 32 columns x 1 head x 64 tokens
    int beta_map;          // 0: no beta prefetch
};

// ------------------------------------------------------------------ cluster helpers
__device__ __forceinline__ uint32_t cluster_ctarank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;\n" : "=r"(r));
    return r;
}

// every thread of every CTA of the cluster (release / acquire)
__device__ __forceinline__ void cluster_sync_all()
{
    asm volatile("barrier.cluster.arrive.release.aligned;\nbarrier.cluster.wait.acquire.aligned;\n"
                 ::: "memory");
}

// relaxed arrive on a peer's mbarrier: it only reports that this CTA has finished with
// a buffer (every read of it has returned and been consumed before the arrive)
__device__ __forceinline__ void mbar_arrive_remote_relaxed(uint32_t mbar, uint32_t rank)
{
    asm volatile("{\n.reg .b32 ra;\nmapa.shared::cluster.u32 ra, %0, %1;\n"
                 "mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [ra];\n}\n"
                 :: "r"(mbar), "r"(rank) : "memory");
}

// TMA prefetch of a tile into L2
__device__ __forceinline__ void tma_prefetch_3d(const CUtensorMap *map, int x, int y, int z)
{
    asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];\n"
                 :: "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z) : "memory");
}
__device__ __forceinline__ void tma_prefetch_2d(const CUtensorMap *map, int x, int y)
{
    asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];\n"
                 :: "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y) : "memory");
}

__device__ __forceinline__ void fence_proxy_async_global() { asm volatile("fence.proxy.async.global;\n" ::: "memory"); }

// 1-D bulk copy global -> shared of every CTA in `mask` (same offset), completing on
// each destination's mbarrier at the same offset
__device__ __forceinline__ void bulk_g2s_multicast(uint32_t dst, const void *src, uint32_t bytes,
                                                   uint32_t mbar, uint16_t mask)
{
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.multicast::cluster "
                 "[%0], [%1], %2, [%3], %4;\n"
                 :: "r"(dst), "l"(src), "r"(bytes), "r"(mbar), "h"(mask) : "memory");
}
// 1-D bulk copy shared -> global (bulk async-group)
__device__ __forceinline__ void bulk_s2g(void *dst, uint32_t src, uint32_t bytes)
{
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;\n"
                 :: "l"(dst), "r"(src), "r"(bytes) : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;\n" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;\n" ::: "memory"); }
// the sources of every committed bulk store have been read (shared memory is reusable)
__device__ __forceinline__ void bulk_wait_read_all() { asm volatile("cp.async.bulk.wait_group.read 0;\n" ::: "memory"); }

// ------------------------------------------------------------------ work walk
// The chunks of a cluster: work items w = c, c + G, ... (item w = sequence w / H, head
// w % H), each cut into 64-token chunks; items with no tokens have no chunks.
struct Cursor {
    int64_t w, bos, eos, t0;
};

// first chunk of the first non-empty item at or after w; false when there is none
__device__ __forceinline__ bool cursor_seek(Cursor &c, const PrefillArgs &a, int64_t w, int64_t G)
{
    const int64_t NH = (int64_t)a.num_seqs * a.num_heads;
    for (; w < NH; w += G) {
        const int64_t n = w / a.num_heads;
        int64_t b, e;
        clamp_range(a.total_tokens, a.cu_seqlens[n], a.cu_seqlens[n + 1], b, e);
        if (b < e) {
            c.w = w; c.bos = b; c.eos = e; c.t0 = b;
            return true;
        }
    }
    c.w = NH;
    return false;
}

__device__ __forceinline__ bool cursor_next(Cursor &c, const PrefillArgs &a, int64_t G)
{
    c.t0 += C;
    if (c.t0 < c.eos) return true;
    return cursor_seek(c, a, c.w + G, G);
}

// Exact-exponential A_kk (to shared memory), A_qk and K^^T (to the record in global
// memory) for a chunk whose gate span leaves the fp16 fast path: one exponential per
// pair and channel.  G is the chunk's exp2-space cumsum, fp32 [64][128], in global scratch.
// With the in-kernel L2 normalisation, nscl holds the rows' 1/|q| and 1/|k| (else null).
__device__ __forceinline__ float row_scale(const float *nscl, int r, int is_k)
{
    return nscl ? nscl[(r >> 4) * 32 + 16 * is_k + (r & 15)] : 1.f;
}
__device__ __noinline__ void exact_pairs(const PrefillArgs &a, int64_t t0, int len, int h,
                                         const float *G, const float *bs, __half *akk,
                                         unsigned char *aqk_g, unsigned char *kht_g, int gtid,
                                         const float *nscl)
{
    const int H = a.num_heads;
    const __nv_bfloat16 *kk = static_cast<const __nv_bfloat16 *>(a.k);
    const __nv_bfloat16 *qq = static_cast<const __nv_bfloat16 *>(a.q);
    for (int p = gtid; p < C * C; p += kGroup) {
        const int r = p >> 6, i = p & 63;
        float sk = 0.f, sq = 0.f;
        if (i <= r && r < len) {
            const __nv_bfloat16 *kr = kk + ((t0 + r) * H + h) * KD, *ki = kk + ((t0 + i) * H + h) * KD;
            const __nv_bfloat16 *qr = qq + ((t0 + r) * H + h) * KD;
            for (int c = 0; c < KD; ++c) {
                const float kic = __bfloat162float(ki[c]) * exp2f(G[r * KD + c] - G[i * KD + c]);
                sk += __bfloat162float(kr[c]) * kic;
                sq += __bfloat162float(qr[c]) * kic;
            }
            const float si = row_scale(nscl, i, 1);
            sk *= si * row_scale(nscl, r, 1);
            sq *= si * row_scale(nscl, r, 0);
        }
        akk[sw128(r, i, C)] = __float2half_rn(i < r ? bs[r] * sk : 0.f);
        reinterpret_cast<__half *>(aqk_g)[sw128(r, i, C)] = __float2half_rn(i <= r ? sq : 0.f);
    }
    // K^^T = (k 2^(G_last - G))^T, one exponential per element (its fast-path factors
    // can leave the fp32 range at such spans); rows past the end have G = G_last
    for (int e = gtid; e < C * KD; e += kGroup) {
        const int r = e >> 7, c = e & 127;
        const float kv = r < len ? __bfloat162float(kk[((t0 + r) * H + h) * KD + c]) * row_scale(nscl, r, 1) : 0.f;
        reinterpret_cast<__half *>(kht_g)[sw128(c, r, KD)] =
            __float2half_rn(kv * exp2f(G[(C - 1) * KD + c] - G[r * KD + c]));
    }
}

template <typename Tout, bool kL2>
__global__ void __cluster_dims__(kRanks, 1, 1) __launch_bounds__(kThreads, 1)
kda_prefill_rr_kernel(const PrefillArgs a, const __grid_constant__ RrMaps maps,
                      unsigned char *__restrict__ ws, int G, const RrWait wt)
{
    extern __shared__ __align__(1024) unsigned char sm[];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int rank = (int)cluster_ctarank();   // = value tile
    const int vt = rank;
    const int64_t cid = blockIdx.x / kRanks;
    const int H = a.num_heads;
    const int64_t NH = (int64_t)a.num_seqs * H;
    auto bar = [&](int b) { return smem_u32(sm + Smem::bars + 8 * b); };
    auto slot = [&](int s) { return sm + s * Smem::slot_bytes; };
    auto record = [&](int64_t ci) { return ws + ((int64_t)cid * kRing + (ci % kRing)) * Rec::bytes; };

    // ---- tensor memory (256 columns: per chunk parity p, [64 p, 64 p + 32) and
    //      [64 p + 32, 64 p + 64) the step accumulator D1 in two K halves (issued by two
    //      threads; the output rows of chunk n are read during chunk n + 1), [128, 160)
    //      the state h^T with lane = key channel, column = value, [192, 256) the A matrices)
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n"
                     :: "r"(smem_u32(sm + Smem::tmem)), "r"(256) : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n" ::: "memory");
    }
    if (tid == 0) {
        for (int b = 0; b < Bar::count; ++b)
            mbar_init(bar(b), (b >= Bar::slot_free && b < Bar::slot_free + kRing) ? kRanks
                              : (b == Bar::s1 || b == Bar::s3) ? 2 : 1);
        *reinterpret_cast<volatile int64_t *>(sm + Smem::consumed) = 0;
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync_all();   // every CTA's barriers exist before any remote arrival
    tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(sm + Smem::tmem);
    const uint32_t tH = tmem + 128, tDA = tmem + 192;
    const uint32_t lane_off = (uint32_t)(32 * (warp & 3)) << 16;   // TMEM lane quadrant of this warp
    bool failed = false;

    if (warp >= 8) {
        // =====================================================================
        // Builder group (warps 8..15): the records of chunks n = rank (mod 4).
        // =====================================================================
        const int gtid = tid - kGroup;
        __half *aop = reinterpret_cast<__half *>(sm + Smem::st_aop);
        __half *bop = reinterpret_cast<__half *>(sm + Smem::st_bk);
        __half *tmh = reinterpret_cast<__half *>(sm + Smem::tm);
        __half *akk = reinterpret_cast<__half *>(sm + Smem::st_akk);
        __half *tw = reinterpret_cast<__half *>(sm + Smem::st_tw);
        float *tot = reinterpret_cast<float *>(sm + Smem::tot);
        float *first = reinterpret_cast<float *>(sm + Smem::first);
        float *bs = reinterpret_cast<float *>(sm + Smem::st_vec);
        float *decs = reinterpret_cast<float *>(sm + Smem::st_vec + (Rec::dec - Rec::beta));
        float *pms = reinterpret_cast<float *>(sm + Smem::st_vec + (Rec::pm - Rec::beta));
        volatile int *flag = reinterpret_cast<volatile int *>(sm + Smem::flag);
        float *nred = reinterpret_cast<float *>(sm + Smem::nred);
        float *nscl = reinterpret_cast<float *>(sm + Smem::nscl);
        constexpr bool l2 = kL2;   // in-kernel L2 normalisation of the q and k rows
        uint32_t a_parity = 0;

        // q, k, g tiles of chunk `ahead` chunks after the cursor's, prefetched into L2 (only
        // this CTA reads them, so they would otherwise come from DRAM with full latency)
        auto prefetch = [&](const Cursor &from, int ahead) {
            Cursor c = from;
            bool ok = true;
            for (int i = 0; i < ahead && ok; ++i) ok = cursor_next(c, a, G);
            if (ok) {
                const int hh = (int)(c.w % H), z = (int)c.t0;
                tma_prefetch_3d(&maps.q, 0, hh, z);
                tma_prefetch_3d(&maps.k, 0, hh, z);
                tma_prefetch_3d(&maps.g, 0, hh, z);
                if (maps.beta_map) tma_prefetch_2d(&maps.beta, hh & ~3, z);
            }
        };
        // The raw g, k and q tiles (64 tokens x 128 channels; g fp32, k and q bf16) of the
        // chunk `ahead` chunks after the cursor's, by TMA into staging areas that are free
        // from the end of one record until P2 of the next (g: [a_k; a_q]; k: b; q: T and
        // A_kk), completing on one barrier: the builder's P1 then reads shared memory only,
        // and the loads of its next chunk run while it finishes this one (thread 0 only)
        uint32_t raw_parity = 0;
        bool raw_pending = false;
        auto load_raw = [&](const Cursor &from, int ahead) {
            Cursor c = from;
            bool ok = true;
            for (int i = 0; i < ahead && ok; ++i) ok = cursor_next(c, a, G);
            if (ok) {
                const int hh = (int)(c.w % H), z = (int)c.t0;
                const uint32_t mb = bar(Bar::raw);
                fence_proxy_async_smem();   // earlier generic accesses of the staging come first
                mbar_arrive_expect_tx(mb, C * KD * (4 + 2 + 2));
                tma_load_3d(smem_u32(sm + Smem::st_aop), &maps.g, 0, hh, z, mb);
                tma_load_3d(smem_u32(sm + Smem::st_bk), &maps.k, 0, hh, z, mb);
                tma_load_3d(smem_u32(sm + Smem::st_tw), &maps.q, 0, hh, z, mb);
            }
            raw_pending = ok;
        };
        Cursor pc;
        bool have = cursor_seek(pc, a, cid, G);
        if (gtid == 0 && have) {
            prefetch(pc, rank);
            load_raw(pc, rank);
        }
        for (int64_t ci = 0; have; ++ci, have = cursor_next(pc, a, G)) {
            if ((int)(ci % kRanks) != rank) continue;
            const int64_t t0 = pc.t0;
            const int len = (int)((pc.eos - t0) < C ? (pc.eos - t0) : C);
            const int h = (int)(pc.w % H);
            unsigned char *rec = record(ci);
            // ring entry ci % 8 is free once this CTA has received record ci - 8: the
            // multicast that read it has then finished reading
            if (gtid == 0 && ci >= kRing) {
                const volatile int64_t *consumed = reinterpret_cast<const volatile int64_t *>(sm + Smem::consumed);
                const uint64_t tw = gtimer();
                while (*consumed <= ci - kRing) {
                    __nanosleep(64);
                    if (gtimer() - tw > wt.wait_ns) { raise_timeout(wt); failed = true; break; }
                }
            }
            if (bar_red_or(kBarBuild, kGroup, failed)) { failed = true; break; }
            if (gtid == 0) *flag = 0;

            // ---------------- P1: gate cumsum in exp2 space; thread = (channel pair, 16-row group E)
            const int pcp = gtid & 63, pE = gtid >> 6, pc0 = 2 * pcp;
            // this thread's 16 rows of g, k and q (channels pc0, pc0 + 1) from the raw tiles
            // (rows past the sequence's end read as zero)
            if (wait_t(bar(Bar::raw), raw_parity, wt)) {
                raw_parity ^= 1u;
                if (gtid == 0) raw_pending = false;
            } else {
                failed = true;
            }
            float2 gx[16];
            uint32_t kq[16], qq[16];   // bf16 pairs
            {
                const float *gsm = reinterpret_cast<const float *>(sm + Smem::st_aop);
                const uint32_t *ksm = reinterpret_cast<const uint32_t *>(sm + Smem::st_bk);
                const uint32_t *qsm = reinterpret_cast<const uint32_t *>(sm + Smem::st_tw);
#pragma unroll
                for (int u = 0; u < 16; ++u) {
                    const int r = 16 * pE + u;
                    gx[u] = r < len ? *reinterpret_cast<const float2 *>(gsm + r * KD + pc0) : make_float2(0.f, 0.f);
                    kq[u] = r < len ? ksm[(r * KD + pc0) >> 1] : 0u;
                    qq[u] = r < len ? qsm[(r * KD + pc0) >> 1] : 0u;
                }
            }
#pragma unroll
            for (int u = 0; u < 16; ++u) gx[u] = make_float2(gx[u].x * kLog2e, gx[u].y * kLog2e);
#pragma unroll
            for (int u = 1; u < 16; ++u) { gx[u].x += gx[u - 1].x; gx[u].y += gx[u - 1].y; }
            *reinterpret_cast<float2 *>(tot + pE * KD + pc0) = gx[15];
            if (pE == 0) *reinterpret_cast<float2 *>(first + pc0) = gx[0];
            if (gtid < C) bs[gtid] = gtid < len ? a.beta[(t0 + gtid) * H + h] : 0.f;
            if (l2) {
                // |q_r|^2 (values 0..15) and |k_r|^2 (16..31) of this thread's rows over its two
                // channels, reduced over the warp so that lane L ends with value L summed over
                // the warp's 64 channels (halving exchanges, 31 shuffles)
                float nv[32];
#pragma unroll
                for (int u = 0; u < 16; ++u) {
                    const float2 qv = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&qq[u]));
                    const float2 kv = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&kq[u]));
                    nv[u] = qv.x * qv.x + qv.y * qv.y;
                    nv[16 + u] = kv.x * kv.x + kv.y * kv.y;
                }
#pragma unroll
                for (int w = 16; w >= 1; w >>= 1) {
                    const bool up = (lane & w) != 0;
#pragma unroll
                    for (int i = 0; i < w; ++i) {
                        const float send = up ? nv[i] : nv[i + w];
                        const float keep = up ? nv[i + w] : nv[i];
                        nv[i] = keep + __shfl_xor_sync(0xffffffffu, send, w);
                    }
                }
                nred[(gtid >> 5) * 32 + lane] = nv[0];
            }
            named_bar_sync(kBarBuild, kGroup);
            if (l2) {   // the two warps of a 16-row group hold the halves of its 128 channels
                const int gw = gtid >> 5;
                if ((gw & 1) == 0)
                    nscl[(gw >> 1) * 32 + lane] = rsqrtf(nred[gw * 32 + lane] + nred[(gw + 1) * 32 + lane] + kQkL2NormEps);
                named_bar_sync(kBarBuild, kGroup);
            }

            // ---------------- P2: reference, factors, fp16 operands; K^^T straight to the record
            float2 pre = make_float2(0.f, 0.f), run = make_float2(0.f, 0.f);
#pragma unroll
            for (int E = 0; E < 4; ++E) {
                const float2 t = *reinterpret_cast<const float2 *>(tot + E * KD + pc0);
                if (E == pE) pre = run;
                run.x += t.x; run.y += t.y;
            }
            const float2 glast = run, g0 = *reinterpret_cast<const float2 *>(first + pc0);
            // reference: the midpoint of the first and last row's G (the midrange when the
            // gate is a decay), capped so that no factor 2^(G - m) exceeds 2^8 then
            const float mx_ = fmaxf(0.5f * (g0.x + glast.x), g0.x - 0.5f * kSpanMax);
            const float my_ = fmaxf(0.5f * (g0.y + glast.y), g0.y - 0.5f * kSpanMax);
            if (pE == 0) {
                *reinterpret_cast<float2 *>(pms + pc0) = make_float2(exp2f(mx_), exp2f(my_));
                *reinterpret_cast<float2 *>(decs + pc0) = make_float2(exp2f(glast.x), exp2f(glast.y));
            }
            const float fx = exp2f(glast.x - mx_), fy = exp2f(glast.y - my_);   // K^ = b 2^(G_last - m)
            const float bx = pre.x - mx_, by = pre.y - my_;       // G_r - m = gx + b
            named_bar_sync(kBarBuild, kGroup);   // the group sums (in the b space) are read
            float amax = 0.f;
#pragma unroll
            for (int hb = 0; hb < 2; ++hb) {
                float khx[8], khy[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const int r = 16 * pE + 8 * hb + u;
                    const float xx = gx[8 * hb + u].x + bx, xy = gx[8 * hb + u].y + by;   // G_r - m
                    amax = fmaxf(amax, fmaxf(fabsf(xx), fabsf(xy)));
                    const float ex = ex2_approx(xx), ey = ex2_approx(xy);
                    const float ix = rcp_approx(ex), iy = rcp_approx(ey);
                    float2 kv = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&kq[8 * hb + u]));
                    float2 qv = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&qq[8 * hb + u]));
                    if (l2) {
                        const float sq = nscl[pE * 32 + 8 * hb + u], sk = nscl[pE * 32 + 16 + 8 * hb + u];
                        qv.x *= sq; qv.y *= sq; kv.x *= sk; kv.y *= sk;
                    }
                    *reinterpret_cast<uint32_t *>(aop + sw128(r, pc0, 2 * C)) = pack_h2(kv.x * ex, kv.y * ey);
                    *reinterpret_cast<uint32_t *>(aop + sw128(C + r, pc0, 2 * C)) = pack_h2(qv.x * ex, qv.y * ey);
                    const float b0 = kv.x * ix, b1 = kv.y * iy;
                    *reinterpret_cast<uint32_t *>(bop + sw128(r, pc0, C)) = pack_h2(b0, b1);
                    khx[u] = b0 * fx;
                    khy[u] = b1 * fy;
                }
                // K^^T: these eight rows are one 16-byte chunk of key-channel rows pc0, pc0 + 1
                // (staged in shared memory; one bulk store moves the tile to the record)
                const int r0 = 16 * pE + 8 * hb;
                __half *kh = reinterpret_cast<__half *>(sm + Smem::st_kht);
                *reinterpret_cast<uint4 *>(kh + sw128(pc0, r0, KD)) =
                    make_uint4(pack_h2(khx[0], khx[1]), pack_h2(khx[2], khx[3]),
                               pack_h2(khx[4], khx[5]), pack_h2(khx[6], khx[7]));
                *reinterpret_cast<uint4 *>(kh + sw128(pc0 + 1, r0, KD)) =
                    make_uint4(pack_h2(khy[0], khy[1]), pack_h2(khy[2], khy[3]),
                               pack_h2(khy[4], khy[5]), pack_h2(khy[6], khy[7]));
            }
            // fast path: every factor 2^(G_r - m) within [2^-8, 2^8]
            if (__any_sync(0xffffffffu, !(amax <= 0.5f * kSpanMax)) && lane == 0) *flag = 1;
            fence_proxy_async_smem();   // the operands are read by tcgen05 and the bulk copy
            named_bar_sync(kBarBuild, kGroup);
            const bool exact_path = *flag != 0;
            // the next own chunk's tiles into L2 while the A MMA runs (issued here, off thread
            // 0's path: at the end of a record its TMA queue holds the record's copies); the
            // raw-tile loads of that chunk, at the end of this record, then find them there
            if (gtid == 32) prefetch(pc, kRanks);
            unsigned char *aqk_g = rec + Rec::ta + C * C * 2;   // rows 64..127 of [T; A_qk]

            if (!exact_path) {
                // ---------------- MMA A: [A_kk'; A_qk'] = [a_k; a_q] b^T
                if (gtid == 0) {
                    bulk_s2g(rec + Rec::kht, smem_u32(sm + Smem::st_kht), KD * C * 2);   // K^^T
                    bulk_commit();
                    tc_fence_after();
#pragma unroll
                    for (int ks = 0; ks < KD / 16; ++ks)
                        umma_f16(tDA, sw128_kdesc(smem_u32(aop), ks, 2 * C), sw128_kdesc(smem_u32(bop), ks, C),
                                 kIdescM128N64, ks > 0);
                    umma_commit(bar(Bar::a));
                    bulk_wait_read_all();   // the K^^T staging is read: A_kk and A_qk may go there
                }
                // ---------------- A epilogue: masked, beta-scaled A_kk and A_qk (both staged)
                //   lanes 0..63 A_kk, 64..127 A_qk; warp w: lane quadrant w % 4, columns [32 ((w / 4) % 2), +32)
                if (!wait_t(bar(Bar::a), a_parity, wt)) failed = true;
                a_parity ^= 1u;
                named_bar_sync(kBarBuild, kGroup);
                tc_fence_after();
                const int c0 = 32 * ((warp >> 2) & 1), rg = 32 * (warp & 3) + lane;
                float av[2][16];
                tmem_ld16(tDA + lane_off + c0, av[0]);
                tmem_ld16(tDA + lane_off + c0 + 16, av[1]);
                const bool kk = rg < C;
                const int r = kk ? rg : rg - C;
                const float sb = kk ? bs[r] : 1.f;
                const int lim = kk ? r : r + 1;   // columns i < lim are kept
                __half *dst = kk ? akk : reinterpret_cast<__half *>(sm + Smem::st_aqk);
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
                // ---------------- exact path: G (fp32) to the record's [a_k; a_q] area as scratch
                float *Gs = reinterpret_cast<float *>(rec + Rec::aop);
#pragma unroll
                for (int u = 0; u < 16; ++u) {
                    const int r = 16 * pE + u;
                    *reinterpret_cast<float2 *>(Gs + r * KD + pc0) = make_float2(gx[u].x + pre.x, gx[u].y + pre.y);
                }
                named_bar_sync(kBarBuild, kGroup);
                exact_pairs(a, t0, len, h, Gs, bs, akk, aqk_g, rec + Rec::kht, gtid, l2 ? nscl : nullptr);
            }
            if (!exact_path) fence_proxy_async_smem();   // A_qk is read by the bulk copy
            named_bar_sync(kBarBuild, kGroup);   // A_kk complete; the G scratch is no longer read
            if (gtid == 0) {   // [a_k; a_q] (and on the fast path A_qk) to the record
                fence_proxy_async_global();
                bulk_s2g(rec + Rec::aop, smem_u32(aop), 2 * C * KD * 2);
                if (!exact_path) bulk_s2g(aqk_g, smem_u32(sm + Smem::st_aqk), C * C * 2);
                bulk_commit();
            }

            // ---------------- T = (I + A_kk)^-1: the diagonal blocks, then the column blocks
            if (warp == 8 || warp == 9) invert_diag_blocks(akk, tmh, warp - 8, lane);
            named_bar_sync(kBarBuild, kGroup);
            if (warp == 10) solve_column_block(akk, tmh, 0, lane);
            else if (warp == 11) solve_column_block(akk, tmh, 1, lane);
            else if (warp == 12) solve_column_block(akk, tmh, 2, lane);
            if (gtid == 0) bulk_wait_read_all();   // the A_qk staging is read: T may go there
            named_bar_sync(kBarBuild, kGroup);
            // T (zeros above its diagonal blocks) -> SW128 rows 0..63 of [T; A_qk]
            for (int e = gtid; e < C * C / 8; e += kGroup) {
                const int r = e >> 3, j = e & 7;
                const uint4 x = (j >> 1) > (r >> 4) ? make_uint4(0, 0, 0, 0)
                                                    : *reinterpret_cast<const uint4 *>(tmh + r * LD64 + 8 * j);
                *reinterpret_cast<uint4 *>(tw + sw128(r, 8 * j, C)) = x;
            }
            fence_proxy_async_smem();   // T and beta / dec / pm are read by the bulk copy
            fence_proxy_async_global(); // K^^T and A_qk went to the record by generic stores
            named_bar_sync(kBarBuild, kGroup);
            if (gtid == 0) {
                bulk_s2g(rec + Rec::ta, smem_u32(tw), C * C * 2);
                bulk_s2g(rec + Rec::beta, smem_u32(bs), Rec::bytes - Rec::beta);
                bulk_commit();
                bulk_wait_all();            // the record is in global memory; the staging is free
                fence_proxy_async_global();
                // every CTA has armed slot ci % 2 for this chunk: one copy to all four
                if (wait_t(bar(Bar::slot_free + (int)(ci % kRing)), (uint32_t)((ci >> 3) & 1), wt, true))
                    bulk_g2s_multicast(smem_u32(slot((int)(ci & 1))), rec, Rec::bytes,
                                       bar(Bar::slot_full + (int)(ci & 1)), (uint16_t)((1u << kRanks) - 1));
                else
                    failed = true;
                if (!failed) load_raw(pc, kRanks);   // the raw tiles of this builder's next chunk
            }
        }
        if (failed) mbar_drain(bar(Bar::a), a_parity);   // an MMA still in flight
        if (raw_pending) mbar_drain(bar(Bar::raw), raw_parity);   // raw tiles still in flight
    } else {
        // =====================================================================
        // State-step group (warps 0..7): the chunks of every work item of this cluster
        // in order, on the records received in slot n % 2.  Thread 64 also arms the
        // slots, two chunks ahead.  Warp w reaches TMEM lanes 32 (w % 4) ..; state roles:
        // key channel sc = 32 (w % 4) + lane, value columns [16 hc, +16).
        // =====================================================================
        const int sc = 32 * (warp & 3) + lane;
        const int hc = (warp >> 2) & 1;
        __half *ht = reinterpret_cast<__half *>(sm + Smem::ht);
        __half *dt = reinterpret_cast<__half *>(sm + Smem::dt);
        __half *xs = reinterpret_cast<__half *>(sm + Smem::xs);
        Tout *out = static_cast<Tout *>(a.out);

        // Arming slot lci % 2 for chunk lci (thread kArmer): the local part -- expected
        // bytes and the TMA of this CTA's v tile -- once the slot's v region is free, then
        // the arrival on the chunk's builder's slot_free barrier once every read of the
        // slot is done (the builder's multicast overwrites it).
        constexpr int kArmer = 64;   // warp 2: idle while S3 runs
        Cursor lc{0, 0, 0, 0};
        int64_t lci = 0;
        bool lhave = false;
        auto arm_local = [&]() {
            const int s = (int)(lci & 1);
            fence_proxy_async_smem();     // earlier generic reads of the slot come first
            const uint32_t mb = bar(Bar::slot_full + s);
            mbar_arrive_expect_tx(mb, Rec::bytes + C * VT * 2);
            tma_load_3d(smem_u32(slot(s) + Smem::slot_v), &maps.v, vt * VT, (int)(lc.w % H), (int)lc.t0, mb);
        };
        auto arm_remote = [&]() {
            mbar_arrive_remote_relaxed(bar(Bar::slot_free + (int)(lci % kRing)), (uint32_t)(lci % kRanks));
            ++lci;
            lhave = cursor_next(lc, a, G);
        };
        if (tid == kArmer) {
            lhave = cursor_seek(lc, a, cid, G);
            for (int i = 0; i < 2 && lhave; ++i) { arm_local(); arm_remote(); }
        }
        // output rows of the previous chunk (warps 2, 3, 6, 7), stored during the next
        // chunk's S1 / X phase, when those warps are otherwise idle
        bool pend = false;
        int pend_par = 0, pend_len = 0, pend_h = 0;
        int64_t pend_t0 = 0;
        auto flush_o = [&]() {
            if (!pend) return;
            tc_fence_after();
            const int r = 32 * (warp & 1) + lane, half = warp >> 2;
            const uint32_t d1 = tmem + 64 * pend_par;
            float ov[16], ob[16];
            tmem_ld16(d1 + lane_off + 16 * half, ov);
            tmem_ld16(d1 + 32 + lane_off + 16 * half, ob);
#pragma unroll
            for (int v = 0; v < 16; ++v) ov[v] += ob[v];
            if (r < pend_len)
                store_row16(out + ((pend_t0 + r) * H + pend_h) * VD + vt * VT + 16 * half, ov, a.scale);
            tc_fence_before();
            pend = false;
        };

        int64_t ci = 0;
        bool gfail = false;   // group-uniform: set only from barrier reductions
        for (int64_t w = cid; w < NH && !gfail; w += G) {
            const int64_t n = w / H;
            const int h = (int)(w % H);
            int64_t bos, eos;
            clamp_range(a.total_tokens, a.cu_seqlens[n], a.cu_seqlens[n + 1], bos, eos);
            const float *init;
            float *fin;
            prefill_state_ptrs(a, n, h, init, fin);
            {   // initial state -> tensor memory
                float hv[16];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const float4 x = init
                        ? *reinterpret_cast<const float4 *>(init + (int64_t)sc * VD + vt * VT + 16 * hc + 4 * j)
                        : make_float4(0.f, 0.f, 0.f, 0.f);
                    hv[4 * j] = x.x; hv[4 * j + 1] = x.y; hv[4 * j + 2] = x.z; hv[4 * j + 3] = x.w;
                }
                tmem_st16(tH + lane_off + 16 * hc, hv);
                tc_fence_before();
            }
            for (int64_t t0 = bos; t0 < eos && !gfail; t0 += C, ++ci) {
                const int len = (int)((eos - t0) < C ? (eos - t0) : C);
                const int s = (int)(ci & 1);
                const uint32_t par = (uint32_t)(ci & 1);
                unsigned char *sl = slot(s);
                if (!wait_t(bar(Bar::slot_full + s), (uint32_t)((ci >> 1) & 1), wt)) failed = true;
                if (bar_red_or(kBarStep, kGroup, failed)) { failed = gfail = true; break; }
                if (tid == 0) *reinterpret_cast<volatile int64_t *>(sm + Smem::consumed) = ci + 1;
                tc_fence_after();
                const uint32_t tD1 = tmem + 64 * s, tD1b = tD1 + 32;   // this chunk's accumulators
                const __half *aop = reinterpret_cast<const __half *>(sl + Rec::aop);
                const __half *kht = reinterpret_cast<const __half *>(sl + Rec::kht);
                const __half *ta = reinterpret_cast<const __half *>(sl + Rec::ta);
                const float *bts = reinterpret_cast<const float *>(sl + Rec::beta);
                const float *decs = reinterpret_cast<const float *>(sl + Rec::dec);
                const float *pms = reinterpret_cast<const float *>(sl + Rec::pm);
                const __nv_bfloat16 *vsl = reinterpret_cast<const __nv_bfloat16 *>(sl + Smem::slot_v);

                // ---------------- fp16 copy (2^m h)^T for S1, then h <- Diag(2^G_last) h
                {
                    float hv[16];
                    tmem_ld16(tH + lane_off + 16 * hc, hv);
                    const float p = pms[sc], d = decs[sc];
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

                // ---------------- MMA S1: D1 = [a_k; a_q] (2^m h) = [K~ h; Q~ h], channels
                //                  0..63 into D1 by thread 0 and 64..127 into D1b by thread 32
                if (tid == 0 || tid == 32) {
                    tc_fence_after();
                    const int k0 = tid == 0 ? 0 : KD / 32;
                    const uint32_t dst = tid == 0 ? tD1 : tD1b;
#pragma unroll
                    for (int ks = 0; ks < KD / 32; ++ks)
                        umma_f16(dst, sw128_kdesc(smem_u32(aop), k0 + ks, 2 * C),
                                 sw128_kdesc(smem_u32(ht), k0 + ks, VT), kIdescM128N32, ks > 0);
                    umma_commit(bar(Bar::s1));
                }
                // ---------------- X = beta (v - K~ h) from rows 0..63 of D1 (warps 0, 1, 4, 5)
                if ((warp & 2) == 0) {
                    if (!wait_t(bar(Bar::s1), par, wt)) failed = true;
                    tc_fence_after();
                    const int r = 32 * (warp & 1) + lane, half = warp >> 2;
                    float xv[16], xb[16];
                    tmem_ld16(tD1 + lane_off + 16 * half, xv);
                    tmem_ld16(tD1b + lane_off + 16 * half, xb);
#pragma unroll
                    for (int v = 0; v < 16; ++v) xv[v] += xb[v];
                    const float b = bts[r];
                    const uint4 *vrow = reinterpret_cast<const uint4 *>(vsl + r * VT + 16 * half);
                    uint32_t xw[8];
#pragma unroll
                    for (int j = 0; j < 2; ++j) {
                        const uint4 wv = vrow[j];
                        const __nv_bfloat162 *p2 = reinterpret_cast<const __nv_bfloat162 *>(&wv);
#pragma unroll
                        for (int u = 0; u < 4; ++u) {
                            const float2 vv = __bfloat1622float2(p2[u]);
                            const int v = 8 * j + 2 * u;
                            xw[4 * j + u] = pack_h2(b * (vv.x - xv[v]), b * (vv.y - xv[v + 1]));
                        }
                    }
                    uint4 *xrow = reinterpret_cast<uint4 *>(xs + r * LDX + 16 * half);
                    xrow[0] = make_uint4(xw[0], xw[1], xw[2], xw[3]);
                    xrow[1] = make_uint4(xw[4], xw[5], xw[6], xw[7]);
                    tc_fence_before();
                } else {
                    flush_o();   // the previous chunk's output rows
                }
                named_bar_sync(kBarStep, kGroup);   // S1 is complete: ht (= xs) and D1 rows are free

                // ---------------- S2: D = T (beta X) on mma.sync, warp w: rows [16 (w % 4), +16),
                //                  value columns [16 (w / 4), +16); T lower triangular: k-blocks
                //                  <= the row block.  D^T goes to dt (SW128) by stmatrix.
                {
                    const int mt = warp & 3, nh = warp >> 2;
                    float dk[4][2][4];   // one accumulator pair per k-block (no chained mma)
                    const int arow = 16 * mt + (lane & 15), akoff = (lane >> 4) << 3;
                    const int xrow = (lane & 7) + (((lane >> 3) & 1) << 3), xcol = 16 * nh + ((lane >> 4) << 3);
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks) {
#pragma unroll
                        for (int nt = 0; nt < 2; ++nt) dk[ks][nt][0] = dk[ks][nt][1] = dk[ks][nt][2] = dk[ks][nt][3] = 0.f;
                        if (ks <= mt) {
                            uint32_t af[4], bf[4];
                            ldsm_x4(smem_u32(ta + sw128(arow, 16 * ks + akoff, 2 * C)), af[0], af[1], af[2], af[3]);
                            ldsm_x4_t(smem_u32(xs + (16 * ks + xrow) * LDX + xcol), bf[0], bf[1], bf[2], bf[3]);
                            mma16816(dk[ks][0], af, bf[0], bf[1]);
                            mma16816(dk[ks][1], af, bf[2], bf[3]);
                        }
                    }
                    uint32_t dw[4];   // stmatrix order: (nt 0, rows g), (nt 0, rows g + 8), (nt 1, g), (nt 1, g + 8)
#pragma unroll
                    for (int nt = 0; nt < 2; ++nt) {
                        float e[4];
#pragma unroll
                        for (int q = 0; q < 4; ++q)
                            e[q] = (dk[0][nt][q] + dk[1][nt][q]) + (dk[2][nt][q] + dk[3][nt][q]);
                        dw[2 * nt] = pack_h2(e[0], e[1]);
                        dw[2 * nt + 1] = pack_h2(e[2], e[3]);
                    }
                    const int mi = lane >> 3, mj = lane & 7;
                    stsm_x4_t(smem_u32(dt + sw128(16 * nh + 8 * (mi >> 1) + mj, 16 * mt + 8 * (mi & 1), VT)),
                              dw[0], dw[1], dw[2], dw[3]);
                }
                fence_proxy_async_smem();
                named_bar_sync(kBarStep, kGroup);

                // ---------------- MMA S3: h += K^^T D (thread 0) ; D1[64..127] += A_qk D (thread 32)
                if (tid == 0) {
                    tc_fence_after();
#pragma unroll
                    for (int ks = 0; ks < C / 16; ++ks)
                        umma_f16(tH, sw128_kdesc(smem_u32(kht), ks, KD), sw128_kdesc(smem_u32(dt), ks, VT),
                                 kIdescM128N32, 1u);
                    umma_commit(bar(Bar::s3));
                } else if (tid == 32) {
                    tc_fence_after();
                    // A = [T (rows 0..63, lands in the consumed X rows); A_qk (rows 64..127)]
#pragma unroll
                    for (int ks = 0; ks < C / 16; ++ks)
                        umma_f16(tD1, sw128_kdesc(smem_u32(ta), ks, 2 * C), sw128_kdesc(smem_u32(dt), ks, VT),
                                 kIdescM128N32, 1u);
                    umma_commit(bar(Bar::s3));
                }
                // slot s's v region is free (X is done): the local part of arming it for
                // chunk ci + 2 runs while S3 does
                const bool arming = tid == kArmer && lhave;
                if (arming) arm_local();
                if (!wait_t(bar(Bar::s3), par, wt)) failed = true;
                tc_fence_after();
                // every read of slot s is done (generic ones before the barrier above, tcgen05
                // ones at the S3 commit): the builder may overwrite it
                if (arming) arm_remote();
                if (warp & 2) {   // rows 64..127 of D1 (the output) are stored during the next chunk
                    pend = true;
                    pend_par = s;
                    pend_t0 = t0;
                    pend_len = len;
                    pend_h = h;
                }
                tc_fence_before();
            }
            if (fin && !gfail) {   // final state (after a failed wait: left unwritten, status reported)
                tc_fence_after();
                float hv[16];
                tmem_ld16(tH + lane_off + 16 * hc, hv);
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    *reinterpret_cast<float4 *>(fin + (int64_t)sc * VD + vt * VT + 16 * hc + 4 * j) =
                        make_float4(hv[4 * j], hv[4 * j + 1], hv[4 * j + 2], hv[4 * j + 3]);
            }
            tc_fence_before();
            named_bar_sync(kBarStep, kGroup);   // TMEM h is read before the next item's init
        }
        if (warp & 2) flush_o();   // the last chunk's output rows
        if (failed) {   // copies and MMAs still in flight get one more bounded wait
            if (tid == kArmer)
                for (int64_t c = ci; c < lci; ++c) mbar_drain(bar(Bar::slot_full + (int)(c & 1)), (uint32_t)((c >> 1) & 1));
            mbar_drain(bar(Bar::s1), (uint32_t)(ci & 1));
            mbar_drain(bar(Bar::s3), (uint32_t)(ci & 1));
        }
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync_all();   // no CTA leaves while a peer may still arrive on its barriers
    if (warp == 0) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" :: "r"(tmem), "r"(256) : "memory");
    }
}

// clusters that can be resident at once (persistent grid), per device.  The value is a
// property of the device and the kernel, not of a context, so the cache stays valid across
// a device reset; threads that race on a device's first query store the same value.
int max_clusters()
{
    static int cached[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 1;
    if (cached[dev] > 0) return cached[dev];
    int n = 0;
    if (cudaFuncSetAttribute(kda_prefill_rr_kernel<__nv_bfloat16, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             Smem::total) == cudaSuccess) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(kRanks * 1024);
        cfg.blockDim = dim3(kThreads);
        cfg.dynamicSmemBytes = Smem::total;
        if (cudaOccupancyMaxActiveClusters(&n, kda_prefill_rr_kernel<__nv_bfloat16, false>, &cfg) != cudaSuccess) n = 0;
    }
    cudaGetLastError();   // a failed query leaves no sticky error behind
    if (n <= 0) {
        int sms = 0;
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        n = sms / kRanks > 0 ? sms / kRanks : 1;
    }
    cached[dev] = n;
    return n;
}

// clusters of a launch: the work items, the resident clusters and the ring the workspace
// holds, whichever is least
int64_t rr_clusters(int64_t items, size_t ring_records)
{
    const int64_t m = max_clusters();
    int64_t g = items < m ? items : m;
    const int64_t cap = (int64_t)(ring_records / kRing);
    return g < cap ? g : cap;
}

std::atomic<unsigned long long> g_wait_ns{2000000000ull};

template <typename Tout, bool kL2>
cudaError_t launch_rr_t(const PrefillArgs &a, void *ws, size_t ws_bytes, cudaStream_t stream)
{
    RrMaps maps;
    memset(&maps, 0, sizeof(maps));
    if (a.total_tokens > 0) {
        const int64_t T = a.total_tokens;
        const int H = a.num_heads;
        if (!encode_map(&maps.q, a.q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, T, H, KD, KD) ||
            !encode_map(&maps.k, a.k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, T, H, KD, KD) ||
            !encode_map(&maps.g, a.g, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, T, H, KD, KD) ||
            !encode_map(&maps.v, a.v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, T, H, VD, VT))
            return cudaErrorInvalidValue;
        maps.beta_map = (H % 4 == 0) && encode_map_2d(&maps.beta, a.beta, T, H);
    }
    cudaError_t e = cudaFuncSetAttribute(kda_prefill_rr_kernel<Tout, kL2>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, Smem::total);
    if (e != cudaSuccess) return e;
    const size_t records = ws_bytes > (size_t)kWsHeader ? (ws_bytes - kWsHeader) / Rec::bytes : 0;
    const int64_t G = rr_clusters((int64_t)a.num_seqs * a.num_heads, records);
    if (G < 1) return cudaErrorInvalidValue;
    unsigned char *base = static_cast<unsigned char *>(ws);
    const RrWait wt{reinterpret_cast<int *>(base), g_wait_ns.load()};
    kda_prefill_rr_kernel<Tout, kL2><<<(unsigned)(G * kRanks), kThreads, Smem::total, stream>>>(
        a, maps, base + kWsHeader, (int)G, wt);
    return cudaGetLastError();
}

}  // namespace

bool prefill_rr_supported(const PrefillArgs &a)
{
    return a.dtype == kDtypeBF16 && a.head_dim_k == KD && a.head_dim_v == VD;
}

size_t prefill_rr_workspace_bytes(const PrefillArgs &a)
{
    if (!prefill_rr_supported(a) || a.num_seqs == 0) return 0;
    const int64_t items = (int64_t)a.num_seqs * a.num_heads;
    const int64_t m = max_clusters();
    return (size_t)kWsHeader + (size_t)(items < m ? items : m) * kRing * Rec::bytes;
}

cudaError_t launch_prefill_rr(const PrefillArgs &a, void *workspace, size_t workspace_bytes,
                              cudaStream_t stream)
{
    if (a.num_seqs == 0) return cudaSuccess;
    const bool l2 = (a.flags & kFlagQkL2Norm) != 0;
    if (a.out_dtype == kDtypeBF16)
        return l2 ? launch_rr_t<__nv_bfloat16, true>(a, workspace, workspace_bytes, stream)
                  : launch_rr_t<__nv_bfloat16, false>(a, workspace, workspace_bytes, stream);
    return l2 ? launch_rr_t<float, true>(a, workspace, workspace_bytes, stream)
              : launch_rr_t<float, false>(a, workspace, workspace_bytes, stream);
}

void set_prefill_wait_limit_ns(unsigned long long ns)
{
    g_wait_ns.store(ns == 0 ? 2000000000ull : ns);
}

}  // namespace kda
