// kda_prefill_wy.cu -- chunked KDA prefill on tensor cores: the chunk-parallel work and
// the serial state scan run on different CTAs of one cooperative launch.
//
// The computation is the chunked prompt path of vllm.cpp PR #110 ("chunk_kda prefill
// AOT port", commit description: the in-chunk gate cumsum in exp2 space, the decayed
// intra-chunk k.k^T, the unit-lower-triangular solve, the WY recompute of w and u, the
// inter-chunk state propagation h and the output o).  Per 64-token chunk of one
// (sequence, head), with G = log2(e) cumsum(g) per key channel and the state h (K x V):
//     A_kk = beta_r strict_lower(sum_c k_rc k_ic 2^(G_rc - G_ic))
//     A_qk = lower(sum_c q_rc k_ic 2^(G_rc - G_ic)),      T = (I + A_kk)^-1
//     W = T Diag(beta) K~,  U = T Diag(beta) v,  K~ = k 2^G,  Q~ = q 2^G,  K^ = k 2^(G_last - G)
//     D = U - W h;   o = scale (Q~ h + A_qk D);   h <- Diag(2^G_last) h + K^^T D
// Everything up to D depends on the chunk's own inputs; only the last line carries
// state.  The two parts run on different CTAs:
//
//   * BUILDER CTAs (two independent groups of 8 warps each) take (scanner, position)
//     tickets and build each chunk's RECORD -- [W; Q~], U, 2^G_last, K^^T and A_qk as
//     fp16 tensor-core operands -- store it with one bulk copy into that scanner's ring
//     of 8 records in the workspace (it stays in L2) and publish it with a release flag;
//   * SCANNER CTAs, one per (sequence, head) work item at a time, keep the state in
//     tensor memory (fp32) and run the chain per chunk:
//         copy  h16 = fp16(hs h) -> shared memory;  h <- Diag(2^G_last) h    CUDA cores
//         S1    [W h; Q~ h] = [W; Q~] h16                (tcgen05 M128 N128 K128)
//         D     D = U - W h  -> fp16                      CUDA cores
//         S3    h += K^^T D;  [.; o] += [.; A_qk] D     (tcgen05 M128 N128 K64)
//     The output rows of a chunk are stored during the next chunk's D step; one of the
//     output warps also pulls the records in (two bulk copies per record, two
//     shared-memory slots).
//
// Deadlock freedom.  The grid is launched cooperatively, so every CTA is resident.
// Tickets j = p S + s (position p of scanner s) go to builder unit j mod NBU, and each
// unit takes its tickets in increasing order.  A builder waits only for ring entry
// p % 8 to be free (scanner s has consumed position p - 8, whose ticket is smaller);
// a scanner waits only for its next record.  The unfinished ticket with the smallest
// index therefore never waits on anything unfinished.  Every wait is bounded in time:
// on expiry it records KDA timeout status in the workspace, raises an abort word that
// every other wait polls, drains its own copies and MMAs in flight and returns.
//
// Numerics (emulated against the fp64 oracle before this kernel was written: 7.0e-4 /
// 4.8e-4 on outputs / final states for a 4096-token prompt, 7.8e-4 / 6.7e-4 on the
// packed varlen batch with nonzero initial states).  All tensor-core operands are fp16,
// accumulation and the state fp32.  The A matrices use per-channel factors centred on a
// reference m (a = x 2^(G - m), b = k 2^(m - G), each within [2^-8, 2^8] while the
// chunk's gate spans at most 16 in log2; wider chunks take an exact-exponential path for
// A_kk, A_qk and K^^T).  W and Q~ leave the builder un-centred (W = (T Diag(beta) a_k)
// 2^(m - M), Q~ = a_q 2^(m - M)), so the scanner's fp16 state copy needs no per-channel
// factor; M = max(0, ceil(max G) - 8) is 0 for any decay gate and keeps W and Q~ in
// range for growth gates (the copy is then scaled by hs = 2^M).
#include <atomic>
#include <cstring>

#include "kda_tc_common.cuh"

namespace kda {
namespace {

constexpr int kThreads = 512;    // 16 warps: scanner chain; builder 2 groups x 8
constexpr int kMoverWarp = 15;   // scanner warp that also moves the records in (an output warp)
constexpr int kChain = 512;      // scanner chain threads
constexpr int kGroup = 256;      // threads of a builder group
constexpr int kBarChain = 1;     // named barrier of the scanner chain warps
constexpr int kRing = kWyRing;   // records per scanner in the workspace ring
constexpr int kScanMax = kWyScanMax;

// ------------------------------------------------------------------ record layout
// The byte image of the shared-memory operand tiles the scanner reads for one chunk.
// Part A (copy step, S1, D step) comes first, part B (S3) after it, so that the two
// parts can be reloaded separately as the scanner frees them.
struct Rec {
    static constexpr int aop = 0;               // SW128 K-major [W; Q~] 128 rows x 128 channels
    static constexpr int u = 32768;             // SW128 [64 rows][128 values] (MN-major B layout)
    static constexpr int dec = 49152;           // f32 [128] 2^G_last
    static constexpr int hs = dec + 512;        // f32 scale of the fp16 state copy (2^M)
    static constexpr int partA = 50176;
    static constexpr int kht = 50176;           // SW128 K-major K^^T 128 channels x 64 rows
    static constexpr int aqk = kht + 16384;     // SW128 K-major A_qk 64 x 64: rows 64..127 of the
                                                // 128-row tile at kht + 8192 (S3's output A operand)
    static constexpr int bytes = aqk + 8192;    // 74,752
};
static_assert(Rec::bytes == kWyRecordBytes, "record size");
static_assert(Rec::bytes % 1024 == 0 && Rec::partA % 1024 == 0 && Rec::kht % 1024 == 0 &&
              Rec::aqk % 1024 == 0 && Rec::u % 1024 == 0, "SW128 tiles need 1024-byte alignment");

// ------------------------------------------------------------------ scanner shared memory
struct Ssm {
    static constexpr int slot = Rec::bytes;                 // slot s at s * slot
    static constexpr int ht = 2 * Rec::bytes;               // SW128 h16 [128 channels][128 values]
    static constexpr int dt = ht + 32768;                   // SW128 D [64 rows][128 values]
    static constexpr int bars = dt + 16384;                 // mbarriers
    static constexpr int total = bars + 128;
};
struct SBar { enum { full = 0, s1 = 2, s3h = 3, s3o = 4, count = 5 }; };
static_assert(Ssm::ht % 1024 == 0 && Ssm::dt % 1024 == 0, "SW128 tiles need 1024-byte alignment");

// ------------------------------------------------------------------ builder shared memory (per group)
struct Cur {            // the scanner's item that holds the positions from pos0 on
    int32_t w, pos0, bos, eos;
};
struct Gsm {
    static constexpr int r1 = 0;              // SW128 [a_k; a_q] 128 x 128, then [W; Q~] (record aop)
    static constexpr int r3 = Rec::u;         // SW128 v (fp16), then U (record u)
    static constexpr int vec = Rec::dec;      // 2^G_last, hs (record)
    static constexpr int kht = Rec::kht;      // record K^^T
    static constexpr int aqk = Rec::aqk;      // record A_qk
    static constexpr int r2 = Rec::bytes;     // SW128 b 64 x 128; then T Diag(beta) (rows 0..63 of a
                                              // 128-row K=64 tile) and A_kk (SW128 64 x 64 at r2 + 8192)
    static constexpr int akk = r2 + 8192;
    static constexpr int tm = r2 + 16384;     // f16 T [64][LD64]
    static constexpr int tot = tm + C * LD64 * 2;   // f32 [4][128] per-16-row column sums of G
    static constexpr int first = tot + 2048;  // f32 [128] G of row 0
    static constexpr int bs = first + 512;    // f32 [64] beta
    static constexpr int pm = bs + 256;       // f32 [128] 2^(m - M)
    static constexpr int wmax = pm + 512;     // f32 [8] per-warp max of G
    static constexpr int cur = wmax + 32;     // Cur [kScanMax]
    static constexpr int tots = cur + 16 * kScanMax;   // i32 [kScanMax] positions per scanner
    static constexpr int misc = tots + 4 * kScanMax;   // i32 [16] ticket broadcast
    static constexpr int bars = misc + 64;    // mbarriers: MMA A, MMA W/U
    static constexpr int group = (bars + 16 + 1023) / 1024 * 1024;
};
static_assert(Gsm::tm % 16 == 0 && Gsm::r2 % 1024 == 0 && Gsm::akk % 1024 == 0, "alignment");

constexpr int kTmemSlot = 2 * Gsm::group;           // u32: tensor-memory base of the CTA
constexpr int kSmemTotal = kTmemSlot + 16;
static_assert(Ssm::total <= kTmemSlot, "scanner map below the tensor-memory slot");
static_assert(kSmemTotal <= 232448, "shared memory budget");

// instruction descriptor: fp16 A (K-major) and B (MN-major), fp32 D, M = 128, N = 128
constexpr uint32_t kIdescM128N128Bmn = (1u << 4) | (1u << 16) | ((128u >> 3) << 17) | ((128u >> 4) << 24);

// Shared-memory descriptor of an SW128 MN-major operand: rows = K index (128 B each, 8-row
// groups 1024 B apart), 64-element MN blocks `lbo` bytes apart.
__device__ __forceinline__ uint64_t sw128_mn_desc(uint32_t saddr, uint32_t lbo)
{
    return (uint64_t)((saddr >> 4) & 0x3FFF) | ((uint64_t)((lbo >> 4) & 0x3FFF) << 16) |
           ((uint64_t)(1024 >> 4) << 32) | ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

// ------------------------------------------------------------------ parameters
struct WyParams {
    unsigned char *rec;               // [S][kRing] records
    unsigned long long *ready;        // [S][kRing] (epoch << 32) | (position + 1)
    unsigned long long *consumed;     // [S] stride 8: (epoch << 32) | positions consumed
    unsigned long long *abort_word;   // epoch of an aborted launch
    int *status;                      // KDA status of the last failed launch (0: none)
    unsigned long long wait_ns;       // limit of every wait
    unsigned int epoch;               // this launch's tag, never 0
    int S;                            // scanner CTAs (= blockIdx 0..S-1)
};

// ------------------------------------------------------------------ small PTX helpers
__device__ __forceinline__ uint64_t gtimer()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
__device__ __forceinline__ uint64_t ld_acquire(const unsigned long long *p)
{
    uint64_t v;
    asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void st_release(unsigned long long *p, uint64_t v)
{
    asm volatile("st.release.gpu.global.u64 [%0], %1;" :: "l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ void fence_proxy_async_global() { asm volatile("fence.proxy.async.global;\n" ::: "memory"); }
__device__ __forceinline__ bool mbar_try(uint32_t mbar, uint32_t parity)
{
    uint32_t done;
    asm volatile("{\n.reg .pred p;\nmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
                 "selp.u32 %0, 1, 0, p;\n}\n"
                 : "=r"(done) : "r"(mbar), "r"(parity) : "memory");
    return done != 0;
}
// 1-D bulk copy global -> this CTA's shared memory, completing on an mbarrier
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void *src, uint32_t bytes, uint32_t mbar)
{
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n"
                 :: "r"(dst), "l"(src), "r"(bytes), "r"(mbar) : "memory");
}
// 1-D bulk copy shared -> global (bulk async-group)
__device__ __forceinline__ void bulk_s2g(void *dst, uint32_t src, uint32_t bytes)
{
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;\n"
                 :: "l"(dst), "r"(src), "r"(bytes) : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;\n" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;\n" ::: "memory"); }

// 32 lanes x 32 columns of fp32 from / to tensor memory (no wait)
__device__ __forceinline__ void tmem_ld32_nw(uint32_t taddr, uint32_t (&r)[32])
{
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x32.b32 "
                 "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
                 "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
                   "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
                   "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
                   "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
                   "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
                   "=r"(r[31])
                 : "r"(taddr));
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory"); }
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32])
{
    uint32_t r[32];
    tmem_ld32_nw(taddr, r);
    tmem_wait_ld();
#pragma unroll
    for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]);
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float (&v)[32])
{
    asm volatile("tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
                 "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
                 "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};\n"
                 :: "r"(taddr), "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])),
                    "r"(__float_as_uint(v[2])), "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])),
                    "r"(__float_as_uint(v[5])), "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])),
                    "r"(__float_as_uint(v[8])), "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])),
                    "r"(__float_as_uint(v[11])), "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])),
                    "r"(__float_as_uint(v[14])), "r"(__float_as_uint(v[15])), "r"(__float_as_uint(v[16])),
                    "r"(__float_as_uint(v[17])), "r"(__float_as_uint(v[18])), "r"(__float_as_uint(v[19])),
                    "r"(__float_as_uint(v[20])), "r"(__float_as_uint(v[21])), "r"(__float_as_uint(v[22])),
                    "r"(__float_as_uint(v[23])), "r"(__float_as_uint(v[24])), "r"(__float_as_uint(v[25])),
                    "r"(__float_as_uint(v[26])), "r"(__float_as_uint(v[27])), "r"(__float_as_uint(v[28])),
                    "r"(__float_as_uint(v[29])), "r"(__float_as_uint(v[30])), "r"(__float_as_uint(v[31]))
                 : "memory");
    asm volatile("tcgen05.wait::st.sync.aligned;\n" ::: "memory");
}

// ------------------------------------------------------------------ failure handling
__device__ __forceinline__ bool aborted(const WyParams &w)
{
    return *reinterpret_cast<volatile unsigned long long *>(w.abort_word) == (unsigned long long)w.epoch;
}
__device__ __noinline__ void raise_timeout(const WyParams &w)
{
    atomicExch(w.status, kStatusTimeout);
    *reinterpret_cast<volatile unsigned long long *>(w.abort_word) = (unsigned long long)w.epoch;
    __threadfence();
}

// Wait on a local mbarrier phase whose completion may depend on other CTAs: bounded by
// the launch's wait limit and abandoned when another CTA has aborted.
__device__ bool mbar_wait_t(uint32_t mbar, uint32_t parity, const WyParams &w)
{
    uint64_t t0 = 0;
    for (uint32_t i = 0;; ++i) {
        if (mbar_try(mbar, parity)) return true;
        if ((i & 31) == 31) {
            const uint64_t t = gtimer();
            if (t0 == 0) t0 = t;
            else if (t - t0 > w.wait_ns) { raise_timeout(w); return false; }
            if (aborted(w)) return false;
        }
    }
}
// Wait for a phase that completes by itself (an MMA commit, a copy already issued):
// a fixed generous bound, for the clean-up after a failure.
__device__ bool mbar_drain(uint32_t mbar, uint32_t parity)
{
    for (int i = 0; i < (1 << 20); ++i)
        if (mbar_try(mbar, parity)) return true;
    return false;
}
// Poll a flag word until (epoch, count) with count >= want: bounded like mbar_wait_t.
__device__ bool flag_wait(const unsigned long long *p, uint32_t want, const WyParams &w)
{
    uint64_t t0 = 0;
    for (uint32_t i = 0;; ++i) {
        const uint64_t v = ld_acquire(p);
        if ((uint32_t)(v >> 32) == w.epoch && (uint32_t)v >= want) return true;
        if ((i & 7) == 7) {
            const uint64_t t = gtimer();
            if (t0 == 0) t0 = t;
            else if (t - t0 > w.wait_ns) { raise_timeout(w); return false; }
            if (aborted(w)) return false;
        }
        __nanosleep(64);
    }
}

__device__ __forceinline__ void item_range(const PrefillArgs &a, int64_t wi, int64_t &bos, int64_t &eos)
{
    const int64_t n = wi / a.num_heads;
    clamp_range(a.total_tokens, a.cu_seqlens[n], a.cu_seqlens[n + 1], bos, eos);
}

// Exact-exponential A_kk, A_qk and K^^T (shared memory) for a chunk whose gate span
// leaves the fp16 factors' range: one exponential per pair and channel.  G is the
// chunk's exp2-space cumsum, fp32 [64][128], in global scratch.
__device__ __noinline__ void exact_pairs(const PrefillArgs &a, int64_t t0, int len, int h,
                                         const float *G, const float *bs, __half *akk, __half *aqk,
                                         __half *kht, int gtid)
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
        }
        akk[sw128(r, i, C)] = __float2half_rn(i < r ? bs[r] * sk : 0.f);
        aqk[sw128(r, i, C)] = __float2half_rn(i <= r ? sq : 0.f);
    }
    // K^^T = (k 2^(G_last - G))^T, one exponential per element; rows past the end have
    // G = G_last and k = 0
    for (int e = gtid; e < C * KD; e += kGroup) {
        const int r = e >> 7, c = e & 127;
        const float kv = r < len ? __bfloat162float(kk[((t0 + r) * H + h) * KD + c]) : 0.f;
        kht[sw128(c, r, KD)] = __float2half_rn(kv * exp2f(G[(C - 1) * KD + c] - G[r * KD + c]));
    }
}

// =====================================================================================
// Builder: two groups of 8 warps per CTA, each an independent unit taking tickets.
// =====================================================================================
__device__ __forceinline__ void builder(const PrefillArgs &a, const WyParams &wp, unsigned char *sm,
                                     uint32_t tmem)
{
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int grp = warp >> 3;
    const int gtid = tid - kGroup * grp, gw = warp & 7;
    const int bar_id = 1 + grp;
    unsigned char *gs = sm + Gsm::group * grp;
    const uint32_t tg = tmem + 256u * (uint32_t)grp;             // the group's 256 TMEM columns
    const uint32_t lane_off = (uint32_t)(32 * (warp & 3)) << 16;  // lane quadrant of this warp
    const int S = wp.S;
    const int64_t NBU = 2 * ((int64_t)gridDim.x - S);
    const int64_t unit = 2 * ((int64_t)blockIdx.x - S) + grp;
    const int H = a.num_heads;
    const int64_t NH = (int64_t)a.num_seqs * H;

    __half *r1 = reinterpret_cast<__half *>(gs + Gsm::r1);
    __half *r2 = reinterpret_cast<__half *>(gs + Gsm::r2);
    __half *r3 = reinterpret_cast<__half *>(gs + Gsm::r3);
    __half *akk = reinterpret_cast<__half *>(gs + Gsm::akk);
    __half *aqk = reinterpret_cast<__half *>(gs + Gsm::aqk);
    __half *kht = reinterpret_cast<__half *>(gs + Gsm::kht);
    __half *tmh = reinterpret_cast<__half *>(gs + Gsm::tm);
    float *tot = reinterpret_cast<float *>(gs + Gsm::tot);
    float *first = reinterpret_cast<float *>(gs + Gsm::first);
    float *bs = reinterpret_cast<float *>(gs + Gsm::bs);
    float *pms = reinterpret_cast<float *>(gs + Gsm::pm);
    float *wmax = reinterpret_cast<float *>(gs + Gsm::wmax);
    float *decs = reinterpret_cast<float *>(gs + Gsm::vec);
    float *hsp = reinterpret_cast<float *>(gs + Gsm::vec + (Rec::hs - Rec::dec));
    Cur *cur = reinterpret_cast<Cur *>(gs + Gsm::cur);
    int *tots = reinterpret_cast<int *>(gs + Gsm::tots);
    volatile int *misc = reinterpret_cast<volatile int *>(gs + Gsm::misc);
    const uint32_t barA = smem_u32(gs + Gsm::bars), barW = barA + 8;
    const float *gin = a.g;
    const __nv_bfloat16 *qin = static_cast<const __nv_bfloat16 *>(a.q);
    const __nv_bfloat16 *kin = static_cast<const __nv_bfloat16 *>(a.k);
    const __nv_bfloat16 *vin = static_cast<const __nv_bfloat16 *>(a.v);

    // ---- positions per scanner (each item's chunks), and the ticket cursors
    for (int s = gtid; s < S; s += kGroup) tots[s] = 0;
    named_bar_sync(bar_id, kGroup);
    for (int64_t wi = gtid; wi < NH; wi += kGroup) {
        int64_t b, e;
        item_range(a, wi, b, e);
        atomicAdd(&tots[wi % S], (int)((e - b + C - 1) / C));
    }
    for (int s = gtid; s < S; s += kGroup) {
        int64_t b, e;
        item_range(a, s, b, e);
        cur[s] = Cur{s, 0, (int32_t)b, (int32_t)e};
    }
    named_bar_sync(bar_id, kGroup);
    int pmax = 0;
    for (int s = 0; s < S; ++s) pmax = tots[s] > pmax ? tots[s] : pmax;

    uint32_t a_par = 0, w_par = 0;
    bool a_pending = false, w_pending = false, failed = false;
    int64_t iter = 0;
    for (int64_t j = unit; ; j += NBU, ++iter) {
        const int64_t p = j / S;
        const int s = (int)(j % S);
        if (p >= pmax) break;
        // ---- ticket -> (item, chunk) through the scanner's cursor (thread 0), broadcast in
        //      a slot of its own per iteration parity: a slot is rewritten two tickets later,
        //      after every thread has passed the next ticket's barrier
        volatile int *bc = misc + 4 * (int)(iter & 1);
        if (gtid == 0) {
            Cur c = cur[s];
            while (c.w < NH) {
                const int nch = (c.eos - c.bos + C - 1) / C;
                if (p < (int64_t)c.pos0 + nch) break;
                c.pos0 += nch;
                c.w += S;
                if (c.w < NH) {
                    int64_t b, e;
                    item_range(a, c.w, b, e);
                    c.bos = (int32_t)b;
                    c.eos = (int32_t)e;
                }
            }
            cur[s] = c;
            const bool ok = c.w < NH;
            bc[0] = ok ? 1 : 0;
            bc[1] = c.w;
            bc[2] = ok ? c.bos + (int)(p - c.pos0) * C : 0;
            bc[3] = ok ? c.eos : 0;
        }
        if (bar_red_or(bar_id, kGroup, gtid == 0 && aborted(wp))) { failed = true; break; }
        if (bc[0] == 0) continue;
        const int64_t wi = bc[1];
        const int64_t t0 = bc[2];
        const int len = (bc[3] - (int)t0) < C ? (bc[3] - (int)t0) : C;
        const int h = (int)(wi % H);
        unsigned char *rec = wp.rec + ((int64_t)s * kRing + p % kRing) * Rec::bytes;
        const unsigned long long *consumed = wp.consumed + 8 * (int64_t)s;
        const uint32_t want_free = p >= kRing ? (uint32_t)(p - kRing + 1) : 0u;
        volatile int *xflag = misc + 8;   // fast-path test of this ticket
        if (gtid == 0) *xflag = 0;

        // ---------------- P1: gate cumsum in exp2 space; thread = (channel pair, 16-row group E)
        const int pcp = gtid & 63, pE = gtid >> 6, pc0 = 2 * pcp;
        float2 gx[16];
        uint32_t kq[16], qq[16];
#pragma unroll
        for (int u = 0; u < 16; ++u) {
            const int r = 16 * pE + u;
            const int64_t off = ((t0 + r) * H + h) * KD + pc0;
            gx[u] = r < len ? __ldg(reinterpret_cast<const float2 *>(gin + off)) : make_float2(0.f, 0.f);
            kq[u] = r < len ? __ldg(reinterpret_cast<const unsigned int *>(kin + off)) : 0u;
            qq[u] = r < len ? __ldg(reinterpret_cast<const unsigned int *>(qin + off)) : 0u;
        }
#pragma unroll
        for (int u = 0; u < 16; ++u) gx[u] = make_float2(gx[u].x * kLog2e, gx[u].y * kLog2e);
#pragma unroll
        for (int u = 1; u < 16; ++u) { gx[u].x += gx[u - 1].x; gx[u].y += gx[u - 1].y; }
        *reinterpret_cast<float2 *>(tot + pE * KD + pc0) = gx[15];
        if (pE == 0) *reinterpret_cast<float2 *>(first + pc0) = gx[0];
        if (gtid < C) bs[gtid] = gtid < len ? a.beta[(t0 + gtid) * H + h] : 0.f;
        named_bar_sync(bar_id, kGroup);

        // ---------------- P2: reference, fp16 factors, K^^T, 2^G_last
        float2 pre = make_float2(0.f, 0.f), run = make_float2(0.f, 0.f);
#pragma unroll
        for (int E = 0; E < 4; ++E) {
            const float2 t = *reinterpret_cast<const float2 *>(tot + E * KD + pc0);
            if (E == pE) pre = run;
            run.x += t.x; run.y += t.y;
        }
        const float2 glast = run, g0 = *reinterpret_cast<const float2 *>(first + pc0);
        // reference: the midpoint of the first and last row's G, capped so that no factor
        // 2^(G - m) exceeds 2^8
        const float mx_ = fmaxf(0.5f * (g0.x + glast.x), g0.x - 0.5f * kSpanMax);
        const float my_ = fmaxf(0.5f * (g0.y + glast.y), g0.y - 0.5f * kSpanMax);
        if (pE == 0)
            *reinterpret_cast<float2 *>(decs + pc0) = make_float2(exp2f(glast.x), exp2f(glast.y));
        const float fx = exp2f(glast.x - mx_), fy = exp2f(glast.y - my_);   // K^ = b 2^(G_last - m)
        const float bx = pre.x - mx_, by = pre.y - my_;                     // G_r - m = gx + b
        float amax = 0.f, gmx = -3.0e38f;
#pragma unroll
        for (int hb = 0; hb < 2; ++hb) {
            float khx[8], khy[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int r = 16 * pE + 8 * hb + u;
                gmx = fmaxf(gmx, fmaxf(gx[8 * hb + u].x + pre.x, gx[8 * hb + u].y + pre.y));
                const float xx = gx[8 * hb + u].x + bx, xy = gx[8 * hb + u].y + by;   // G_r - m
                amax = fmaxf(amax, fmaxf(fabsf(xx), fabsf(xy)));
                const float ex = exp2f(xx), ey = exp2f(xy);
                const float ix = rcp_approx(ex), iy = rcp_approx(ey);
                const float2 kv = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&kq[8 * hb + u]));
                const float2 qv = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&qq[8 * hb + u]));
                *reinterpret_cast<uint32_t *>(r1 + sw128(r, pc0, 2 * C)) = pack_h2(kv.x * ex, kv.y * ey);
                *reinterpret_cast<uint32_t *>(r1 + sw128(C + r, pc0, 2 * C)) = pack_h2(qv.x * ex, qv.y * ey);
                const float b0 = kv.x * ix, b1 = kv.y * iy;
                *reinterpret_cast<uint32_t *>(r2 + sw128(r, pc0, C)) = pack_h2(b0, b1);
                khx[u] = b0 * fx;
                khy[u] = b1 * fy;
            }
            const int r0 = 16 * pE + 8 * hb;
            *reinterpret_cast<uint4 *>(kht + sw128(pc0, r0, KD)) =
                make_uint4(pack_h2(khx[0], khx[1]), pack_h2(khx[2], khx[3]),
                           pack_h2(khx[4], khx[5]), pack_h2(khx[6], khx[7]));
            *reinterpret_cast<uint4 *>(kht + sw128(pc0 + 1, r0, KD)) =
                make_uint4(pack_h2(khy[0], khy[1]), pack_h2(khy[2], khy[3]),
                           pack_h2(khy[4], khy[5]), pack_h2(khy[6], khy[7]));
        }
        // v as fp16 (the B operand of U = T Diag(beta) v), rows of this thread
#pragma unroll
        for (int u = 0; u < 16; ++u) {
            const int r = 16 * pE + u;
            const uint32_t vv = r < len ? __ldg(reinterpret_cast<const unsigned int *>(vin + ((t0 + r) * H + h) * VD + pc0)) : 0u;
            const float2 vf = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&vv));
            *reinterpret_cast<uint32_t *>(r3 + sw128(r, pc0, C)) = pack_h2(vf.x, vf.y);
        }
        // largest G of the chunk (for M) and the fast-path test: every 2^(G_r - m) in [2^-8, 2^8]
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) gmx = fmaxf(gmx, __shfl_xor_sync(0xffffffffu, gmx, o));
        if (lane == 0) wmax[gw] = gmx;
        if (__any_sync(0xffffffffu, !(amax <= 0.5f * kSpanMax)) && lane == 0) *xflag = 1;
        fence_proxy_async_smem();   // the operands are read by tcgen05
        named_bar_sync(bar_id, kGroup);
        const bool exact_path = *xflag != 0;
        {   // M = max(0, ceil(max G) - 8); 2^(m - M) per channel and hs = 2^M
            float gm = wmax[0];
#pragma unroll
            for (int i = 1; i < 8; ++i) gm = fmaxf(gm, wmax[i]);
            const float M = fmaxf(0.f, ceilf(gm) - 8.f);
            if (pE == 0) *reinterpret_cast<float2 *>(pms + pc0) = make_float2(exp2f(mx_ - M), exp2f(my_ - M));
            if (gtid == 0) *hsp = exp2f(M);
        }

        if (!exact_path) {
            // ---------------- MMA A: [A_kk'; A_qk'] = [a_k; a_q] b^T into columns 0..63
            if (gtid == 0) {
                tc_fence_after();
#pragma unroll
                for (int ks = 0; ks < KD / 16; ++ks)
                    umma_f16(tg, sw128_kdesc(smem_u32(r1), ks, 2 * C), sw128_kdesc(smem_u32(r2), ks, C),
                             kIdescM128N64, ks > 0);
                umma_commit(barA);
            }
            a_pending = true;
            const bool ok = mbar_wait_t(barA, a_par, wp);
            if (bar_red_or(bar_id, kGroup, !ok)) { failed = true; break; }
            a_par ^= 1u;
            a_pending = false;
            tc_fence_after();
            // ---------------- A epilogue: lanes 0..63 A_kk (beta-scaled, strict lower),
            //                  64..127 A_qk (lower); warp: lane quadrant, 32 columns
            const int c0 = 32 * ((gw >> 2) & 1), rg = 32 * (warp & 3) + lane;
            float av[32];
            tmem_ld32(tg + lane_off + c0, av);
            const bool kk = rg < C;
            const int r = kk ? rg : rg - C;
            const float sb = kk ? bs[r] : 1.f;
            const int lim = kk ? r : r + 1;   // columns i < lim are kept
            __half *dst = kk ? akk : aqk;
#pragma unroll
            for (int t = 0; t < 4; ++t) {
                uint32_t wv[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int e = 8 * t + 2 * u, i = c0 + e;
                    wv[u] = pack_h2(i < lim ? sb * av[e] : 0.f, i + 1 < lim ? sb * av[e + 1] : 0.f);
                }
                *reinterpret_cast<uint4 *>(dst + sw128(r, c0 + 8 * t, C)) = make_uint4(wv[0], wv[1], wv[2], wv[3]);
            }
            tc_fence_before();
        } else {
            // ---------------- exact path: G (fp32) to the ring entry as scratch, once it is free
            bool ok = true;
            if (gtid == 0 && want_free > 0) ok = flag_wait(consumed, want_free, wp);
            if (bar_red_or(bar_id, kGroup, !ok)) { failed = true; break; }
            float *Gs = reinterpret_cast<float *>(rec);
#pragma unroll
            for (int u = 0; u < 16; ++u) {
                const int r = 16 * pE + u;
                *reinterpret_cast<float2 *>(Gs + r * KD + pc0) = make_float2(gx[u].x + pre.x, gx[u].y + pre.y);
            }
            named_bar_sync(bar_id, kGroup);
            exact_pairs(a, t0, len, h, Gs, bs, akk, aqk, kht, gtid);
        }
        named_bar_sync(bar_id, kGroup);   // A_kk, A_qk complete; a_q no longer read by MMA A

        // ---------------- Q~ = a_q 2^(m - M) in place (rows 64..127 of [a_k; a_q])
        {
            const int r = C + (gtid >> 2), cq = 32 * (gtid & 3);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                uint4 *pp = reinterpret_cast<uint4 *>(r1 + sw128(r, cq + 8 * j, 2 * C));
                uint4 x = *pp;
                __half2 *hx = reinterpret_cast<__half2 *>(&x);
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const float2 f = __half22float2(hx[u]);
                    const int c = cq + 8 * j + 2 * u;
                    hx[u] = __floats2half2_rn(f.x * pms[c], f.y * pms[c + 1]);
                }
                *pp = x;
            }
        }
        // ---------------- T = (I + A_kk)^-1: the diagonal blocks, then the column blocks
        if (gw == 0 || gw == 1) invert_diag_blocks(akk, tmh, gw, lane);
        named_bar_sync(bar_id, kGroup);
        if (gw == 2) solve_column_block(akk, tmh, 0, lane);
        else if (gw == 3) solve_column_block(akk, tmh, 1, lane);
        else if (gw == 4) solve_column_block(akk, tmh, 2, lane);
        named_bar_sync(bar_id, kGroup);
        // T Diag(beta) (zeros above its diagonal blocks) -> rows 0..63 of the r2 tile
        for (int e = gtid; e < C * C / 8; e += kGroup) {
            const int r = e >> 3, jj = e & 7;
            uint4 x = make_uint4(0, 0, 0, 0);
            if ((jj >> 1) <= (r >> 4)) {
                x = *reinterpret_cast<const uint4 *>(tmh + r * LD64 + 8 * jj);
                __half2 *hx = reinterpret_cast<__half2 *>(&x);
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const float2 f = __half22float2(hx[u]);
                    hx[u] = __floats2half2_rn(f.x * bs[8 * jj + 2 * u], f.y * bs[8 * jj + 2 * u + 1]);
                }
            }
            *reinterpret_cast<uint4 *>(r2 + sw128(r, 8 * jj, 2 * C)) = x;
        }
        fence_proxy_async_smem();
        named_bar_sync(bar_id, kGroup);

        // ---------------- MMA W, U: (T Diag(beta)) [a_k | v] into columns 0..127 | 128..255
        if (gtid == 0) {
            tc_fence_after();
#pragma unroll
            for (int ks = 0; ks < C / 16; ++ks)
                umma_f16(tg, sw128_kdesc(smem_u32(r2), ks, 2 * C),
                         sw128_mn_desc(smem_u32(r1) + 2048u * ks, 2 * C * 128), kIdescM128N128Bmn, ks > 0);
#pragma unroll
            for (int ks = 0; ks < C / 16; ++ks)
                umma_f16(tg + 128, sw128_kdesc(smem_u32(r2), ks, 2 * C),
                         sw128_mn_desc(smem_u32(r3) + 2048u * ks, C * 128), kIdescM128N128Bmn, ks > 0);
            umma_commit(barW);
        }
        w_pending = true;
        {
            const bool ok = mbar_wait_t(barW, w_par, wp);
            if (bar_red_or(bar_id, kGroup, !ok)) { failed = true; break; }
        }
        w_par ^= 1u;
        w_pending = false;
        tc_fence_after();
        // ---------------- W (x 2^(m - M)) and U to fp16, rows 0..63 (warps of lane quadrants 0, 1)
        if ((warp & 2) == 0) {
            const int r = 32 * (warp & 1) + lane, half = (gw >> 2) & 1;
#pragma unroll
            for (int part = 0; part < 2; ++part) {
                const int cb = 64 * half + 32 * part;
                float x[32];
                tmem_ld32(tg + lane_off + cb, x);
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    uint32_t wv[4];
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const int e = 8 * j + 2 * u;
                        wv[u] = pack_h2(x[e] * pms[cb + e], x[e + 1] * pms[cb + e + 1]);
                    }
                    *reinterpret_cast<uint4 *>(r1 + sw128(r, cb + 8 * j, 2 * C)) = make_uint4(wv[0], wv[1], wv[2], wv[3]);
                }
                tmem_ld32(tg + 128 + lane_off + cb, x);
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    uint32_t wv[4];
#pragma unroll
                    for (int u = 0; u < 4; ++u) wv[u] = pack_h2(x[8 * j + 2 * u], x[8 * j + 2 * u + 1]);
                    *reinterpret_cast<uint4 *>(r3 + sw128(r, cb + 8 * j, C)) = make_uint4(wv[0], wv[1], wv[2], wv[3]);
                }
            }
        }
        tc_fence_before();
        fence_proxy_async_smem();   // the record image is read by the bulk copy
        named_bar_sync(bar_id, kGroup);

        // ---------------- publish: ring entry free -> one bulk store -> release flag
        if (gtid == 0) {
            bool ok = true;
            if (!exact_path && want_free > 0) ok = flag_wait(consumed, want_free, wp);
            if (ok) {
                fence_proxy_async_global();
                bulk_s2g(rec, smem_u32(gs), Rec::bytes);
                bulk_commit();
                bulk_wait_all();
                fence_proxy_async_global();
                st_release(wp.ready + (int64_t)s * kRing + p % kRing,
                           ((unsigned long long)wp.epoch << 32) | (unsigned long long)(p + 1));
            }   // else: the abort word is raised; the next ticket's barrier ends the loop
        }
        // (the next ticket's first barrier orders the reuse of the staging area)
    }
    if (failed || a_pending || w_pending) {
        if (gtid == 0) {
            if (a_pending) mbar_drain(barA, a_par);
            if (w_pending) mbar_drain(barW, w_par);
        }
    }
    if (gtid == 0) bulk_wait_all();
    named_bar_sync(bar_id, kGroup);
}

// =====================================================================================
// Scanner: the serial chain of every work item w = s, s + S, ... of scanner s.  Warp 15
// also moves the records in: part A of position p + 2 once chunk p's D step is done
// (waiting for the builder's flag), part B of position p + 1 once chunk p - 1's S3 is.
// =====================================================================================
template <typename Tout>
__device__ __forceinline__ void scanner(const PrefillArgs &a, const WyParams &wp, unsigned char *sm,
                                     uint32_t tmem)
{
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int s = blockIdx.x, S = wp.S;
    const int H = a.num_heads;
    const int64_t NH = (int64_t)a.num_seqs * H;
    auto bar = [&](int b) { return smem_u32(sm + Ssm::bars + 8 * b); };
    const unsigned char *ring = wp.rec + (int64_t)s * kRing * Rec::bytes;
    const bool mover = warp == kMoverWarp;

    // positions of this scanner (chunks of its items)
    int64_t total = 0;
    for (int64_t wi = s; wi < NH; wi += S) {
        int64_t b, e;
        item_range(a, wi, b, e);
        total += (e - b + C - 1) / C;
    }
    // record movement (warp 15; lane 0 issues): part A waits for the builder's flag
    int64_t nA = 0, nB = 0;   // positions whose part A / part B has been issued
    auto issueA = [&]() -> bool {
        bool ok = true;
        if (lane == 0) {
            const int64_t q = nA;
            ok = flag_wait(wp.ready + (int64_t)s * kRing + q % kRing, (uint32_t)(q + 1), wp);
            if (ok) {
                fence_proxy_async_global();
                const uint32_t fb = bar(SBar::full + (int)(q & 1));
                mbar_arrive_expect_tx(fb, Rec::bytes);
                bulk_g2s(smem_u32(sm + (int)(q & 1) * Ssm::slot), ring + (q % kRing) * Rec::bytes, Rec::partA, fb);
            }
        }
        ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
        if (ok) ++nA;
        return ok;
    };
    auto issueB = [&]() {
        if (lane == 0) {
            const int64_t q = nB;
            bulk_g2s(smem_u32(sm + (int)(q & 1) * Ssm::slot) + Rec::partA,
                     ring + (q % kRing) * Rec::bytes + Rec::partA, Rec::bytes - Rec::partA,
                     bar(SBar::full + (int)(q & 1)));
        }
        __syncwarp();
        ++nB;
    };
    bool mfail = false;   // the mover's flag wait failed (reported at the next barrier)
    if (mover)
        for (int i = 0; i < 2 && nA < total && !mfail; ++i) {
            if (issueA()) issueB();
            else mfail = true;
        }

    // copy step: warp w holds key channel c = 32 (w % 4) + lane, value columns [32 (w / 4), +32);
    // D step (warps of lane quadrants 0, 1): row r = 32 (w % 4) + lane; output (quadrants 2, 3):
    // row r = 32 (w % 4 - 2) + lane; both over value columns [32 (w / 4), +32).
    const int q4 = warp & 3, cg = warp >> 2;
    const int c = 32 * q4 + lane;
    const uint32_t lane_off = (uint32_t)(32 * q4) << 16;
    const uint32_t tH = tmem, tAcc = tmem + 128;   // h: lane = key channel; acc[par] at +128 par
    __half *ht = reinterpret_cast<__half *>(sm + Ssm::ht);
    __half *dtl = reinterpret_cast<__half *>(sm + Ssm::dt);
    Tout *out = static_cast<Tout *>(a.out);

    int64_t p = 0;
    bool fail = false;
    int64_t n_s1 = 0, n_s3 = 0;   // MMA batches issued (thread 0)
    bool pend = false;            // output rows of chunk p - 1 not yet stored
    int pend_len = 0, pend_h = 0;
    int64_t pend_t0 = 0;

    for (int64_t wi = s; wi < NH && !fail; wi += S) {
        const int64_t n = wi / H;
        const int h = (int)(wi % H);
        int64_t bos, eos;
        item_range(a, wi, bos, eos);
        const float *init;
        float *fin;
        prefill_state_ptrs(a, n, h, init, fin);
        {   // initial state -> tensor memory
            float hv[32];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const float4 x = init ? *reinterpret_cast<const float4 *>(init + (int64_t)c * VD + 32 * cg + 4 * j)
                                      : make_float4(0.f, 0.f, 0.f, 0.f);
                hv[4 * j] = x.x; hv[4 * j + 1] = x.y; hv[4 * j + 2] = x.z; hv[4 * j + 3] = x.w;
            }
            tmem_st32(tH + lane_off + 32 * cg, hv);
        }
        for (int64_t t0 = bos; t0 < eos; t0 += C, ++p) {
            const int len = (int)((eos - t0) < C ? (eos - t0) : C);
            const int sl = (int)(p & 1);
            const unsigned char *slot = sm + sl * Ssm::slot;
            const uint32_t par = (uint32_t)(p & 1);
            const uint32_t tA = tAcc + 128u * (uint32_t)sl;
            // both parts of record p were issued before this point (or the mover failed)
            const bool ok = !mfail && mbar_wait_t(bar(SBar::full + sl), (uint32_t)((p >> 1) & 1), wp);
            if (ok && tid == 0)
                st_release(wp.consumed + 8 * (int64_t)s, ((unsigned long long)wp.epoch << 32) | (unsigned long long)(p + 1));
            tc_fence_after();
            // ---------------- copy: h16 = fp16(hs h) (MN-major: row = channel), h <- 2^G_last h
            {
                const float d = reinterpret_cast<const float *>(slot + Rec::dec)[c];
                const float hs = *reinterpret_cast<const float *>(slot + Rec::hs);
                float hv[32];
                tmem_ld32(tH + lane_off + 32 * cg, hv);
                if (hs != 1.f) {
#pragma unroll
                    for (int v = 0; v < 32; ++v) hv[v] *= hs;
                }
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    *reinterpret_cast<uint4 *>(ht + sw128(c, 32 * cg + 8 * j, KD)) =
                        make_uint4(pack_h2(hv[8 * j], hv[8 * j + 1]), pack_h2(hv[8 * j + 2], hv[8 * j + 3]),
                                   pack_h2(hv[8 * j + 4], hv[8 * j + 5]), pack_h2(hv[8 * j + 6], hv[8 * j + 7]));
                const float dd = hs != 1.f ? d / hs : d;
#pragma unroll
                for (int v = 0; v < 32; ++v) hv[v] *= dd;
                tmem_st32(tH + lane_off + 32 * cg, hv);
            }
            fence_proxy_async_smem();
            tc_fence_before();
            if (bar_red_or(kBarChain, kChain, !ok)) { fail = true; break; }

            // ---------------- S1: acc = [W; Q~] h16
            if (tid == 0) {
                tc_fence_after();
#pragma unroll
                for (int ks = 0; ks < KD / 16; ++ks)
                    umma_f16(tA, sw128_kdesc(smem_u32(slot + Rec::aop), ks, 2 * C),
                             sw128_mn_desc(smem_u32(ht) + 2048u * ks, KD * 128), kIdescM128N128Bmn, ks > 0);
                umma_commit(bar(SBar::s1));
                ++n_s1;
            }
            bool ok2 = true;
            if ((warp & 2) == 0) {
                // ---------------- D = U - W h -> fp16 (rows 0..63)
                ok2 = mbar_drain(bar(SBar::s1), par);
                tc_fence_after();
                const int r = c;   // lanes 0..63
                float x[32];
                tmem_ld32(tA + lane_off + 32 * cg, x);
                const __half *uu = reinterpret_cast<const __half *>(slot + Rec::u);
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    uint4 uv = *reinterpret_cast<const uint4 *>(uu + sw128(r, 32 * cg + 8 * j, C));
                    const __half2 *u2 = reinterpret_cast<const __half2 *>(&uv);
                    uint32_t wv[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float2 f = __half22float2(u2[e]);
                        wv[e] = pack_h2(f.x - x[8 * j + 2 * e], f.y - x[8 * j + 2 * e + 1]);
                    }
                    *reinterpret_cast<uint4 *>(dtl + sw128(r, 32 * cg + 8 * j, C)) = make_uint4(wv[0], wv[1], wv[2], wv[3]);
                }
                tc_fence_before();
            } else if (pend) {
                // ---------------- output rows of chunk p - 1 (rows 64..127 of its accumulator)
                const uint32_t ppar = (uint32_t)((p - 1) & 1);
                ok2 = mbar_drain(bar(SBar::s3o), ppar);
                tc_fence_after();
                const int r = 32 * (q4 - 2) + lane;
                float o[32];
                tmem_ld32(tAcc + 128u * ppar + lane_off + 32 * cg, o);
                if (r < pend_len) {
                    Tout *dst = out + ((pend_t0 + r) * H + pend_h) * VD + 32 * cg;
                    store_row16(dst, *reinterpret_cast<float (*)[16]>(&o[0]), a.scale);
                    store_row16(dst + 16, *reinterpret_cast<float (*)[16]>(&o[16]), a.scale);
                }
                tc_fence_before();
                // S3 of chunk p - 1 is complete: part B of position p + 1 may replace its operands
                if (mover && nB < nA) issueB();
            }
            fence_proxy_async_smem();
            if (bar_red_or(kBarChain, kChain, !ok2)) { fail = true; break; }
            pend = false;

            // ---------------- S3: h += K^^T D ; acc rows 64..127 += A_qk D
            if (tid == 0) {
                tc_fence_after();
#pragma unroll
                for (int ks = 0; ks < C / 16; ++ks)
                    umma_f16(tH, sw128_kdesc(smem_u32(slot + Rec::kht), ks, KD),
                             sw128_mn_desc(smem_u32(dtl) + 2048u * ks, C * 128), kIdescM128N128Bmn, 1u);
                umma_commit(bar(SBar::s3h));
#pragma unroll
                for (int ks = 0; ks < C / 16; ++ks)
                    umma_f16(tA, sw128_kdesc(smem_u32(slot + Rec::kht + 8192), ks, KD),
                             sw128_mn_desc(smem_u32(dtl) + 2048u * ks, C * 128), kIdescM128N128Bmn, 1u);
                umma_commit(bar(SBar::s3o));
                ++n_s3;
            }
            // part A of this slot (copy step, S1, D step) is no longer read: position p + 2
            if (mover && nA < total && nA == p + 2 && !mfail && !issueA()) mfail = true;
            pend = true;
            pend_t0 = t0;
            pend_len = len;
            pend_h = h;
            if (!mbar_drain(bar(SBar::s3h), par)) fail = true;   // h is final for the next copy
            tc_fence_after();
        }
        fail = bar_red_or(kBarChain, kChain, fail || mfail);
        if (!fail && fin) {   // final state
            float hv[32];
            tmem_ld32(tH + lane_off + 32 * cg, hv);
#pragma unroll
            for (int j = 0; j < 8; ++j)
                *reinterpret_cast<float4 *>(fin + (int64_t)c * VD + 32 * cg + 4 * j) =
                    make_float4(hv[4 * j], hv[4 * j + 1], hv[4 * j + 2], hv[4 * j + 3]);
        }
        tc_fence_before();
    }
    if (!fail && pend && (warp & 2) != 0) {   // the last chunk's output rows
        const uint32_t ppar = (uint32_t)((p - 1) & 1);
        mbar_drain(bar(SBar::s3o), ppar);
        tc_fence_after();
        const int r = 32 * (q4 - 2) + lane;
        float o[32];
        tmem_ld32(tAcc + 128u * ppar + lane_off + 32 * cg, o);
        if (r < pend_len) {
            Tout *dst = out + ((pend_t0 + r) * H + pend_h) * VD + 32 * cg;
            store_row16(dst, *reinterpret_cast<float (*)[16]>(&o[0]), a.scale);
            store_row16(dst + 16, *reinterpret_cast<float (*)[16]>(&o[16]), a.scale);
        }
    }
    if (fail && tid == 0) {   // MMAs in flight finish before the tensor memory is released
        if (n_s1 > 0) mbar_drain(bar(SBar::s1), (uint32_t)((n_s1 - 1) & 1));
        if (n_s3 > 0) {
            mbar_drain(bar(SBar::s3h), (uint32_t)((n_s3 - 1) & 1));
            mbar_drain(bar(SBar::s3o), (uint32_t)((n_s3 - 1) & 1));
        }
    }
    named_bar_sync(kBarChain, kChain);
    if (mover) {   // no copy may be in flight when the CTA exits
        while (nB < nA) issueB();
        if (lane == 0)
            for (int64_t q = nA > 2 ? nA - 2 : 0; q < nA; ++q)
                mbar_drain(bar(SBar::full + (int)(q & 1)), (uint32_t)((q >> 1) & 1));
        __syncwarp();
    }
    tc_fence_before();
}

template <typename Tout>
__global__ void __launch_bounds__(kThreads, 1)
kda_prefill_wy_kernel(const PrefillArgs a, const WyParams wp)
{
    extern __shared__ __align__(1024) unsigned char sm[];
    const int tid = threadIdx.x, warp = tid >> 5;
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n"
                     :: "r"(smem_u32(sm + kTmemSlot)), "r"(512) : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n" ::: "memory");
    }
    const bool is_scanner = (int)blockIdx.x < wp.S;
    if (tid == 0) {
        if (is_scanner) {
            for (int b = 0; b < SBar::count; ++b) mbar_init(smem_u32(sm + Ssm::bars + 8 * b), 1);
        } else {
            for (int g = 0; g < 2; ++g)
                for (int b = 0; b < 2; ++b) mbar_init(smem_u32(sm + Gsm::group * g + Gsm::bars + 8 * b), 1);
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(sm + kTmemSlot);
    if (is_scanner) scanner<Tout>(a, wp, sm, tmem);
    else builder(a, wp, sm, tmem);
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" :: "r"(tmem), "r"(512) : "memory");
    }
}

// ------------------------------------------------------------------ host side
struct Layout {
    size_t consumed, ready, rec, total;
};

constexpr Layout layout_for(int S)
{
    return Layout{128, 128 + (size_t)S * 64,
                  (128 + (size_t)S * 64 + (size_t)S * kRing * 8 + 1023) / 1024 * 1024,
                  (128 + (size_t)S * 64 + (size_t)S * kRing * 8 + 1023) / 1024 * 1024 +
                      (size_t)S * kRing * Rec::bytes};
}
static_assert(layout_for(kScanMax).total == wy_workspace_bytes_for(kScanMax) &&
              layout_for(3).total == wy_workspace_bytes_for(3), "workspace layout");

int scanners_for(int64_t num_seqs, int32_t num_heads)
{
    const int64_t nh = num_seqs * (int64_t)num_heads;
    return (int)(nh < kScanMax ? nh : kScanMax);
}

std::atomic<unsigned int> g_epoch{0};
std::atomic<unsigned long long> g_wait_ns{2000000000ull};

template <typename Tout>
cudaError_t launch_wy_t(const PrefillArgs &a, void *ws, cudaStream_t stream)
{
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(kda_prefill_wy_kernel<Tout>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemTotal);
    if (e != cudaSuccess) return e;
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kda_prefill_wy_kernel<Tout>, kThreads, kSmemTotal);
    if (e != cudaSuccess) return e;
    const int64_t resident = (int64_t)per_sm * sms;
    const int S_ws = scanners_for(a.num_seqs, a.num_heads);
    int S = S_ws;
    if (resident < 2) return cudaErrorInvalidConfiguration;
    if (S > resident - 1) S = (int)(resident - 1);
    // builder CTAs: no more than the chunks can use (two units each, at most a ring ahead)
    const int64_t chunk_bound = (int64_t)a.num_heads * (a.total_tokens / C + a.num_seqs);
    int64_t units = chunk_bound < (int64_t)(kRing + 1) * S ? chunk_bound : (int64_t)(kRing + 1) * S;
    int64_t nb = (units + 1) / 2;
    if (nb < 1) nb = 1;
    if (nb > resident - S) nb = resident - S;
    const Layout l = layout_for(S_ws);
    unsigned char *base = static_cast<unsigned char *>(ws);
    WyParams wp;
    wp.rec = base + l.rec;
    wp.ready = reinterpret_cast<unsigned long long *>(base + l.ready);
    wp.consumed = reinterpret_cast<unsigned long long *>(base + l.consumed);
    wp.abort_word = reinterpret_cast<unsigned long long *>(base + 64);
    wp.status = reinterpret_cast<int *>(base);
    wp.wait_ns = g_wait_ns.load();
    unsigned int ep = ++g_epoch;
    if (ep == 0) ep = ++g_epoch;
    wp.epoch = ep;
    wp.S = S;

    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(S + nb));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemTotal;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, kda_prefill_wy_kernel<Tout>, a, wp);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace

bool prefill_wy_supported(const PrefillArgs &a)
{
    return a.dtype == kDtypeBF16 && a.head_dim_k == KD && a.head_dim_v == VD;
}

size_t prefill_wy_workspace_bytes(int64_t num_seqs, int32_t num_heads)
{
    if (num_seqs <= 0 || num_heads < 1) return 0;
    return layout_for(scanners_for(num_seqs, num_heads)).total;
}

cudaError_t launch_prefill_wy(const PrefillArgs &a, void *workspace, cudaStream_t stream)
{
    if (a.num_seqs == 0) return cudaSuccess;
    return a.out_dtype == kDtypeBF16 ? launch_wy_t<__nv_bfloat16>(a, workspace, stream)
                                     : launch_wy_t<float>(a, workspace, stream);
}

void set_prefill_wait_limit_ns(unsigned long long ns)
{
    g_wait_ns.store(ns == 0 ? 2000000000ull : ns);
}

}  // namespace kda
