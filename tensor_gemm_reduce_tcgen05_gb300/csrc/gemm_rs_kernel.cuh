// The fused GEMM + reduce-scatter kernels for sm_103a.
//
// Persistent CTAs walk the global tile order of schedule.cuh.  Each work item
// is one rank-tile (r, mt, nt): an output tile of logical rank r's GEMM
// A_r * B_r over its K/W shard.  Two kernels share the roles below:
//   gemm_rs_fused_kernel<BN>   one CTA per 128 x BN tile, tcgen05.mma with
//                              M = 128 (cta_group::1); one CTA per SM.
//   gemm_rs_pair_kernel<256>   a cluster of two CTAs per 256 x 256 tile,
//                              tcgen05.mma with M = 256 (cta_group::2); each
//                              CTA loads its own 128 rows of A and 128 columns
//                              of B (no multicast) and drains its own half.
//
// Warp roles (320 threads):
//   warp 0      TMA producer (one thread).  For each k-block it loads the A_r
//               box [128 x 64] and the B_r tile [64 x BN] (one 4D box of BN/64
//               64-column atoms, or one 3D box per atom when N is not a
//               multiple of 64) into a stage of the shared-memory ring,
//               128-byte swizzled, completing the stage's `full` mbarrier.  In
//               a host-streamed call it first waits for rank r's ready word.
//   warp 1      TMEM allocator and MMA issuer (one thread).  It issues
//               tcgen05.mma (bf16 -> fp32) into one of two TMEM accumulators;
//               tcgen05.commit frees each stage and, at the end of the tile,
//               signals `acc_full`.
//   warps 2-5   epilogue visitor.  Each warp drains 32 TMEM lanes (one row per
//               thread) and computes p = alpha*acc + beta*C
//               ("flux实现：sm80 gemm+rs", section "custom_evt_d()").  Where p
//               goes is the reduce mode's (run_epilogue):
//                 LAST_ARRIVER  p is stored in the tile's rank-r slot of the
//                               chunk workspace ("evt_store_d()": the store
//                               goes to the reduce-scatter buffer, not to Y);
//                               the rank that arrives last on the tile's
//                               32-bit counter resets it and queues the tile.
//                 CHAIN         p is added onto the tile's running sum when
//                               its turn comes (or stored, and folded on by
//                               whoever holds the fold); the last position
//                               writes Y.
//                 TWO_LEVEL     CHAIN within each of two rank groups; the
//                               group that finishes second adds the two sums.
//   warps 6-9   LAST_ARRIVER: reducers, folding each queued tile's W partials
//               in rank order and writing Y beside the epilogue (a reduction
//               never holds a TMEM accumulator).  CHAIN and TWO_LEVEL: a second
//               epilogue group (each of the eight warps drains half of its lane
//               quarter's column slabs).
//
// Waits between CTAs: LAST_ARRIVER has none (the last arriver waits for no one,
// so the kernel cannot deadlock however many CTAs it has; the deadlock of a
// device-wide barrier with more CTAs than fit at once is described in
// "flux实现：sm80 gemm+rs", section "device side barrier").  CHAIN has one,
// bounded: a position may wait a few thousand cycles for the position before
// it, which lies earlier in the tile order, so the waits form no cycle.
// Every mbarrier wait, and every wait for a streamed call's ready word, is
// bounded in SM cycles too.  A wait that runs out
// records a code in the status word, and the CTA drains its TMA loads and
// MMAs, frees TMEM and exits.
//
// Partial slot layout: slot (tile, s) holds 4 x (BN/32) blocks of 32 rows x 32
// columns (fp32).  Inside a block, float4 j (columns 4j .. 4j+3) of row t is
// at float4 index j*32 + t, so each warp-wide 16-byte store or load covers 512
// contiguous bytes.  Slots are ordered by row tile, so the slots of the tiles
// keyed to one chunk form one contiguous region: the chunk's workspace.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>

#include "ptx.cuh"
#include "schedule.cuh"

namespace gemm_rs {

constexpr int kBM = 128;
constexpr int kBK = 64;
constexpr int kThreads = 320;
constexpr int kEpiWarp0 = 2;
constexpr int kRedWarp0 = 6;
constexpr int kRQ = 32;          // depth of the reduce queue (entries are quarter-tiles)
constexpr int kConsumers = 8;    // warps that take reduce jobs: 4 reducers + 4 epilogue warps
static_assert(kRQ >= 2 * kConsumers, "queue slots must outnumber consumers (parity reuse)");
constexpr uint32_t kBarEpi = 1;  // named barrier of the epilogue threads
constexpr int kMaxStages = 8;

// Status word codes (first failure wins).
enum : uint32_t {
    kStatusOk = 0,
    kStatusTimeoutProducer = 1,
    kStatusTimeoutMma = 2,
    kStatusTimeoutEpilogue = 3,
    kStatusTimeoutReducer = 4,
    kStatusOutOfBounds = 5, // checked build: an access outside its buffer was skipped
};

template <int BN>
struct TileCfg {
    static_assert(BN == 64 || BN == 128 || BN == 256, "BN must be 64, 128 or 256");
    static constexpr int kABytes = kBM * kBK * 2;            // 16 KB
    static constexpr int kBBytes = BN * kBK * 2;             // BN/64 boxes of 8 KB
    static constexpr int kStageBytes = kABytes + kBBytes;
    static constexpr int kStages = BN == 256 ? 4 : (BN == 128 ? 6 : 8);
    static constexpr int kTmemCols = 2 * BN;                 // two accumulators
    static constexpr int kSlabs = BN / 32;
    static constexpr uint32_t kIdesc = ptx::idesc_bf16_f32(kBM, BN, false, true);
    static constexpr int64_t kSlotFloats = int64_t(kBM) * BN; // one partial tile
    static_assert(kStages <= kMaxStages, "too many stages");
    static_assert(kStageBytes % 1024 == 0, "stages must keep 1024-byte alignment");
};

// CTA-pair variant: a 256 x BN output tile per cluster of two CTAs.  Each CTA
// loads its own 128 rows of A and its own BN/2 columns of B (no multicast),
// and the even CTA issues tcgen05.mma.cta_group::2 with M = 256.
template <int BN>
struct PairCfg {
    static_assert(BN == 256, "the pair kernel uses 256-column tiles");
    static constexpr int kABytes = kBM * kBK * 2;            // own 128 rows
    static constexpr int kBBytes = (BN / 2) * kBK * 2;       // own BN/2 columns
    static constexpr int kStageBytes = kABytes + kBBytes;    // 32 KB
    // 7 x 32 KB: all of the shared memory but the control block (measured
    // against 6 stages: 2-3 % faster on the large workloads)
    static constexpr int kStages = 7;
    static constexpr int kTmemCols = 2 * BN;
    static constexpr uint32_t kIdesc = ptx::idesc_bf16_f32(2 * kBM, BN, false, true);
    static_assert(kStageBytes % 1024 == 0, "stages must keep 1024-byte alignment");
};

struct KernelArgs {
    int W, M, N, nM, nN, nK;
    int nMs;        // row tiles of the schedule (nM, or ceil(M/256) for CTA pairs)
    int colgroup;   // column tiles per schedule group (>= nN: one group)
    int rowgroup;   // row tiles per sweep (>= a chunk's row tiles: one sweep per step)
    int chain;      // 1: chain reduction (in-order fold as tiles land), 0: last arriver reduces
    int seq;        // 1: the ranks' tiles one rank after another, 0: the ranks side by side
    long long chain_wait; // SM cycles a chain position waits for its turn before storing
    int split;      // chain mode, two-level fold: ranks [0, split) and [split, W) fold
                    // separately, then the two sums are added (0: one fold over all W)
    int64_t part_floats; // floats in the partial slots, and state words: the buffers'
    int64_t nflags;      // extents, for the checked build's bounds checks
    int64_t R;      // rows per chunk
    int64_t total;  // W * nM * nN work items
    float alpha, beta;
    const uint16_t *C; // bf16 bits, NULL when beta == 0
    void *Y;
    int y_fp32;
    float *part;
    uint32_t *flags;
    uint32_t *status;
    int32_t *record;
    unsigned long long timeout;
    int stall_producer;
    int b4d;        // 1: the B tensor map is 4D (one load per stage), 0: 3D (one per 64 columns)
    // Host-streamed inputs (gemm_rs_run_streamed): ready[r] reaches `epoch` once
    // rank r's A_r and B_r have landed, ready[W] once C has; NULL otherwise.
    const uint32_t *ready;
    uint32_t epoch;
};

struct SmemCtl {
    uint64_t full[kMaxStages];
    uint64_t empty[kMaxStages];
    uint64_t acc_full[2];
    uint64_t acc_empty[2];
    uint64_t rq_full[kRQ];
    uint64_t rq_empty[kRQ];
    uint64_t drain;
    uint64_t peer_drained; // CTA pairs: the odd CTA's loads have landed (the even CTA arrives)
    int32_t rq_tile[kRQ];
    uint32_t rq_head; // next queue entry to claim
    int epi_direct[2]; // chain mode: the epilogue owns the fold of the tile in TMEM buffer b
    int epi_fold;      // chain mode: position the epilogue folds on from (-1: none)
    int epi_fold_end;  // chain mode: last stored position of the current fold
    uint32_t epi_seen; // chain mode: the state word as the fold's owner last saw it
    int epi_combine;   // two-level fold: this CTA adds the two groups' sums into Y
    uint32_t tmem_base;
    int abort;
};

template <int BN>
constexpr int smem_bytes()
{
    return 1024 + TileCfg<BN>::kStages * TileCfg<BN>::kStageBytes + int(sizeof(SmemCtl));
}

template <int BN>
constexpr int smem_bytes_pair()
{
    return 1024 + PairCfg<BN>::kStages * PairCfg<BN>::kStageBytes + int(sizeof(SmemCtl));
}
static_assert(smem_bytes_pair<256>() <= 232448, "the pair kernel's shared memory exceeds 227 KB");

// Checked build (compiled with GEMM_RS_CHECKED): the global accesses of the
// epilogue and the folds are tested against their buffers first.  An access
// outside its buffer is skipped, and the first one is recorded in the status
// word.  In the normal build every check is the constant true.
__device__ __forceinline__ bool bounds_ok(const KernelArgs &a, bool ok)
{
#ifdef GEMM_RS_CHECKED
    if (!ok)
        atomicCAS(a.status, 0u, static_cast<uint32_t>(kStatusOutOfBounds));
    return ok;
#else
    (void)a;
    (void)ok;
    return true;
#endif
}

// [p, p + n) lies in the partial slots.
__device__ __forceinline__ bool in_part(const KernelArgs &a, const float *p, int64_t n)
{
#ifdef GEMM_RS_CHECKED
    const int64_t off = p - a.part;
    return bounds_ok(a, off >= 0 && off + n <= a.part_floats);
#else
    (void)p;
    (void)n;
    return bounds_ok(a, true);
#endif
}

// Columns [n, n + 8) of row m lie in Y and C ([M][N]).
__device__ __forceinline__ bool in_mn(const KernelArgs &a, int64_t m, int64_t n)
{
    return bounds_ok(a, m >= 0 && m < a.M && n >= 0 && n + 8 <= a.N);
}

// A state word lies in the flags.
__device__ __forceinline__ bool in_flags(const KernelArgs &a, const uint32_t *f)
{
    return bounds_ok(a, f >= a.flags && f - a.flags < a.nflags);
}

__device__ __forceinline__ void report(const KernelArgs &a, SmemCtl *ctl, uint32_t code)
{
    // The first role to fail records its code.  Roles that fail only because
    // another role aborted leave the code alone.
    if (*reinterpret_cast<volatile int *>(&ctl->abort) == 0)
        atomicCAS(a.status, 0u, code);
    *reinterpret_cast<volatile int *>(&ctl->abort) = 1;
}

// Host-streamed inputs: wait until the ready word *p has reached `epoch`
// (compared modulo 2^32), with acquire semantics, so that the copy it follows
// is visible.  Bounded by `limit` SM cycles; false when it runs out or the CTA
// aborts.
__device__ __forceinline__ bool wait_ready(const uint32_t *p, uint32_t epoch,
                                           unsigned long long limit, const volatile int *abort)
{
    const long long t0 = clock64();
    while (static_cast<int32_t>(ptx::ld_acquire_gpu(p) - epoch) < 0) {
        if (*abort != 0 || static_cast<unsigned long long>(clock64() - t0) > limit)
            return false;
        __nanosleep(256);
    }
    return true;
}

// Before a producer loads rank r's operands: with host-streamed inputs, wait
// for rank r's copy once (a bit per rank remembers it), then order the copy's
// writes before the TMA reads (async proxy).
__device__ __forceinline__ bool operands_ready(const KernelArgs &a, int r, uint32_t &seen,
                                               const volatile int *abort)
{
    if (a.ready == nullptr || ((seen >> r) & 1u))
        return true;
    if (!wait_ready(a.ready + r, a.epoch, a.timeout, abort))
        return false;
    asm volatile("fence.proxy.async.global;" ::: "memory");
    seen |= 1u << r;
    return true;
}

// Epilogue threads: warps 2-5, or warps 2-9 in the chain mode (which has no
// reduce jobs for warps 6-9 to take).
__device__ __forceinline__ int epi_threads(const KernelArgs &a) { return a.chain ? 256 : 128; }

// ------------------------------------------------------------------ producer
template <int BN>
__device__ __forceinline__ void run_producer(const KernelArgs &a, const Sched &sch,
                                             const CUtensorMap *tmA, const CUtensorMap *tmB,
                                             uint8_t *smem, SmemCtl *ctl)
{
    using Cfg = TileCfg<BN>;
    const volatile int *abort_flag = &ctl->abort;
    const uint64_t pol = ptx::policy_evict_normal();
    uint32_t stage = 0, phase = 0;
    int64_t issued = 0;
    bool ok = true;
    uint32_t ranks_ready = 0;
    if (!a.stall_producer) {
        for (int64_t g = blockIdx.x; g < a.total && ok; g += gridDim.x) {
            int r, mt, nt;
            decode_tile(sch, g, r, mt, nt);
            if (a.record != nullptr) {
                int32_t *rec = a.record + 4 * g;
                rec[0] = r;
                rec[1] = mt;
                rec[2] = nt;
                rec[3] = static_cast<int32_t>(blockIdx.x);
            }
            if (!operands_ready(a, r, ranks_ready, abort_flag)) {
                ok = false;
                break;
            }
            for (int kb = 0; kb < a.nK; ++kb) {
                if (!ptx::mbar_wait(ptx::smem_u32(&ctl->empty[stage]), phase ^ 1u, a.timeout,
                                    abort_flag)) {
                    ok = false;
                    break;
                }
                const uint32_t fb = ptx::smem_u32(&ctl->full[stage]);
                ptx::mbar_arrive_expect_tx(fb, Cfg::kStageBytes);
                const uint32_t sa = ptx::smem_u32(smem + stage * Cfg::kStageBytes);
                ptx::tma_load_3d(sa, tmA, fb, kb * kBK, mt * kBM, r, pol);
                if (a.b4d) {
                    ptx::tma_load_4d(sa + Cfg::kABytes, tmB, fb, 0, kb * kBK, nt * (BN / 64), r, pol);
                } else {
#pragma unroll
                    for (int j = 0; j < BN / 64; ++j)
                        ptx::tma_load_3d(sa + Cfg::kABytes + j * 8192, tmB, fb, nt * BN + j * 64,
                                         kb * kBK, r, pol);
                }
                ++issued;
                if (++stage == Cfg::kStages) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
        }
    }
    if (ok) {
        // Tail: wait until the MMA warp has released every stage, so that
        // every tcgen05.commit arrival on this CTA's barriers has landed
        // before the CTA exits.
        for (int i = 0; i < Cfg::kStages; ++i) {
            if (!ptx::mbar_wait(ptx::smem_u32(&ctl->empty[stage]), phase ^ 1u, a.timeout,
                                abort_flag)) {
                ok = false;
                break;
            }
            if (++stage == Cfg::kStages) {
                stage = 0;
                phase ^= 1u;
            }
        }
    }
    if (!ok) {
        report(a, ctl, kStatusTimeoutProducer);
        // Drain: the most recent fill of each stage must have landed before
        // the CTA's shared memory is released.
        const int64_t n = issued < Cfg::kStages ? issued : Cfg::kStages;
        for (int64_t i = 1; i <= n; ++i) {
            const int64_t pos = issued - i;
            const uint32_t s = static_cast<uint32_t>(pos % Cfg::kStages);
            const uint32_t ph = static_cast<uint32_t>((pos / Cfg::kStages) & 1);
            ptx::mbar_wait(ptx::smem_u32(&ctl->full[s]), ph, a.timeout, nullptr);
        }
    }
}

// ------------------------------------------------------------------ MMA issuer
template <int BN>
__device__ __forceinline__ void run_mma(const KernelArgs &a, uint32_t tmem, uint8_t *smem,
                                        SmemCtl *ctl)
{
    using Cfg = TileCfg<BN>;
    const volatile int *abort_flag = &ctl->abort;
    uint32_t stage = 0, phase = 0;
    bool ok = true;
    int it = 0;
    // The MMA thread's loop is on the critical path (the tensor pipe idles
    // while it prepares the next k-block), so the descriptors of stage 0 are
    // built once and moved to a stage and K step by additions.
    // A: K-major, rows of 128 bytes, 8-row groups 1024 bytes apart; K step of
    //    16 elements = 32 bytes inside the swizzle atom.
    // B: MN-major, 64-column atoms 8192 bytes apart (LBO), 8-row K groups 1024
    //    bytes apart (SBO); K step of 16 rows = 2048 bytes.
    const uint32_t s0 = ptx::smem_u32(smem);
    const uint64_t ad0 = ptx::sdesc_sw128(s0, 0, 1024);
    const uint64_t bd0 = ptx::sdesc_sw128(s0 + Cfg::kABytes, 8192, 1024);
    const uint32_t empty0 = ptx::smem_u32(&ctl->empty[0]);
    for (int64_t g = blockIdx.x; g < a.total; g += gridDim.x, ++it) {
        const int buf = it & 1;
        const uint32_t aph = static_cast<uint32_t>(it >> 1) & 1u;
        if (!ptx::mbar_wait(ptx::smem_u32(&ctl->acc_empty[buf]), aph ^ 1u, a.timeout, abort_flag)) {
            ok = false;
            break;
        }
        ptx::tc_fence_after();
        const uint32_t d = tmem + static_cast<uint32_t>(buf * BN);
        for (int kb = 0; kb < a.nK; ++kb) {
            if (!ptx::mbar_wait(ptx::smem_u32(&ctl->full[stage]), phase, a.timeout, abort_flag)) {
                ok = false;
                break;
            }
            ptx::tc_fence_after();
            const uint32_t so = stage * Cfg::kStageBytes;
#pragma unroll
            for (int kk = 0; kk < kBK / 16; ++kk)
                ptx::mma_bf16_ss(d, ptx::sdesc_advance(ad0, so + kk * 32),
                                 ptx::sdesc_advance(bd0, so + kk * 2048), Cfg::kIdesc,
                                 (kb | kk) != 0 ? 1u : 0u);
            ptx::mma_commit(empty0 + stage * 8u);
            if (++stage == Cfg::kStages) {
                stage = 0;
                phase ^= 1u;
            }
        }
        if (!ok)
            break;
        if (a.nK > 0)
            ptx::mma_commit(ptx::smem_u32(&ctl->acc_full[buf]));
        else
            ptx::mbar_arrive(ptx::smem_u32(&ctl->acc_full[buf]));
    }
    if (!ok) {
        report(a, ctl, kStatusTimeoutMma);
        // Drain every MMA issued so far before TMEM is freed.
        ptx::mma_commit(ptx::smem_u32(&ctl->drain));
        ptx::mbar_wait(ptx::smem_u32(&ctl->drain), 0u, a.timeout, nullptr);
    }
}

__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xffff0000u); }

// Write 8 consecutive output columns (m, n .. n+7) of Y in its dtype.  The
// kernel never reads Y back, so its lines go first when L2 needs room (the
// running sums and operands stay): `pol` is an evict-first policy.
__device__ __forceinline__ void store_y8(const KernelArgs &a, int64_t m, int64_t n, float4 lo,
                                         float4 hi, uint64_t pol)
{
#ifdef GEMM_RS_CHECKED
    if (!in_mn(a, m, n))
        return;
#endif
    if (a.y_fp32) {
        float *yp = static_cast<float *>(a.Y) + m * a.N + n;
        ptx::st_f4_hint(yp, lo, pol);
        ptx::st_f4_hint(yp + 4, hi, pol);
    } else {
        const __nv_bfloat162 h0 = __floats2bfloat162_rn(lo.x, lo.y);
        const __nv_bfloat162 h1 = __floats2bfloat162_rn(lo.z, lo.w);
        const __nv_bfloat162 h2 = __floats2bfloat162_rn(hi.x, hi.y);
        const __nv_bfloat162 h3 = __floats2bfloat162_rn(hi.z, hi.w);
        uint4 w;
        w.x = *reinterpret_cast<const uint32_t *>(&h0);
        w.y = *reinterpret_cast<const uint32_t *>(&h1);
        w.z = *reinterpret_cast<const uint32_t *>(&h2);
        w.w = *reinterpret_cast<const uint32_t *>(&h3);
        ptx::st_u4_hint(static_cast<uint16_t *>(a.Y) + m * a.N + n, w, pol);
    }
}

// ------------------------------------------------------------------ reduce queue
// Single producer (epilogue thread 0), several consumer warps.  An entry is
// (tile << 2) | quarter, or -1 to stop one consumer.  Consumers claim entries
// in order through ctl->rq_head.  An entry's slot is released as soon as it is
// read.
__device__ __forceinline__ bool rq_push(const KernelArgs &a, SmemCtl *ctl, uint32_t &rq_n,
                                        int32_t entry)
{
    const uint32_t s = rq_n % kRQ;
    const uint32_t ph = (rq_n / kRQ) & 1u;
    if (!ptx::mbar_wait(ptx::smem_u32(&ctl->rq_empty[s]), ph ^ 1u, a.timeout, &ctl->abort))
        return false;
    ctl->rq_tile[s] = entry;
    ptx::mbar_arrive(ptx::smem_u32(&ctl->rq_full[s]));
    ++rq_n;
    return true;
}

// y = slot[b] + slot[f] + slot[f+1] + ... + slot[hi] with f = max(lo, b+1),
// folded left to right in fp32, for the 32-column slabs slab0 .. slab1-1 of
// one quarter (32 rows) of tile `tile`, by one warp (lane = row).  Slot b
// holds a running sum (chain mode: b = 0, or the first slot of the second
// rank group in the two-level fold) or rank 0's partial (last-arriver mode,
// b = lo = 0: the W partials in rank order).  to_y: convert and write Y.
// Otherwise the sum is written back to slot b.  The slots f .. hi (and slot b
// after writing Y) are dead afterwards, so their L2 lines are dropped without
// write-back.
template <int BN>
__device__ __forceinline__ void fold_quarter(const KernelArgs &a, int tile, int q, int lane, int b,
                                             int lo, int hi, bool to_y, int slab0, int slab1)
{
    using Cfg = TileCfg<BN>;
    constexpr int S = Cfg::kSlabs;
    const int mt = tile / a.nN;
    const int nt = tile - mt * a.nN;
    const int64_t m = static_cast<int64_t>(mt) * kBM + q * 32 + lane;
    const bool row_ok = m < a.M;
    // slot 0's 32-row quarter; slot s's is s * kSlotFloats further on
    float *q0 = a.part + static_cast<int64_t>(tile) * a.W * Cfg::kSlotFloats +
                static_cast<int64_t>(q) * S * 1024;
    float *qb = q0 + static_cast<int64_t>(b) * Cfg::kSlotFloats; // slot b
    const int first = lo > b + 1 ? lo : b + 1;
    const uint64_t y_pol = ptx::policy_evict_first();
#pragma unroll 1
    for (int slab = slab0; slab < slab1; ++slab) {
        // One slab of a slot is 8 float4 per lane (a 4 KB block per warp),
        // loaded at once.  Fixed order: y = slot[0], then y = y + slot[s].
        const float *sb = qb + slab * 1024 + lane * 4;
        const float *s0 = q0 + slab * 1024 + lane * 4;
        // a lane touches floats [p, p + 7*128 + 4) of a slot's slab block
        constexpr int64_t kLaneSpan = 7 * 128 + 4;
        const bool sb_ok = in_part(a, sb, kLaneSpan);
        float4 y[8];
#pragma unroll
        for (int j = 0; j < 8; ++j)
            y[j] = sb_ok ? ptx::ld_cg_f4(sb + j * 128) : make_float4(0.f, 0.f, 0.f, 0.f);
        // Two slots per round trip (16 loads in flight), added in slot order.
#pragma unroll 1
        for (int sl = first; sl <= hi; sl += 2) {
            const bool two = sl + 1 <= hi;
            const float *pu = s0 + static_cast<int64_t>(sl) * Cfg::kSlotFloats;
            const float *pw = pu + Cfg::kSlotFloats;
            const bool u_ok = in_part(a, pu, kLaneSpan);
            const bool w_ok = !two || in_part(a, pw, kLaneSpan);
            float4 u[8], w2[8];
#pragma unroll
            for (int j = 0; j < 8; ++j)
                u[j] = u_ok ? ptx::ld_cg_f4(pu + j * 128) : make_float4(0.f, 0.f, 0.f, 0.f);
            if (two) {
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    w2[j] = w_ok ? ptx::ld_cg_f4(pw + j * 128) : make_float4(0.f, 0.f, 0.f, 0.f);
            }
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                y[j].x += u[j].x; y[j].y += u[j].y; y[j].z += u[j].z; y[j].w += u[j].w;
            }
            if (two) {
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    y[j].x += w2[j].x; y[j].y += w2[j].y; y[j].z += w2[j].z; y[j].w += w2[j].w;
                }
            }
        }
        if (to_y) {
            // Y is written 8 columns at a time.
#pragma unroll
            for (int j2 = 0; j2 < 4; ++j2) {
                const int64_t n = static_cast<int64_t>(nt) * BN + slab * 32 + j2 * 8;
                if (row_ok && n < a.N) // N is a multiple of 8
                    store_y8(a, m, n, y[2 * j2], y[2 * j2 + 1], y_pol);
            }
        } else if (sb_ok) {
            float *dst = qb + slab * 1024 + lane * 4;
#pragma unroll
            for (int j = 0; j < 8; ++j)
                ptx::st_f4(dst + j * 128, y[j]);
        }
        // Every lane has read this slab of every slot: drop the dead lines
        // (lane l drops line l of each 4 KB block).
        __syncwarp();
        if (to_y && in_part(a, qb + slab * 1024 + lane * 32, 32))
            ptx::discard_l2_line(qb + slab * 1024 + lane * 32);
        for (int s = first; s <= hi; ++s) {
            float *line = q0 + static_cast<int64_t>(s) * Cfg::kSlotFloats + slab * 1024 + lane * 32;
            if (in_part(a, line, 32))
                ptx::discard_l2_line(line);
        }
    }
}

// ---------------------------------------------------------------- chain reduction state
// In the chain mode each output tile has one 32-bit state word:
//   bits  0-15  positions whose partial is stored in their slot and not yet folded
//   bits 16-20  k: positions 0 .. k-1 are folded; their running sum is in slot 0
//   bit  24     owned: one CTA is folding from position k on
// Position i is the contribution's place in the tile's arrival order (the step
// in which its rank reaches the tile, or the rank itself when the ranks run one
// after another), so in a steady run the positions arrive in order and each one
// folds itself straight from TMEM.
// The flag's release/acquire chain orders the folds: position i's additions
// to slot 0 all happen before position i+1's, so every element is summed in
// position order, the same order on every run.
constexpr uint32_t kChainOwn = 1u << 24;
__device__ __forceinline__ uint32_t chain_k(uint32_t s) { return (s >> 16) & 31u; }

// Take the fold at position i: true if positions 0 .. i-1 are folded, nobody
// owns the tile, and the caller now owns it; `seen` is then the state it took
// the tile in (its pending bits tell which positions after i are stored).  The
// first compare-and-swap guesses `guess` (by default the usual state: k = i,
// nothing stored ahead), so the common case costs one atomic.  Taking the fold
// publishes nothing, so the compare-and-swap only acquires: the additions and
// slots of positions 0 .. k-1 (released by whoever published k) are ordered
// before the caller's.  A release here would add a gpu-scope fence per tile,
// which on this two-die part is broadcast to the other die's L2 slices.
__device__ __forceinline__ bool chain_try_own(uint32_t *flag, uint32_t i, uint32_t guess,
                                              uint32_t &seen)
{
    uint32_t s = ptx::atom_cas_acquire_gpu(flag, guess, guess | kChainOwn);
    if (s == guess) {
        seen = s;
        return true;
    }
    while (chain_k(s) == i && !(s & kChainOwn)) {
        const uint32_t prev = ptx::atom_cas_acquire_gpu(flag, s, s | kChainOwn);
        if (prev == s) {
            seen = s;
            return true;
        }
        s = prev;
    }
    return false;
}

__device__ __forceinline__ bool chain_try_own(uint32_t *flag, uint32_t i)
{
    uint32_t seen;
    return chain_try_own(flag, i, i << 16, seen);
}

// The last position j >= k such that positions k+1 .. j are stored in state s
// (clen positions in the chain).
__device__ __forceinline__ int chain_stored_end(uint32_t s, int k, int clen)
{
    int j = k;
    while (j + 1 < clen && ((s >> (j + 1)) & 1u))
        ++j;
    return j;
}

// The owner has folded positions 0 .. kn-1 (running sum in slot 0).  If
// position kn is already stored, it keeps the ownership and returns true (the
// caller folds on from kn), with `seen` a state that shows kn stored.
// Otherwise it publishes k = kn and releases.  `guess` is the state the
// caller last saw (the owner alone clears pending bits, so a bit set there is
// still set); a wrong guess costs one more compare-and-swap.  The release side
// of the compare-and-swap publishes the running sum, which every epilogue
// thread stored before the CTA barrier that precedes this call.
__device__ __forceinline__ bool chain_pass_on(uint32_t *flag, uint32_t kn, uint32_t guess,
                                              uint32_t &seen)
{
    uint32_t s = guess;
    while (true) {
        if ((s >> kn) & 1u) {
            seen = s;
            return true;
        }
        const uint32_t nv = (kn << 16) | ((s & 0xFFFFu) & ~((1u << kn) - 1u));
        const uint32_t prev = ptx::atom_cas_acq_rel_gpu(flag, s, nv);
        if (prev == s)
            return false;
        s = prev;
    }
}

// Wait for the turn of position i (positions 0 .. i-1 folded), then take the
// fold.  The wait is bounded by `limit` SM cycles: after that the caller stores
// its partial and the fold happens later.  Waiting cannot deadlock: position
// i-1 lies earlier in the global tile order, and a CTA that waits only ever
// waits for earlier items; the bound keeps even a stalled peer from holding it.
__device__ __forceinline__ bool chain_wait_own(uint32_t *flag, uint32_t i, long long limit)
{
    const long long t0 = clock64();
    while (true) {
        const uint32_t s = ptx::ld_acquire_gpu(flag);
        if (chain_k(s) == i && !(s & kChainOwn) && chain_try_own(flag, i))
            return true;
        if (chain_k(s) > i || clock64() - t0 > limit)
            return false;
        __nanosleep(64);
    }
}

// Two-level fold: a rank group has folded all its positions (its sum is in
// its first slot, published by the caller's barrier and this atomic's release
// side).  The groups count themselves in on the tile's third state word; the
// second to arrive returns 1, puts the word back to 0 for the next call, and
// adds the two sums.
__device__ __forceinline__ int group_done(const KernelArgs &a, int tile)
{
    uint32_t *done = a.flags + 2 * static_cast<int64_t>(a.nM) * a.nN + tile;
    if (!in_flags(a, done))
        done = a.flags;
    if (ptx::atom_add_acq_rel_gpu(done, 1u) == 0u)
        return 0;
    ptx::st_relaxed_gpu(done, 0u);
    return 1;
}

// A consumer warp: claim entries until it takes a stop entry.  Entry kinds:
//   (tile << 2) | q   last-arriver mode: fold all W slots of quarter q into Y
//   -1                stop
template <int BN>
__device__ __forceinline__ void run_consumer(const KernelArgs &a, SmemCtl *ctl, int lane)
{
    const volatile int *abort_flag = &ctl->abort;
    while (true) {
        uint32_t n = 0;
        int entry = -1, waited = 1;
        if (lane == 0) {
            n = atomicAdd(&ctl->rq_head, 1u);
            const uint32_t s = n % kRQ;
            const uint32_t ph = (n / kRQ) & 1u;
            waited = ptx::mbar_wait(ptx::smem_u32(&ctl->rq_full[s]), ph, a.timeout, abort_flag) ? 1 : 0;
            if (waited) {
                entry = *reinterpret_cast<volatile int32_t *>(&ctl->rq_tile[s]);
                ptx::mbar_arrive(ptx::smem_u32(&ctl->rq_empty[s]));
            }
        }
        waited = __shfl_sync(0xffffffffu, waited, 0);
        entry = __shfl_sync(0xffffffffu, entry, 0);
        if (!waited) {
            if (lane == 0)
                report(a, ctl, kStatusTimeoutReducer);
            break;
        }
        if (entry < 0)
            break;
        fold_quarter<BN>(a, entry >> 2, entry & 3, lane, 0, 0, a.W - 1, true, 0, TileCfg<BN>::kSlabs);
    }
}

// ------------------------------------------------------------------ epilogue
// PAIR: the CTA is half `crank` of a 256-row pair tile.  It drains its own
// TMEM, waits with cluster-scope acquire, and hands the accumulator back to
// the pair's MMA thread (in CTA 0).
//
// Last-arriver mode: every rank stores its partial in slot r, counts itself in
// on the tile's counter, and the rank that arrives last queues the tile: the
// consumers fold slots 0 .. W-1 (rank order) into Y.
// Chain mode: the rank at position i (the tile's arrival order: its step when
// the ranks run side by side, its rank when they run one after another) folds
// its own partial straight from TMEM onto the running sum in slot 0 when
// positions 0 .. i-1 are done: position 0 stores it, positions 1 .. W-2 add to
// it in L2 (red.add, nothing comes back to the SM), and the last position reads
// it and writes Y.  A rank that is early stores its partial in slot i.
// Whoever owns the fold when the positions after it are already stored (or
// the early rank itself, once its turn has come) folds them from their slots.
// The chain mode has no reduce jobs, so warps 6-9 join the epilogue: two warps
// per TMEM lane quarter, each draining half of the tile's 32-column slabs.
template <int BN, bool PAIR>
__device__ __forceinline__ void run_epilogue(const KernelArgs &a, const Sched &sch, uint32_t tmem,
                                             SmemCtl *ctl, int warp, int lane, int64_t g0,
                                             int64_t gstride, uint32_t crank)
{
    using Cfg = TileCfg<BN>;
    const volatile int *abort_flag = &ctl->abort;
    const int q = warp & 3;                           // TMEM lanes [32q, 32q + 32)
    const int etid = threadIdx.x - kEpiWarp0 * 32;    // 0 .. nthr-1
    const int nthr = epi_threads(a);
    // slabs [sl0, sl1) of every tile: all of them with one warp per quarter
    const int half = (warp - kEpiWarp0) >> 2;
    const int sl0 = a.chain ? half * (Cfg::kSlabs / 2) : 0;
    const int sl1 = a.chain ? sl0 + Cfg::kSlabs / 2 : Cfg::kSlabs;
    const uint32_t lane_base = static_cast<uint32_t>(q * 32) << 16;
    // Last-arriver partials are read back only at the end of the schedule: do
    // not let them push the B panels out of L2.  Chain-mode slots are read at
    // the next step: keep them.
    const uint64_t st_pol = a.chain ? ptx::policy_evict_normal() : ptx::policy_evict_first();
    const uint64_t y_pol = ptx::policy_evict_first();
    bool ok = true;
    uint32_t rq_n = 0;
    int it = 0;
    // Host-streamed inputs: C must have landed before the first read of it.
    // Thread 0 waits; the first tile's barrier passes a failure on and orders
    // the other threads' reads after its acquire.
    if (a.ready != nullptr && a.C != nullptr && etid == 0 &&
        !wait_ready(a.ready + a.W, a.epoch, a.timeout, abort_flag)) {
        report(a, ctl, kStatusTimeoutEpilogue);
        ok = false;
    }
    for (int64_t g = g0; g < a.total; g += gstride, ++it) {
        int r, mts, nt, pos;
        decode_tile(sch, g, r, mts, nt, pos);
        const int mt = PAIR ? 2 * mts + static_cast<int>(crank) : mts;
        const bool half_ok = mt < a.nM; // a pair's second half may lie wholly below M
        const int tile = mt * a.nN + nt;
        const int buf = it & 1;
        // The chain this contribution joins.  One fold over all W ranks at
        // position pos, or, for the two-level fold, the fold of its rank group
        // (ranks [0, split) or [split, W)) at its place in the group, with the
        // group's own state word and its running sum in the group's first slot.
        const int grp = (a.split > 0 && r >= a.split) ? 1 : 0;
        const int base = grp ? a.split : 0;
        const int cpos = a.split > 0 ? r - base : pos;
        const int clen = a.split > 0 ? (grp ? a.W - a.split : a.split) : a.W;
        uint32_t *cflag = a.flags + static_cast<int64_t>(grp) * a.nM * a.nN + tile;
        if (!in_flags(a, cflag))
            cflag = a.flags; // checked build only: keep the atomics in bounds
        // Chain mode: try to take the fold while the accumulator is still being
        // computed, so the decision is ready when it lands.
        if (etid == 0)
            ctl->epi_direct[buf] =
                (a.chain && half_ok && chain_try_own(cflag, static_cast<uint32_t>(cpos))) ? 1 : 0;
        const uint32_t aph = static_cast<uint32_t>(it >> 1) & 1u;
        const uint32_t fb = ptx::smem_u32(&ctl->acc_full[buf]);
        const bool waited = PAIR ? ptx::mbar_wait_cluster(fb, aph, a.timeout, abort_flag)
                                 : ptx::mbar_wait(fb, aph, a.timeout, abort_flag);
        // If position pos-1 was not folded yet at the start, wait a little for
        // it now that the accumulator has landed (a.chain_wait cycles; the host
        // sets it where positions arrive staggered, as at the first step of a
        // column group with the ranks side by side, whose B panels are not in
        // L2 yet).  Where positions land together, storing at once and folding
        // once is cheaper than a queue of waits.
        if (etid == 0 && a.chain && waited && half_ok) {
            if (ctl->epi_direct[buf] == 0)
                ctl->epi_direct[buf] =
                    chain_wait_own(cflag, static_cast<uint32_t>(cpos), a.chain_wait) ? 1 : 0;
            // Two-level fold, last position of a group: if the other group is
            // already done, this position adds all three terms and writes Y
            // (direct = 2) instead of publishing its group's sum.
            if (a.split > 0 && ctl->epi_direct[buf] != 0 && cpos == clen - 1 &&
                in_flags(a, a.flags + 2 * static_cast<int64_t>(a.nM) * a.nN + tile) &&
                ptx::ld_acquire_gpu(a.flags + 2 * static_cast<int64_t>(a.nM) * a.nN + tile) != 0u)
                ctl->epi_direct[buf] = 2;
        }
        if (ptx::named_bar_or(kBarEpi, nthr, !(waited && ok))) {
            ok = false;
            break;
        }
        ptx::tc_fence_after();
        if (!half_ok) {
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                if (PAIR)
                    ptx::mbar_arrive_cluster(ptx::mapa(ptx::smem_u32(&ctl->acc_empty[buf]), 0));
                else
                    ptx::mbar_arrive(ptx::smem_u32(&ctl->acc_empty[buf]));
            }
            continue;
        }
        const int dmode = *reinterpret_cast<volatile int *>(&ctl->epi_direct[buf]);
        const bool direct = dmode != 0;
        const bool final = dmode == 2; // two-level: the other group's sum is ready
        // Chain mode: the running sum lives in slot `base`.  Position 0 stores
        // it, the middle positions add to it in L2, and the last position of a
        // one-level fold reads it and writes Y.  The last position of a group
        // of the two-level fold adds to it like the middle ones, unless the
        // other group is done: then it reads both sums and writes
        // Y = (other group's sum) + (running sum + partial).  An early
        // position stores its partial in its own slot.
        const int sidx = a.chain ? (direct ? base : base + cpos) : r; // slot written
        const bool to_y = direct && (a.split == 0 || final) && cpos == clen - 1;
        const bool add_prev = to_y && cpos > 0;                      // read the running sum
        const bool add_l2 = direct && cpos > 0 && !to_y;             // add to it in L2

        const int64_t m = static_cast<int64_t>(mt) * kBM + q * 32 + lane;
        const bool row_ok = m < a.M;
        // A quarter wholly below M (a short last row tile) has nothing to do.
        const bool q_live = static_cast<int64_t>(mt) * kBM + q * 32 < a.M;
        float *tb = a.part + static_cast<int64_t>(tile) * a.W * Cfg::kSlotFloats +
                    static_cast<int64_t>(q) * Cfg::kSlabs * 1024 + lane * 4;
        float *slot = tb + static_cast<int64_t>(sidx) * Cfg::kSlotFloats;
        const float *prev = tb + static_cast<int64_t>(base) * Cfg::kSlotFloats; // running sum
        // the other group's sum (two-level, final position)
        const float *other = tb + static_cast<int64_t>(grp ? 0 : a.split) * Cfg::kSlotFloats;
        if (!q_live) {
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                if (PAIR)
                    ptx::mbar_arrive_cluster(ptx::mapa(ptx::smem_u32(&ctl->acc_empty[buf]), 0));
                else
                    ptx::mbar_arrive(ptx::smem_u32(&ctl->acc_empty[buf]));
            }
        }
        // The running sum is loaded before the slab's TMEM read; the other
        // warp of the lane quarter covers its latency.
#pragma unroll 1
        for (int slab = sl0; slab < (q_live ? sl1 : sl0); ++slab) {
            float4 rs[8];
            if (add_prev) {
                const bool ok = in_part(a, prev + slab * 1024, 7 * 128 + 4);
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    rs[j] = ok ? ptx::ld_cg_f4(prev + slab * 1024 + j * 128)
                               : make_float4(0.f, 0.f, 0.f, 0.f);
            }
            uint32_t v[32];
            if (a.nK > 0) {
                ptx::tmem_ld_32x32b_x32(tmem + lane_base + static_cast<uint32_t>(buf * BN + slab * 32),
                                        v);
            } else {
#pragma unroll
                for (int i = 0; i < 32; ++i)
                    v[i] = 0u;
            }
            if (slab == sl1 - 1) {
                // The warp's share of the accumulator is read: hand it back to
                // the MMA thread.
                ptx::tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    if (PAIR)
                        ptx::mbar_arrive_cluster(ptx::mapa(ptx::smem_u32(&ctl->acc_empty[buf]), 0));
                    else
                        ptx::mbar_arrive(ptx::smem_u32(&ctl->acc_empty[buf]));
                }
            }
            float p[32];
#pragma unroll
            for (int i = 0; i < 32; ++i)
                p[i] = a.alpha * __uint_as_float(v[i]);
            if (a.beta != 0.0f) {
                const int64_t n0 = static_cast<int64_t>(nt) * BN + slab * 32;
#pragma unroll
                for (int g8 = 0; g8 < 4; ++g8) {
                    const int64_t n = n0 + 8 * g8;
                    if (row_ok && n < a.N && in_mn(a, m, n)) {
                        const uint4 c = ptx::ld_nc_u4(a.C + m * a.N + n);
                        const uint32_t cw[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            p[8 * g8 + 2 * e] = fmaf(a.beta, bf16_lo(cw[e]), p[8 * g8 + 2 * e]);
                            p[8 * g8 + 2 * e + 1] =
                                fmaf(a.beta, bf16_hi(cw[e]), p[8 * g8 + 2 * e + 1]);
                        }
                    }
                }
            }
            if (add_prev) {
                // running sum first, then this position's partial
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    p[4 * j] = rs[j].x + p[4 * j];
                    p[4 * j + 1] = rs[j].y + p[4 * j + 1];
                    p[4 * j + 2] = rs[j].z + p[4 * j + 2];
                    p[4 * j + 3] = rs[j].w + p[4 * j + 3];
                }
            }
            if (final) {
                // then the other group's sum (fp32 addition is commutative, so
                // this is y0 + y1 whichever group finishes second)
                const bool ok = in_part(a, other + slab * 1024, 7 * 128 + 4);
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    rs[j] = ok ? ptx::ld_cg_f4(other + slab * 1024 + j * 128)
                               : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    p[4 * j] = rs[j].x + p[4 * j];
                    p[4 * j + 1] = rs[j].y + p[4 * j + 1];
                    p[4 * j + 2] = rs[j].z + p[4 * j + 2];
                    p[4 * j + 3] = rs[j].w + p[4 * j + 3];
                }
            }
            if (to_y) {
                const int64_t n0 = static_cast<int64_t>(nt) * BN + slab * 32;
#pragma unroll
                for (int g8 = 0; g8 < 4; ++g8) {
                    const int64_t n = n0 + 8 * g8;
                    if (row_ok && n < a.N)
                        store_y8(a, m, n,
                                 make_float4(p[8 * g8], p[8 * g8 + 1], p[8 * g8 + 2], p[8 * g8 + 3]),
                                 make_float4(p[8 * g8 + 4], p[8 * g8 + 5], p[8 * g8 + 6], p[8 * g8 + 7]),
                                 y_pol);
                }
            } else if (add_l2) {
                // running sum + this position's partial, added in L2
                float *dst = slot + slab * 1024;
                if (in_part(a, dst, 7 * 128 + 4)) {
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        ptx::red_add_f4(dst + j * 128, make_float4(p[4 * j], p[4 * j + 1],
                                                                   p[4 * j + 2], p[4 * j + 3]));
                }
            } else if (in_part(a, slot + slab * 1024, 7 * 128 + 4)) {
                float *dst = slot + slab * 1024;
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    ptx::st_f4_hint(dst + j * 128,
                                    make_float4(p[4 * j], p[4 * j + 1], p[4 * j + 2], p[4 * j + 3]),
                                    st_pol);
            }
            if (add_prev || final) {
                // the sums read are dead: drop their lines of this warp's 4 KB block
                __syncwarp();
                const float *lp = prev - lane * 4 + slab * 1024 + lane * 32; // line `lane`
                const float *lo = other - lane * 4 + slab * 1024 + lane * 32;
                if (add_prev && in_part(a, lp, 32))
                    ptx::discard_l2_line(lp);
                if (final && in_part(a, lo, 32))
                    ptx::discard_l2_line(lo);
            }
        }

        // Every epilogue thread has issued its stores.  The barrier orders them
        // before thread 0's flag atomic, whose release side publishes them at
        // gpu scope; the thread that acquires the flag, and through the next
        // barrier its CTA, then sees them.
        ptx::named_bar_sync(kBarEpi, nthr);
        if (etid == 0) {
            if (!a.chain) {
                uint32_t *flag = a.flags + tile;
                if (!in_flags(a, flag))
                    flag = a.flags;
                const uint32_t old = ptx::atom_add_acq_rel_gpu(flag, 1u);
                if (old == static_cast<uint32_t>(a.W - 1)) {
                    // Last arriver: the counter goes back to 0 for the next call
                    // (no memset), and the tile goes to the reducers.
                    ptx::st_relaxed_gpu(flag, 0u);
                    for (int qq = 0; qq < 4 && ok; ++qq)
                        if (static_cast<int64_t>(mt) * kBM + qq * 32 < a.M)
                            ok = rq_push(a, ctl, rq_n, (tile << 2) | qq);
                }
            } else {
                int fold_from = -1, combine = 0;
                uint32_t seen = 0;
                if (direct) {
                    if (cpos == clen - 1) {
                        ptx::st_relaxed_gpu(cflag, 0u); // back to 0 for the next call
                        if (final && in_flags(a, a.flags + 2 * static_cast<int64_t>(a.nM) * a.nN + tile))
                            // Y is written; the group count goes back to 0
                            ptx::st_relaxed_gpu(a.flags + 2 * static_cast<int64_t>(a.nM) * a.nN + tile, 0u);
                        else if (a.split > 0)
                            combine = group_done(a, tile);
                    } else if (chain_pass_on(cflag, static_cast<uint32_t>(cpos + 1),
                                             (static_cast<uint32_t>(cpos) << 16) | kChainOwn, seen)) {
                        fold_from = cpos + 1;
                    }
                } else {
                    const uint32_t bit = 1u << cpos;
                    const uint32_t old = ptx::atom_or_acq_rel_gpu(cflag, bit);
                    if (chain_k(old) == static_cast<uint32_t>(cpos) && !(old & kChainOwn) &&
                        chain_try_own(cflag, static_cast<uint32_t>(cpos), old | bit, seen))
                        fold_from = cpos;
                }
                ctl->epi_fold = fold_from;
                if (fold_from >= 0)
                    ctl->epi_fold_end = chain_stored_end(seen, fold_from, clen);
                ctl->epi_seen = seen;
                ctl->epi_combine = combine;
            }
        }
        if (a.chain) {
            // Fold on while the positions after the running sum are already
            // stored, then, for the two-level fold, add the two groups' sums if
            // this CTA completed the second group.  A fold reads only global
            // memory, so the (quarter, slab) units of the live quarters are
            // spread over all epilogue warps.
            ptx::named_bar_sync(kBarEpi, nthr);
            int k = *reinterpret_cast<volatile int *>(&ctl->epi_fold);
            bool combine = *reinterpret_cast<volatile int *>(&ctl->epi_combine) != 0;
            while (k >= 0 || combine) {
                int fb = 0, flo = a.split, fhi = a.split; // the combine: y = slot[0] + slot[split]
                bool fy = true, last = false;
                if (k >= 0) {
                    // positions k .. j are stored (from the state the owner
                    // took or kept the fold in)
                    const int j = *reinterpret_cast<volatile int *>(&ctl->epi_fold_end);
                    last = j == clen - 1;
                    fb = base;
                    flo = base + k;
                    fhi = base + j;
                    fy = last && a.split == 0;
                }
                const int64_t rows_left = a.M - static_cast<int64_t>(mt) * kBM;
                const int nlive = rows_left >= kBM ? 4 : static_cast<int>((rows_left + 31) / 32);
                for (int u = (warp - kEpiWarp0); u < nlive * Cfg::kSlabs; u += nthr / 32)
                    fold_quarter<BN>(a, tile, u / Cfg::kSlabs, lane, fb, flo, fhi, fy, u % Cfg::kSlabs,
                                     u % Cfg::kSlabs + 1);
                if (k < 0)
                    break; // the combine wrote Y
                ptx::named_bar_sync(kBarEpi, nthr);
                if (etid == 0) {
                    int next = -1;
                    if (last) {
                        ptx::st_relaxed_gpu(cflag, 0u);
                        if (a.split > 0)
                            ctl->epi_combine = group_done(a, tile);
                    } else {
                        uint32_t seen = ctl->epi_seen;
                        if (chain_pass_on(cflag, static_cast<uint32_t>(fhi - base + 1), seen, seen)) {
                            next = fhi - base + 1;
                            ctl->epi_fold_end = chain_stored_end(seen, next, clen);
                            ctl->epi_seen = seen;
                        }
                    }
                    ctl->epi_fold = next;
                }
                ptx::named_bar_sync(kBarEpi, nthr);
                k = *reinterpret_cast<volatile int *>(&ctl->epi_fold);
                combine = *reinterpret_cast<volatile int *>(&ctl->epi_combine) != 0;
            }
        }
    }
    // No more tiles: one stop entry per consumer warp (last-arriver mode).
    if (etid == 0) {
        if (!a.chain)
            for (int i = 0; i < kConsumers && ok; ++i)
                ok = rq_push(a, ctl, rq_n, -1);
        if (!ok)
            report(a, ctl, kStatusTimeoutEpilogue);
    }
    // Once its own tiles are done, the epilogue helps with the reductions.
    if (!ptx::named_bar_or(kBarEpi, nthr, !ok) && !a.chain)
        run_consumer<BN>(a, ctl, lane);
}

// ------------------------------------------------------------------ kernel
template <int BN>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_rs_fused_kernel(const __grid_constant__ CUtensorMap tmA,
                         const __grid_constant__ CUtensorMap tmB, const KernelArgs a)
{
    using Cfg = TileCfg<BN>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = ptx::smem_u32(smem_raw);
    uint8_t *smem = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
    SmemCtl *ctl = reinterpret_cast<SmemCtl *>(smem + Cfg::kStages * Cfg::kStageBytes);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < Cfg::kStages; ++s) {
            ptx::mbar_init(ptx::smem_u32(&ctl->full[s]), 1);
            ptx::mbar_init(ptx::smem_u32(&ctl->empty[s]), 1);
        }
        for (int b = 0; b < 2; ++b) {
            ptx::mbar_init(ptx::smem_u32(&ctl->acc_full[b]), 1);
            ptx::mbar_init(ptx::smem_u32(&ctl->acc_empty[b]), epi_threads(a) / 32);
        }
        for (int s = 0; s < kRQ; ++s) {
            ptx::mbar_init(ptx::smem_u32(&ctl->rq_full[s]), 1);
            ptx::mbar_init(ptx::smem_u32(&ctl->rq_empty[s]), 1);
        }
        ptx::mbar_init(ptx::smem_u32(&ctl->drain), 1);
        ctl->abort = 0;
        ctl->rq_head = 0;
        ptx::fence_barrier_init();
    }
    if (warp == 0 && lane == 0 && a.nK > 0) {
        ptx::prefetch_tensormap(&tmA);
        ptx::prefetch_tensormap(&tmB);
    }
    if (warp == 1) {
        ptx::tmem_alloc(ptx::smem_u32(&ctl->tmem_base), Cfg::kTmemCols);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = ctl->tmem_base;
    const Sched sch{a.W, a.nMs, a.nN, 7, a.R, a.colgroup, a.rowgroup, a.seq};
    // Everything above touches only this CTA's shared memory and TMEM, so it
    // may overlap the previous kernel on the stream; global memory waits.
    ptx::grid_dependency_wait();
    ptx::grid_launch_dependents();

    if (warp == 0) {
        if (lane == 0)
            run_producer<BN>(a, sch, &tmA, &tmB, smem, ctl);
        __syncwarp();
    } else if (warp == 1) {
        if (lane == 0)
            run_mma<BN>(a, tmem, smem, ctl);
        __syncwarp();
    } else if (warp < kRedWarp0 || a.chain) {
        run_epilogue<BN, false>(a, sch, tmem, ctl, warp, lane, blockIdx.x, gridDim.x, 0u);
    } else {
        run_consumer<BN>(a, ctl, lane);
    }

    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, Cfg::kTmemCols);
    }
}

// ------------------------------------------------------------------ CTA-pair kernel
// End of a pair producer.  Both CTAs' loads complete on the even CTA's `full`
// barriers, so only the even CTA can see them land.  After a failure the even
// CTA waits (bounded) for its last fills of every stage; after a normal run
// its tail has already waited for every stage to be released, which follows
// the stage's loads.  Either way it then arrives on the odd CTA's
// `peer_drained` barrier.  The odd CTA, after a failure of its own, waits on
// that barrier (bounded) before the pair tears down, so it never leaves with
// one of its loads still writing into its shared memory.
__device__ __forceinline__ void pair_producer_finish(SmemCtl *ctl, uint32_t crank, bool ok,
                                                     int64_t issued, int stages,
                                                     unsigned long long timeout)
{
    if (crank == 0) {
        if (!ok) {
            const int64_t n = issued < stages ? issued : stages;
            for (int64_t i = 1; i <= n; ++i) {
                const int64_t pos = issued - i;
                const uint32_t s = static_cast<uint32_t>(pos % stages);
                const uint32_t ph = static_cast<uint32_t>((pos / stages) & 1);
                ptx::mbar_wait_cluster(ptx::smem_u32(&ctl->full[s]), ph, timeout, nullptr);
            }
        }
        ptx::mbar_arrive_cluster(ptx::mapa(ptx::smem_u32(&ctl->peer_drained), 1));
    } else if (!ok) {
        ptx::mbar_wait_cluster(ptx::smem_u32(&ctl->peer_drained), 0u, timeout, nullptr);
    }
}

// Producer of one CTA of a pair.  Both CTAs load into their own shared memory.
// The loads count their bytes on the even CTA's `full` barrier, which only the
// even CTA arms (expect_tx of both CTAs' bytes).
template <int BN>
__device__ __forceinline__ void run_producer_pair(const KernelArgs &a, const Sched &sch,
                                                  const CUtensorMap *tmA, const CUtensorMap *tmB,
                                                  uint8_t *smem, SmemCtl *ctl, uint32_t crank)
{
    using Cfg = PairCfg<BN>;
    const volatile int *abort_flag = &ctl->abort;
    const uint64_t polA = ptx::policy_evict_normal();
    const uint64_t polB = ptx::policy_evict_last(); // B panels are swept again every step
    const int64_t ncl = gridDim.x / 2;
    const int64_t cid = blockIdx.x / 2;
    uint32_t stage = 0, phase = 0;
    int64_t issued = 0;
    bool ok = true;
    uint32_t ranks_ready = 0;
    if (!a.stall_producer) {
        for (int64_t g = cid; g < a.total && ok; g += ncl) {
            int r, mt2, nt;
            decode_tile(sch, g, r, mt2, nt);
            if (a.record != nullptr && crank == 0) {
                int32_t *rec = a.record + 4 * g;
                rec[0] = r;
                rec[1] = mt2;
                rec[2] = nt;
                rec[3] = static_cast<int32_t>(cid);
            }
            if (!operands_ready(a, r, ranks_ready, abort_flag)) {
                ok = false;
                break;
            }
            for (int kb = 0; kb < a.nK; ++kb) {
                if (!ptx::mbar_wait_cluster(ptx::smem_u32(&ctl->empty[stage]), phase ^ 1u, a.timeout,
                                            abort_flag)) {
                    ok = false;
                    break;
                }
                const uint32_t fb = ptx::smem_u32(&ctl->full[stage]);
                if (crank == 0)
                    ptx::mbar_arrive_expect_tx(fb, 2 * Cfg::kStageBytes);
                const uint32_t fb_leader = ptx::mapa(fb, 0);
                const uint32_t sa = ptx::smem_u32(smem + stage * Cfg::kStageBytes);
                ptx::tma_load_3d_pair(sa, tmA, fb_leader, kb * kBK, mt2 * (2 * kBM) + crank * kBM, r,
                                      polA);
                if (a.b4d) {
                    ptx::tma_load_4d_pair(sa + Cfg::kABytes, tmB, fb_leader, 0, kb * kBK,
                                          (nt * BN + static_cast<int>(crank) * (BN / 2)) / 64, r,
                                          polB);
                } else {
#pragma unroll
                    for (int j = 0; j < BN / 128; ++j)
                        ptx::tma_load_3d_pair(sa + Cfg::kABytes + j * 8192, tmB, fb_leader,
                                              nt * BN + crank * (BN / 2) + j * 64, kb * kBK, r,
                                              polB);
                }
                ++issued;
                if (++stage == Cfg::kStages) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
        }
    }
    if (ok) {
        // Tail: every stage released by the pair's MMA, so that every arrival
        // on this CTA's barriers has landed before the CTA exits.
        for (int i = 0; i < Cfg::kStages; ++i) {
            if (!ptx::mbar_wait_cluster(ptx::smem_u32(&ctl->empty[stage]), phase ^ 1u, a.timeout,
                                        abort_flag)) {
                ok = false;
                break;
            }
            if (++stage == Cfg::kStages) {
                stage = 0;
                phase ^= 1u;
            }
        }
    }
    if (!ok)
        report(a, ctl, kStatusTimeoutProducer);
    pair_producer_finish(ctl, crank, ok, issued, Cfg::kStages, a.timeout);
}

// MMA issuer of the pair (one thread of the even CTA).
template <int BN>
__device__ __forceinline__ void run_mma_pair(const KernelArgs &a, uint32_t tmem, uint8_t *smem,
                                             SmemCtl *ctl)
{
    using Cfg = PairCfg<BN>;
    const volatile int *abort_flag = &ctl->abort;
    const int64_t ncl = gridDim.x / 2;
    const int64_t cid = blockIdx.x / 2;
    uint32_t stage = 0, phase = 0;
    bool ok = true;
    int it = 0;
    // As in run_mma: stage 0's descriptors, moved by additions.  They describe
    // this CTA's 128 rows of A and BN/2 columns of B; the peer CTA holds its
    // halves at the same offsets.  One multicast commit releases a stage in
    // both CTAs.
    const uint32_t s0 = ptx::smem_u32(smem);
    const uint64_t ad0 = ptx::sdesc_sw128(s0, 0, 1024);
    const uint64_t bd0 = ptx::sdesc_sw128(s0 + Cfg::kABytes, 8192, 1024);
    const uint32_t empty0 = ptx::smem_u32(&ctl->empty[0]);
    for (int64_t g = cid; g < a.total; g += ncl, ++it) {
        const int buf = it & 1;
        const uint32_t aph = static_cast<uint32_t>(it >> 1) & 1u;
        if (!ptx::mbar_wait_cluster(ptx::smem_u32(&ctl->acc_empty[buf]), aph ^ 1u, a.timeout,
                                    abort_flag)) {
            ok = false;
            break;
        }
        ptx::tc_fence_after();
        const uint32_t d = tmem + static_cast<uint32_t>(buf * BN);
        for (int kb = 0; kb < a.nK; ++kb) {
            if (!ptx::mbar_wait_cluster(ptx::smem_u32(&ctl->full[stage]), phase, a.timeout,
                                        abort_flag)) {
                ok = false;
                break;
            }
            ptx::tc_fence_after();
            const uint32_t so = stage * Cfg::kStageBytes;
#pragma unroll
            for (int kk = 0; kk < kBK / 16; ++kk)
                ptx::mma_bf16_ss_pair(d, ptx::sdesc_advance(ad0, so + kk * 32),
                                      ptx::sdesc_advance(bd0, so + kk * 2048), Cfg::kIdesc,
                                      (kb | kk) != 0 ? 1u : 0u);
            ptx::mma_commit_pair_both(empty0 + stage * 8u);
            if (++stage == Cfg::kStages) {
                stage = 0;
                phase ^= 1u;
            }
        }
        if (!ok)
            break;
        const uint32_t ab = ptx::smem_u32(&ctl->acc_full[buf]);
        if (a.nK > 0) {
            ptx::mma_commit_pair_both(ab);
        } else {
            ptx::mbar_arrive_cluster(ptx::mapa(ab, 0));
            ptx::mbar_arrive_cluster(ptx::mapa(ab, 1));
        }
    }
    if (!ok) {
        report(a, ctl, kStatusTimeoutMma);
        ptx::mma_commit_pair(ptx::mapa(ptx::smem_u32(&ctl->drain), 0));
        ptx::mbar_wait_cluster(ptx::smem_u32(&ctl->drain), 0u, a.timeout, nullptr);
    }
}

template <int BN>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    gemm_rs_pair_kernel(const __grid_constant__ CUtensorMap tmA,
                        const __grid_constant__ CUtensorMap tmB, const KernelArgs a)
{
    using Cfg = PairCfg<BN>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = ptx::smem_u32(smem_raw);
    uint8_t *smem = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
    SmemCtl *ctl = reinterpret_cast<SmemCtl *>(smem + Cfg::kStages * Cfg::kStageBytes);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t crank = ptx::cluster_ctarank();

    if (threadIdx.x == 0) {
        for (int s = 0; s < Cfg::kStages; ++s) {
            ptx::mbar_init(ptx::smem_u32(&ctl->full[s]), 1);
            ptx::mbar_init(ptx::smem_u32(&ctl->empty[s]), 1);
        }
        for (int b = 0; b < 2; ++b) {
            ptx::mbar_init(ptx::smem_u32(&ctl->acc_full[b]), 1);
            // epilogue warps x 2 CTAs
            ptx::mbar_init(ptx::smem_u32(&ctl->acc_empty[b]), 2 * (epi_threads(a) / 32));
        }
        for (int s = 0; s < kRQ; ++s) {
            ptx::mbar_init(ptx::smem_u32(&ctl->rq_full[s]), 1);
            ptx::mbar_init(ptx::smem_u32(&ctl->rq_empty[s]), 1);
        }
        ptx::mbar_init(ptx::smem_u32(&ctl->drain), 1);
        ptx::mbar_init(ptx::smem_u32(&ctl->peer_drained), 1);
        ctl->abort = 0;
        ctl->rq_head = 0;
        ptx::fence_barrier_init();
    }
    if (warp == 0 && lane == 0 && a.nK > 0) {
        ptx::prefetch_tensormap(&tmA);
        ptx::prefetch_tensormap(&tmB);
    }
    if (warp == 1) {
        ptx::tmem_alloc_pair(ptx::smem_u32(&ctl->tmem_base), Cfg::kTmemCols);
        ptx::tmem_relinquish_pair();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::cluster_sync(); // the peer's barriers are initialised before any remote arrival
    ptx::tc_fence_after();
    const uint32_t tmem = ctl->tmem_base;
    const Sched sch{a.W, a.nMs, a.nN, 8, a.R, a.colgroup, a.rowgroup, a.seq};
    // Everything above touches only this CTA pair's shared memory and TMEM, so
    // it may overlap the previous kernel on the stream; global memory waits.
    ptx::grid_dependency_wait();
    ptx::grid_launch_dependents();

    if (warp == 0) {
        if (lane == 0)
            run_producer_pair<BN>(a, sch, &tmA, &tmB, smem, ctl, crank);
        __syncwarp();
    } else if (warp == 1) {
        if (lane == 0 && crank == 0)
            run_mma_pair<BN>(a, tmem, smem, ctl);
        __syncwarp();
    } else if (warp < kRedWarp0 || a.chain) {
        run_epilogue<BN, true>(a, sch, tmem, ctl, warp, lane, blockIdx.x / 2, gridDim.x / 2, crank);
    } else {
        run_consumer<BN>(a, ctl, lane);
    }

    ptx::tc_fence_before();
    __syncthreads();
    ptx::cluster_sync(); // no CTA leaves while its peer may still signal it
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc_pair(tmem, Cfg::kTmemCols);
    }
}

} // namespace gemm_rs
