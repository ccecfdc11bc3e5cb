// The fused all-gather + GEMM (AG+GEMM) kernel for sm_103a: the first GEMM of
// a tensor-parallel FFN, whose input rows are all-gathered from the ranks
// ("flux精读" §3 Design: the AllGather GEMM; "通信 overlap 实现", section
// "Flux 的 tile 级融合解决了什么？": AG+GEMM, prologue fusion).
//
// W logical ranks on one GPU.  Rank r holds row chunk r of X (rows
// [r*M/W, (r+1)*M/W)) and the column shard B1_r; it needs all of X.  The
// all-gather delivers chunk c to rank r as a copy into rank r's gather buffer
// G_r, and signals it with a 32-bit counter per (rank, chunk) (the pages: a
// signal per tile, set when its copy is done, 32-bit contiguous memory).
// Each GEMM CTA waits for the signal of the chunk its tile reads, in the order
// the chunks are sent, before it loads the tile; a rank's own chunk needs no
// wait ("flux精读" §4.1: each rank starts at its own chunk).
//
// One persistent kernel emulates all ranks: the copies that a copy engine
// would make between GPUs are made by copy warps of the same kernel, so no
// kernel ever waits for another launch.  The kernel is launched cooperatively
// (all CTAs resident), and every wait is bounded.
//
// CTA pair (cluster of 2, tcgen05.mma.cta_group::2), 256x256 output tiles,
// 320 threads per CTA:
//   warp 0      TMA producer: waits for the tile's chunk signal (acquire, then
//               a proxy fence so that the TMA reads see the copied rows), then
//               loads its 128 rows of A (from X for the rank's own chunk, from
//               G_r otherwise) and its 128 columns of B1_r per k-block.
//   warp 1      TMEM allocation and, in the even CTA, the MMA issuer (the
//               CTA-pair mainloop of the GEMM+RS kernel).
//   warps 2-5   epilogue: alpha * acc from TMEM, stored to H_r.
//   warps 6-9   copy role: the all-gather.  Each chunk copy is cut into slices;
//               CTA b copies slices b, b + grid, ... in the order the chunks are
//               consumed, and after each slice adds one to its (rank, chunk)
//               counter with release semantics.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>

#include "gemm_rs_kernel.cuh"
#include "ptx.cuh"

namespace gemm_rs {

struct AgArgs {
    int W, M, N, K;
    int nK;          // k-blocks of 64
    int nMs;         // 256-row tiles
    int nN;          // 256-column tiles
    int R;           // rows per chunk (M / W)
    int cntp;        // 256-row tiles per chunk
    int64_t total;   // W * nMs * nN work items
    float alpha;
    void *H;         // [W][M][N], bf16 or fp32
    int y_fp32;
    const uint16_t *X; // [M][K] bf16
    uint16_t *G;     // [W][M][K] bf16 gather buffers
    uint32_t *ready; // [W][W] chunk signals
    uint32_t *status;
    int32_t *record; // optional: (r, mt2, nt, pair) per entry
    int slice_rows;  // rows per copy slice
    int nslices;     // slices per chunk
    uint32_t epoch;  // this call's index: a chunk is ready at epoch * nslices
    unsigned long long timeout;
    int skip_copies; // debug: deliver nothing, so remote-chunk waits run out
    int b4d;         // 1: B1's map is 4D (one box per stage), 0: 3D (one per 64 columns)
};

constexpr uint32_t kBarCopy = 2; // named barrier of the 128 copy threads

// Decode entry g of the AG order: rank r = g / T (T = nMs*nN tiles per rank);
// inside a rank, chunk step s (chunk (r+s) mod W), then column tile nt, then
// the chunk's 256-row tile.
// 32-bit arithmetic: the host bounds the entry count below 2^31.
__host__ __device__ __forceinline__ void ag_decode(const AgArgs &g, int64_t e64, int &r, int &mt2,
                                                   int &nt, int &c)
{
    const uint32_t e = static_cast<uint32_t>(e64);
    const uint32_t T = static_cast<uint32_t>(g.nMs) * static_cast<uint32_t>(g.nN);
    const uint32_t rr = e / T;
    const uint32_t p = e - rr * T;
    const uint32_t cntp = static_cast<uint32_t>(g.cntp);
    const uint32_t per_chunk = cntp * static_cast<uint32_t>(g.nN);
    const uint32_t s = p / per_chunk;
    const uint32_t q = p - s * per_chunk;
    uint32_t cc = rr + s;
    if (cc >= static_cast<uint32_t>(g.W))
        cc -= static_cast<uint32_t>(g.W);
    const uint32_t n = q / cntp;
    r = static_cast<int>(rr);
    c = static_cast<int>(cc);
    nt = static_cast<int>(n);
    mt2 = static_cast<int>(cc * cntp + (q - n * cntp));
}

// Bounded wait for a chunk signal: true once *p has reached `target` (compared
// modulo 2^32), false when `limit` cycles pass or the CTA aborts.
// Checked build (GEMM_RS_CHECKED): as in the GEMM+RS kernel, an access outside
// its buffer is skipped and recorded in the status word; the normal build
// compiles the checks away.
__device__ __forceinline__ bool ag_bounds_ok(const AgArgs &g, bool ok)
{
#ifdef GEMM_RS_CHECKED
    if (!ok)
        atomicCAS(g.status, 0u, static_cast<uint32_t>(kStatusOutOfBounds));
    return ok;
#else
    (void)g;
    (void)ok;
    return true;
#endif
}

__device__ __forceinline__ bool wait_signal(const uint32_t *p, uint32_t target, unsigned long long limit,
                                            const volatile int *abort_flag)
{
    const long long t0 = clock64();
    while (true) {
        const uint32_t v = ptx::ld_acquire_gpu(p);
        if (static_cast<int32_t>(v - target) >= 0)
            return true;
        if (*abort_flag != 0 || static_cast<unsigned long long>(clock64() - t0) > limit)
            return false;
        __nanosleep(128);
    }
}

template <int BN>
__device__ __forceinline__ void run_ag_producer(const AgArgs &g, const KernelArgs &ka,
                                                const CUtensorMap *tmX, const CUtensorMap *tmG,
                                                const CUtensorMap *tmB, uint8_t *smem, SmemCtl *ctl,
                                                uint32_t crank)
{
    using Cfg = PairCfg<BN>;
    const volatile int *abort_flag = &ctl->abort;
    const uint64_t pol = ptx::policy_evict_normal();
    const int64_t ncl = gridDim.x / 2;
    const int64_t cid = blockIdx.x / 2;
    const uint32_t target = g.epoch * static_cast<uint32_t>(g.nslices);
    uint32_t stage = 0, phase = 0;
    int64_t issued = 0;
    bool ok = true;
    for (int64_t e = cid; e < g.total && ok; e += ncl) {
        int r, mt2, nt, c;
        ag_decode(g, e, r, mt2, nt, c);
        if (g.record != nullptr && crank == 0) {
            int32_t *rec = g.record + 4 * e;
            rec[0] = r;
            rec[1] = mt2;
            rec[2] = nt;
            rec[3] = static_cast<int32_t>(cid);
        }
        const bool local = c == r;
        if (!local && ag_bounds_ok(g, r >= 0 && r < g.W && c >= 0 && c < g.W)) {
            if (!wait_signal(g.ready + r * g.W + c, target, g.timeout, abort_flag)) {
                ok = false;
                break;
            }
            // The copied rows were written by generic stores; the TMA reads
            // below go through the async proxy.
            asm volatile("fence.proxy.async.global;" ::: "memory");
        }
        const int row = (2 * mt2 + static_cast<int>(crank)) * kBM;
        for (int kb = 0; kb < g.nK; ++kb) {
            if (!ptx::mbar_wait_cluster(ptx::smem_u32(&ctl->empty[stage]), phase ^ 1u, g.timeout,
                                        abort_flag)) {
                ok = false;
                break;
            }
            const uint32_t fb = ptx::smem_u32(&ctl->full[stage]);
            if (crank == 0)
                ptx::mbar_arrive_expect_tx(fb, 2 * Cfg::kStageBytes);
            const uint32_t fb_leader = ptx::mapa(fb, 0);
            const uint32_t sa = ptx::smem_u32(smem + stage * Cfg::kStageBytes);
            if (local)
                ptx::tma_load_3d_pair(sa, tmX, fb_leader, kb * kBK, row, 0, pol);
            else
                ptx::tma_load_3d_pair(sa, tmG, fb_leader, kb * kBK, row, r, pol);
            if (g.b4d) {
                ptx::tma_load_4d_pair(sa + Cfg::kABytes, tmB, fb_leader, 0, kb * kBK,
                                      (nt * BN + static_cast<int>(crank) * (BN / 2)) / 64, r, pol);
            } else {
#pragma unroll
                for (int j = 0; j < BN / 128; ++j)
                    ptx::tma_load_3d_pair(sa + Cfg::kABytes + j * 8192, tmB, fb_leader,
                                          nt * BN + static_cast<int>(crank) * (BN / 2) + j * 64,
                                          kb * kBK, r, pol);
            }
            ++issued;
            if (++stage == Cfg::kStages) {
                stage = 0;
                phase ^= 1u;
            }
        }
    }
    if (ok) {
        // Tail: every stage released by the pair's MMA before the CTA exits.
        for (int i = 0; i < Cfg::kStages; ++i) {
            if (!ptx::mbar_wait_cluster(ptx::smem_u32(&ctl->empty[stage]), phase ^ 1u, g.timeout,
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
        report(ka, ctl, kStatusTimeoutProducer);
    pair_producer_finish(ctl, crank, ok, issued, Cfg::kStages, g.timeout);
}

// Epilogue (warps 2-5): H_r[m, n] = alpha * acc, 32 columns per step.
template <int BN>
__device__ __forceinline__ void run_ag_epilogue(const AgArgs &g, const KernelArgs &ka, uint32_t tmem,
                                                SmemCtl *ctl, int warp, int lane, uint32_t crank)
{
    const volatile int *abort_flag = &ctl->abort;
    const int q = warp & 3;
    const uint32_t lane_base = static_cast<uint32_t>(q * 32) << 16;
    const int64_t ncl = gridDim.x / 2;
    const int64_t cid = blockIdx.x / 2;
    int it = 0;
    for (int64_t e = cid; e < g.total; e += ncl, ++it) {
        int r, mt2, nt, c;
        ag_decode(g, e, r, mt2, nt, c);
        const int buf = it & 1;
        const uint32_t aph = static_cast<uint32_t>(it >> 1) & 1u;
        const bool waited =
            ptx::mbar_wait_cluster(ptx::smem_u32(&ctl->acc_full[buf]), aph, g.timeout, abort_flag);
        if (ptx::named_bar_or(kBarEpi, 128, !waited)) {
            if (warp == kEpiWarp0 && lane == 0)
                report(ka, ctl, kStatusTimeoutEpilogue);
            break;
        }
        ptx::tc_fence_after();
        const int64_t m = static_cast<int64_t>(2 * mt2 + static_cast<int>(crank)) * kBM + q * 32 + lane;
        const bool row_ok = m < g.M;
#pragma unroll 1
        for (int slab = 0; slab < BN / 32; ++slab) {
            uint32_t v[32];
            if (g.nK > 0) {
                ptx::tmem_ld_32x32b_x32(tmem + lane_base + static_cast<uint32_t>(buf * BN + slab * 32), v);
            } else {
#pragma unroll
                for (int i = 0; i < 32; ++i)
                    v[i] = 0u;
            }
            if (slab == BN / 32 - 1) {
                ptx::tc_fence_before();
                __syncwarp();
                if (lane == 0)
                    ptx::mbar_arrive_cluster(ptx::mapa(ptx::smem_u32(&ctl->acc_empty[buf]), 0));
            }
            const int64_t n0 = static_cast<int64_t>(nt) * BN + slab * 32;
            const int64_t base = (static_cast<int64_t>(r) * g.M + m) * g.N;
#pragma unroll
            for (int g8 = 0; g8 < 4; ++g8) {
                const int64_t n = n0 + 8 * g8;
                if (!row_ok || n >= g.N) // N is a multiple of 8
                    continue;
                if (!ag_bounds_ok(g, r >= 0 && r < g.W && m >= 0 && m < g.M && n + 8 <= g.N))
                    continue;
                float p[8];
#pragma unroll
                for (int e2 = 0; e2 < 8; ++e2)
                    p[e2] = g.alpha * __uint_as_float(v[8 * g8 + e2]);
                if (g.y_fp32) {
                    float *yp = static_cast<float *>(g.H) + base + n;
                    ptx::st_f4(yp, make_float4(p[0], p[1], p[2], p[3]));
                    ptx::st_f4(yp + 4, make_float4(p[4], p[5], p[6], p[7]));
                } else {
                    const __nv_bfloat162 h0 = __floats2bfloat162_rn(p[0], p[1]);
                    const __nv_bfloat162 h1 = __floats2bfloat162_rn(p[2], p[3]);
                    const __nv_bfloat162 h2 = __floats2bfloat162_rn(p[4], p[5]);
                    const __nv_bfloat162 h3 = __floats2bfloat162_rn(p[6], p[7]);
                    uint4 w;
                    w.x = *reinterpret_cast<const uint32_t *>(&h0);
                    w.y = *reinterpret_cast<const uint32_t *>(&h1);
                    w.z = *reinterpret_cast<const uint32_t *>(&h2);
                    w.w = *reinterpret_cast<const uint32_t *>(&h3);
                    ptx::st_u4(static_cast<uint16_t *>(g.H) + base + n, w);
                }
            }
        }
    }
}

// Copy role (warps 6-9): the all-gather.  Slice q of the global slice order is
// rank r's step s (chunk c = (r+s) mod W, s = 1 .. W-1), slice j of the chunk:
// rows [c*R + j*slice_rows, ... + slice_rows) of X into the same rows of G_r.
__device__ __forceinline__ void run_ag_copy(const AgArgs &g, int ct)
{
    const int64_t per_rank = static_cast<int64_t>(g.W - 1) * g.nslices;
    const int64_t total = per_rank * g.W;
    const int64_t n16 = static_cast<int64_t>(g.slice_rows) * g.K / 8; // 16-byte units per slice
    if (g.skip_copies)
        return;
    for (int64_t q = blockIdx.x; q < total; q += gridDim.x) {
        const int r = static_cast<int>(q / per_rank);
        const int64_t rem = q - static_cast<int64_t>(r) * per_rank;
        const int s = 1 + static_cast<int>(rem / g.nslices);
        const int j = static_cast<int>(rem - static_cast<int64_t>(s - 1) * g.nslices);
        const int c = (r + s) % g.W;
        const int64_t row0 = static_cast<int64_t>(c) * g.R + static_cast<int64_t>(j) * g.slice_rows;
        const uint4 *src = reinterpret_cast<const uint4 *>(g.X + row0 * g.K);
        uint4 *dst = reinterpret_cast<uint4 *>(g.G + (static_cast<int64_t>(r) * g.M + row0) * g.K);
        // the slice's rows [row0, row0 + slice_rows) of X and of rank r's buffer
        const bool in = ag_bounds_ok(g, row0 >= 0 && row0 + g.slice_rows <= g.M && r < g.W &&
                                            c >= 0 && c < g.W);
        int64_t i = in ? ct : n16;
        for (; i + 3 * 128 < n16; i += 4 * 128) {
            uint4 t[4];
#pragma unroll
            for (int u = 0; u < 4; ++u)
                t[u] = ptx::ld_nc_u4(src + i + u * 128);
#pragma unroll
            for (int u = 0; u < 4; ++u)
                ptx::st_u4(dst + i + u * 128, t[u]);
        }
        for (; i < n16; i += 128)
            ptx::st_u4(dst + i, ptx::ld_nc_u4(src + i));
        // Every copy thread's stores are ordered before the signal's release.
        ptx::named_bar_sync(kBarCopy, 128);
        if (ct == 0 && in)
            ptx::atom_add_acq_rel_gpu(g.ready + r * g.W + c, 1u);
    }
}

template <int BN>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    ag_gemm_pair_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmG,
                        const __grid_constant__ CUtensorMap tmB, const AgArgs g)
{
    using Cfg = PairCfg<BN>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = ptx::smem_u32(smem_raw);
    uint8_t *smem = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
    SmemCtl *ctl = reinterpret_cast<SmemCtl *>(smem + Cfg::kStages * Cfg::kStageBytes);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t crank = ptx::cluster_ctarank();

    // The fields of the GEMM+RS arguments that the shared mainloop and the
    // status report read.
    KernelArgs ka = {};
    ka.W = g.W;
    ka.nK = g.nK;
    ka.total = g.total;
    ka.status = g.status;
    ka.timeout = g.timeout;

    if (threadIdx.x == 0) {
        for (int s = 0; s < Cfg::kStages; ++s) {
            ptx::mbar_init(ptx::smem_u32(&ctl->full[s]), 1);
            ptx::mbar_init(ptx::smem_u32(&ctl->empty[s]), 1);
        }
        for (int b = 0; b < 2; ++b) {
            ptx::mbar_init(ptx::smem_u32(&ctl->acc_full[b]), 1);
            ptx::mbar_init(ptx::smem_u32(&ctl->acc_empty[b]), 8); // 4 epilogue warps x 2 CTAs
        }
        ptx::mbar_init(ptx::smem_u32(&ctl->drain), 1);
        ptx::mbar_init(ptx::smem_u32(&ctl->peer_drained), 1);
        ctl->abort = 0;
        ptx::fence_barrier_init();
    }
    if (warp == 0 && lane == 0 && g.nK > 0) {
        ptx::prefetch_tensormap(&tmX);
        ptx::prefetch_tensormap(&tmG);
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

    if (warp == 0) {
        if (lane == 0)
            run_ag_producer<BN>(g, ka, &tmX, &tmG, &tmB, smem, ctl, crank);
        __syncwarp();
    } else if (warp == 1) {
        if (lane == 0 && crank == 0)
            run_mma_pair<BN>(ka, tmem, smem, ctl);
        __syncwarp();
    } else if (warp < kRedWarp0) {
        run_ag_epilogue<BN>(g, ka, tmem, ctl, warp, lane, crank);
    } else {
        run_ag_copy(g, static_cast<int>(threadIdx.x) - kRedWarp0 * 32);
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
