// Tile schedule of the fused GEMM+RS kernel: the rank-offset swizzle.
//
// Rank r visits its chunks in the order (r+1+s) mod W, s = 0 .. W-1.  So the
// W-1 remote chunks come first and its own chunk r last
// ("flux实现：sm80 gemm+rs", section "gemmrs版本的swizzle如何编排").  Each
// rank's start is shifted by its rank, so at every step the W ranks target W
// different chunks ("flux精读" §4.1 Tile coordination swizzling).  The
// communication unit is one output tile, not one chunk (same section of the
// first page: ReduceScatterOp<T, kM, kN, ...>): a row tile belongs to the
// chunk of its first row, and the chunk shape need not match the tile shape.
//
// The order of one rank:
//   for each column group (G column tiles; one group when G >= nN):
//     for each step s = 0 .. W-1 (chunk (r+1+s) mod W):
//       for each row group of the chunk (RG row tiles; one group when RG
//       covers the chunk):
//         one sweep over the column tiles of the column group,
//           for each row tile of the row group, ascending.
// Inside a column group of gn tiles, rank r's sweep starts at the group's tile
// ((W-r) mod W)*gn/W and wraps around within the group, so all ranks cover
// the same columns in a group and each B panel of the group stays in use for
// all W steps.  Row groups bound the A rows a sweep keeps live, so they can
// stay in L2 while the columns go by.
//
// Two rank orders:
//   interleaved  the ranks advance side by side: global entry g is rank
//                (g mod W)'s (g / W)-th tile, so at every step the W ranks
//                target W different chunks.  Every sweep runs forward, and the
//                rank that reaches a tile at step s+1 (rank r-1) starts its
//                sweep gn/W columns earlier than rank r: it reaches the tile
//                between 1 - 1/W and about 2 steps after rank r did, so a
//                tile's contributions arrive in step order.
//   sequential   for each column group, the ranks run one after another: the
//                group's entries are rank 0's tiles of the group, then rank
//                1's, and so on.  One rank's operands and one group's running
//                sums are live at a time, and a tile's contributions arrive in
//                rank order, most of a rank's pass over the group apart.
// The chain reduction folds a tile's contributions in that arrival order, its
// "position": the step (interleaved) or the rank (sequential).
#pragma once

#include <cstdint>

namespace gemm_rs {

struct Sched {
    int W;
    int nM, nN;
    int bm_shift; // log2(BM)
    int64_t R;    // rows per chunk, M / W
    int G;        // column tiles per group (>= nN: one group)
    int RG;       // row tiles per row group (>= a chunk's row tiles: one group)
    int seq;      // 1: ranks one after another, 0: ranks side by side
};

// Decode global entry g into (r, mt, nt) and the tile's position (0 .. W-1)
// in its contributions' arrival order: the step in which rank r reaches the
// tile's chunk (interleaved), or r (sequential).  g must be < W*nM*nN.
//
// Every quantity fits in 32 bits (the host bounds W*nM*nN below 2^31 and M
// below 2^31), and the arithmetic is 32-bit: the producer decodes each tile
// on its critical path, where 64-bit divisions cost about a microsecond.
__host__ __device__ __forceinline__ void decode_tile(const Sched &s, int64_t g64, int &r, int &mt,
                                                     int &nt, int &pos)
{
    const uint32_t g = static_cast<uint32_t>(g64);
    const uint32_t W = static_cast<uint32_t>(s.W);
    const uint32_t nM = static_cast<uint32_t>(s.nM);
    const uint32_t nN = static_cast<uint32_t>(s.nN);
    const uint32_t G = static_cast<uint32_t>(s.G) < nN ? static_cast<uint32_t>(s.G) : nN;
    // Every column group but the last is full, so the group index follows
    // directly.  p becomes rank r's index inside the group.
    uint32_t p, grp, rr;
    if (s.seq) {
        const uint32_t full = W * nM * G; // entries of a full group
        grp = g / full;
        const uint32_t gn = (nN - grp * G) < G ? (nN - grp * G) : G;
        const uint32_t q = g - grp * full;
        const uint32_t per_rank = nM * gn;
        rr = q / per_rank;
        p = q - rr * per_rank;
    } else {
        rr = g % W;
        p = g / W;
        grp = p / (G * nM);
        p -= grp * G * nM;
    }
    r = static_cast<int>(rr);
    const uint32_t g0 = grp * G;
    const uint32_t gn = (nN - g0) < G ? (nN - g0) : G;
    const uint32_t rot = (((W - rr) % W) * gn) / W;
    const uint32_t R = static_cast<uint32_t>(s.R);
    const uint32_t bmask = (1u << s.bm_shift) - 1u;
    // Step st visits chunk c = (r+1+st) mod W, whose row tiles are the ones
    // whose first row lies in the chunk: [ceil(c*R/BM), ceil((c+1)*R/BM)).
    uint32_t c = rr + 1 >= W ? rr + 1 - W : rr + 1;
    uint32_t first = (c * R + bmask) >> s.bm_shift;
    for (uint32_t st = 0; st < W; ++st) {
        const uint32_t last = ((c + 1) * R + bmask) >> s.bm_shift;
        const uint32_t cnt = last - first;
        const uint32_t items = cnt * gn;
        if (p < items) {
            // Every row group but the chunk's last is full.
            const uint32_t RG = static_cast<uint32_t>(s.RG) < cnt ? static_cast<uint32_t>(s.RG) : cnt;
            const uint32_t rg = p / (RG * gn);
            const uint32_t q = p - rg * RG * gn;
            const uint32_t rn = (cnt - rg * RG) < RG ? (cnt - rg * RG) : RG;
            const uint32_t jl = q / rn;
            mt = static_cast<int>(first + rg * RG + (q - jl * rn));
            uint32_t n = jl + rot;
            if (n >= gn)
                n -= gn;
            nt = static_cast<int>(g0 + n);
            pos = s.seq ? static_cast<int>(rr) : static_cast<int>(st);
            return;
        }
        p -= items;
        if (++c == W) {
            c = 0;
            first = 0;
        } else {
            first = last;
        }
    }
    mt = -1;
    nt = -1;
    pos = -1;
}

__host__ __device__ __forceinline__ void decode_tile(const Sched &s, int64_t g, int &r, int &mt,
                                                     int &nt)
{
    int pos;
    decode_tile(s, g, r, mt, nt, pos);
}

} // namespace gemm_rs
