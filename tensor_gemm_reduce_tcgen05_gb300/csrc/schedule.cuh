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

__host__ __device__ __forceinline__ int64_t ceil_shift(int64_t x, int s)
{
    return (x + (int64_t(1) << s) - 1) >> s;
}

// Decode global entry g into (r, mt, nt) and the tile's position (0 .. W-1)
// in its contributions' arrival order: the step in which rank r reaches the
// tile's chunk (interleaved), or r (sequential).  g must be < W*nM*nN.
__host__ __device__ __forceinline__ void decode_tile(const Sched &s, int64_t g, int &r, int &mt,
                                                     int &nt, int &pos)
{
    const int64_t G = s.G < s.nN ? s.G : s.nN;
    // Every column group but the last is full, so the group index follows
    // directly.  p becomes rank r's index inside the group.
    int64_t p, grp;
    if (s.seq) {
        const int64_t full = static_cast<int64_t>(s.W) * s.nM * G; // entries of a full group
        grp = g / full;
        const int64_t gn = (s.nN - grp * G) < G ? (s.nN - grp * G) : G;
        const int64_t q = g - grp * full;
        const int64_t per_rank = static_cast<int64_t>(s.nM) * gn;
        r = static_cast<int>(q / per_rank);
        p = q - static_cast<int64_t>(r) * per_rank;
    } else {
        r = static_cast<int>(g % s.W);
        p = g / s.W;
        grp = p / (G * s.nM);
        p -= grp * G * s.nM;
    }
    const int64_t g0 = grp * G;
    const int64_t gn = (s.nN - g0) < G ? (s.nN - g0) : G;
    const int64_t rot = (static_cast<int64_t>((s.W - r) % s.W) * gn) / s.W;
    for (int st = 0; st < s.W; ++st) {
        int c = r + 1 + st;
        if (c >= s.W)
            c -= s.W;
        if (c >= s.W)
            c -= s.W;
        // row tiles whose first row lies in chunk c: [ceil(c*R/BM), ceil((c+1)*R/BM))
        const int64_t first = ceil_shift(static_cast<int64_t>(c) * s.R, s.bm_shift);
        const int64_t last = ceil_shift(static_cast<int64_t>(c + 1) * s.R, s.bm_shift);
        const int64_t cnt = last - first;
        const int64_t items = cnt * gn;
        const int64_t RG = s.RG < cnt ? s.RG : cnt;
        if (p < items) {
            // Every row group but the chunk's last is full.
            const int64_t rg = p / (RG * gn);
            const int64_t q = p - rg * RG * gn;
            const int64_t rn = (cnt - rg * RG) < RG ? (cnt - rg * RG) : RG;
            const int64_t jl = q / rn;
            mt = static_cast<int>(first + rg * RG + (q - jl * rn));
            int64_t n = jl + rot;
            if (n >= gn)
                n -= gn;
            nt = static_cast<int>(g0 + n);
            pos = s.seq ? r : st;
            return;
        }
        p -= items;
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
