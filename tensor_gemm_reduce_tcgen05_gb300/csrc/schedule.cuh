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
// Inside a chunk, rank r walks the column tiles starting at (r*nN)/W.  For
// each column tile it takes the chunk's row tiles in ascending order, so the
// chunk's A rows stay in L2 while the column tiles go by.  The ranks advance
// side by side: global entry g is rank (g mod W)'s (g / W)-th tile.
#pragma once

#include <cstdint>

namespace gemm_rs {

struct Sched {
    int W;
    int nM, nN;
    int bm_shift; // log2(BM)
    int64_t R;    // rows per chunk, M / W
};

__host__ __device__ __forceinline__ int64_t ceil_shift(int64_t x, int s)
{
    return (x + (int64_t(1) << s) - 1) >> s;
}

// Decode global entry g into (r, mt, nt).  g must be < W*nM*nN.
__host__ __device__ __forceinline__ void decode_tile(const Sched &s, int64_t g, int &r, int &mt,
                                                     int &nt)
{
    r = static_cast<int>(g % s.W);
    int64_t p = g / s.W;
    const int64_t rot = (static_cast<int64_t>(r) * s.nN) / s.W;
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
        const int64_t items = cnt * s.nN;
        if (p < items) {
            const int64_t j = p / cnt;
            const int64_t q = p - j * cnt;
            mt = static_cast<int>(first + q);
            int64_t n = j + rot;
            if (n >= s.nN)
                n -= s.nN;
            nt = static_cast<int>(n);
            return;
        }
        p -= items;
    }
    mt = -1;
    nt = -1;
}

} // namespace gemm_rs
