// The prefill tile classifier: which view(s) a 128x128 (query, key) tile needs.
//
// The pages compute prefill as three attention passes -- local(window, exact
// RoPE) + remote(all, aliased) - remote(window, aliased) -- merged on
// log-sum-exp statistics (ResearchPod transcript on the prefill phase).  The
// merge is exactly one softmax in which each key is scored once with the view
// its distance selects, so a tile only needs the view(s) its pairs select:
// a tile wholly inside the window needs exact scores, a tile wholly outside
// it needs aliased scores, and only the tiles the boundary i - j = w crosses
// need both.
#pragma once

namespace jl {

enum TileClass : int { kTileMasked = 0, kTileExact = 1, kTileRemote = 2, kTileBand = 3 };

// Query rows [i0, i0+bm) and key columns [j0, j0+bn), clipped to S; g the
// group factor, w the local window (key j is local for query i iff
// 0 <= i - j < w).  With g == 1 both views coincide and the tile is exact.
__host__ __device__ inline int tile_class(int i0, int j0, int bm, int bn, int S, int w, int g)
{
    int i1 = (i0 + bm < S ? i0 + bm : S) - 1;  // last query row of the tile
    int j1 = (j0 + bn < S ? j0 + bn : S) - 1;  // last key column of the tile
    if (j0 > i1) return kTileMasked;           // every key after every query
    if (g == 1) return kTileExact;
    if (i1 - j0 < w) return kTileExact;        // largest distance still local
    if (i0 - j1 >= w) return kTileRemote;      // smallest distance already remote
    return kTileBand;
}

}  // namespace jl
