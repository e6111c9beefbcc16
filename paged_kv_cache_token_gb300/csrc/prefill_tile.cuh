// The work of one prefill CTA of the tensor-core kernels: two chains (c = 0, 1) of 128 query
// rows that share one KV head's key/value stream, each with its own scores, softmax state
// and output accumulator in tensor memory.
//   heads_per_tile == 2 (an even KV group): the same 128 rows for query heads 2u and 2u + 1;
//   heads_per_tile == 1 (one query head per KV head): query tiles 2u and 2u + 1 of one head.
// In the second form the stream covers the keys of the later tile; the earlier tile sees
// its extra keys fully masked (they lie past every one of its rows).  A chain whose tile
// lies past the end of the chunk has no valid rows and writes nothing.
#pragma once

#include "common.cuh"
#include "launch.h"

namespace pkv {

struct PairTile {
    int r, g, q_off;
    int head[2], q_row[2], rows_valid[2], first_pos[2];
    int kv_len, n_kv, npages_seq;   // of the key/value stream both chains share
};

// tl: the tile record {request, unit (query tile, or pair of query tiles), slot, -}
__device__ __forceinline__ PairTile pair_tile(const StepArgs& a, const int4 tl, int rows_per_tile,
                                              int keys_per_tile) {
    PairTile t;
    t.r = tl.x;
    const bool heads = a.heads_per_tile == 2;
    const int ctx = a.context_lens[t.r];
    const int ql = a.q_lens[t.r];
    t.q_off = a.q_offsets[t.r];
    int kv = 0;
#pragma unroll
    for (int c = 0; c < 2; ++c) {
        const int qt = heads ? tl.y : 2 * tl.y + c;
        t.head[c] = heads ? 2 * tl.z + c : tl.z;
        t.q_row[c] = t.q_off + qt * rows_per_tile;
        t.rows_valid[c] = max(0, min(rows_per_tile, ql - qt * rows_per_tile));
        t.first_pos[c] = ctx + qt * rows_per_tile;
        if (t.rows_valid[c] > 0) kv = max(kv, t.first_pos[c] + t.rows_valid[c]);
    }
    t.g = t.head[0] / (a.num_q_heads / a.num_kv_heads);
    t.kv_len = kv;
    t.n_kv = cdiv(kv, keys_per_tile);
    t.npages_seq = cdiv(kv, kPage);
    return t;
}

}  // namespace pkv
