// Tiling of packed (varlen) samples, shared by the scheduler and the attention kernels.
//
// Query tiles and key/value blocks start at their sample's first token, so a
// block never straddles two samples except for the ragged tail of the sample's
// last block, which the kernels mask. For causal attention, key block n of a
// sample is needed by query rows from block n on; the block holding the
// diagonal, and any block that runs past the sample end, get an element mask,
// every other block is either fully visible or skipped.
#pragma once

#include <cstdint>

#include "common.cuh"

namespace usp {

// Number of key/value blocks a query tile starting at row q0 of sample [s, e) visits.
__host__ __device__ __forceinline__ int kv_blocks_for_query_tile(int q0, int s, int e, int causal) {
    if (q0 >= e) return 0;
    if (causal) {
        const int last = (q0 + kTileM - 1 < e - 1) ? (q0 + kTileM - 1) : (e - 1);
        return (last - s) / kBlockN + 1;
    }
    return (e - s + kBlockN - 1) / kBlockN;
}

// First query block (index from the sample start, 128 rows each) that key block n sees.
__host__ __device__ __forceinline__ int first_query_block_for_kv_block(int n, int causal) {
    return causal ? n : 0;
}

__host__ __device__ __forceinline__ int query_blocks_in_sample(int s, int e) {
    return (e - s + kTileM - 1) / kTileM;
}

// Scheduling cost of a forward item of `rows` query rows: KV blocks over its query tiles.
__host__ __device__ __forceinline__ int fwd_item_cost(int tile, int s, int e, int causal, int rows) {
    const int q0 = s + tile * rows;
    int c = 0;
    for (int r = 0; r < rows; r += kTileM) c += kv_blocks_for_query_tile(q0 + r, s, e, causal);
    return c;
}

// Scheduling cost of a backward item: query blocks it visits, times query heads per kv head.
__host__ __device__ __forceinline__ int bwd_item_cost(int tile, int s, int e, int causal, int group) {
    const int nq = query_blocks_in_sample(s, e);
    return group * (nq - first_query_block_for_kv_block(tile, causal));
}

}  // namespace usp
