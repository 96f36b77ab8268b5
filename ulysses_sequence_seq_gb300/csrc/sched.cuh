// Varlen work scheduler interface (see sched.cu).
#pragma once

#include <cuda_runtime.h>

#include "common.cuh"

namespace usp {

struct SchedArgs {
    const int32_t* cu;   // device cu_seqlens [num_seqs + 1]
    int num_seqs;
    int64_t T;
    int heads;           // query heads (forward) or key/value heads (backward)
    int bwd;             // 0: forward items (fwd_rows query rows), 1: backward items (one kv tile)
    int fwd_rows;        // fwd_rows_per_item(head_dim) for the forward
    int causal;
    int group;           // query heads per key/value head
    int hist_len;
    int max_items;
    WsHeader* hdr;
    int* hist;
    int* prefix;
    int* sbase;          // per-sample start in the work order, in tiles
    int head_major_from; // samples of at least this many tokens are ordered head by head
    WorkItem* items;
};

// Writes the work list and the header (status, item count, a zeroed item counter). With
// after_prep the launch may overlap the backward's operand-conversion kernel launched just
// before it on s.
cudaError_t launch_schedule(const SchedArgs& a, cudaStream_t s, bool after_prep);

// Sample length from which work items are ordered head by head: the backward always (its
// persistent CTAs follow the list order closely), the forward once a sample's keys and
// values for all heads exceed half of the 129 MB L2.
inline int head_major_from_tokens(int hkv, int head_dim, int bwd) {
    if (bwd) return 0;
    const int64_t kv_bytes_per_token = 2ll * hkv * head_dim * 2;
    const int64_t t = (int64_t)(64ll << 20) / (kv_bytes_per_token > 0 ? kv_bytes_per_token : 1);
    return (int)(t + 1);
}

}  // namespace usp
