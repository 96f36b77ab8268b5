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
    int bwd;             // 0: forward items (two 128-row query tiles), 1: backward items (one kv tile)
    int causal;
    int group;           // query heads per key/value head
    int hist_len;
    int max_items;
    WsHeader* hdr;
    int* hist;
    int* prefix;
    int* sbase;          // backward: per-sample start in the work order, in tiles
    WorkItem* items;
};

cudaError_t launch_schedule(const SchedArgs& a, cudaStream_t s);

}  // namespace usp
