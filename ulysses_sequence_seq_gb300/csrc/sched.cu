// Varlen work scheduler: validates cu_seqlens on the device and builds the list of
// attention work items, heaviest first (longest-processing-time order), so that the
// long causal tiles at the end of long samples start early and the grid's tail is
// made of short items.
//
// One CTA: sample tiles are counted and prefix-summed, every (sample, tile) gets a
// cost in key/value blocks, a counting sort over the cost puts the items in
// descending cost order, and each (sample, tile) is expanded to all heads, kept
// adjacent so that query heads sharing a key/value head run close together.
#include <cuda_runtime.h>

#include "common.cuh"
#include "sched.cuh"
#include "tiles.cuh"

namespace usp {

__device__ __forceinline__ int find_sample(const int* prefix, int nseq, int p) {
    // largest b with prefix[b] <= p (prefix is non-decreasing, prefix[0] = 0)
    int lo = 0, hi = nseq - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (prefix[mid] <= p) lo = mid;
        else hi = mid - 1;
    }
    return lo;
}

__global__ void __launch_bounds__(1024) schedule_kernel(SchedArgs a) {
    __shared__ int bad;
    __shared__ int total_tiles;
    const int tid = threadIdx.x;
    const int nthr = blockDim.x;
    if (tid == 0) bad = 0;
    for (int c = tid; c < a.hist_len; c += nthr) a.hist[c] = 0;
    __syncthreads();
    if (tid == 0 && (a.cu[0] != 0 || (int64_t)a.cu[a.num_seqs] != a.T)) bad = 1;
    for (int b = tid; b < a.num_seqs; b += nthr)
        if (a.cu[b + 1] < a.cu[b]) bad = 1;
    __syncthreads();
    if (bad) {
        if (tid == 0) {
            a.hdr->status = USP_ERR_DEVICE_CHECK;
            if (a.bwd) a.hdr->bwd_count = 0;
            else a.hdr->fwd_count = 0;
        }
        return;
    }
    const int rows = a.bwd ? kBwdRowsPerItem : kFwdRowsPerItem;
    if (tid == 0) {
        int acc = 0;
        for (int b = 0; b < a.num_seqs; ++b) {
            a.prefix[b] = acc;
            acc += (a.cu[b + 1] - a.cu[b] + rows - 1) / rows;
        }
        a.prefix[a.num_seqs] = acc;
        total_tiles = acc;
    }
    __syncthreads();
    const int ntiles = total_tiles;
    if ((int64_t)ntiles * a.heads > a.max_items) {  // cannot happen for valid cu_seqlens
        if (tid == 0) {
            a.hdr->status = USP_ERR_DEVICE_CHECK;
            if (a.bwd) a.hdr->bwd_count = 0;
            else a.hdr->fwd_count = 0;
        }
        return;
    }
    for (int p = tid; p < ntiles; p += nthr) {
        const int b = find_sample(a.prefix, a.num_seqs, p);
        const int tile = p - a.prefix[b];
        const int s = a.cu[b], e = a.cu[b + 1];
        int cost = a.bwd ? bwd_item_cost(tile, s, e, a.causal, a.group) : fwd_item_cost(tile, s, e, a.causal);
        cost = cost < 0 ? 0 : (cost >= a.hist_len ? a.hist_len - 1 : cost);
        atomicAdd(&a.hist[cost], 1);
    }
    __syncthreads();
    if (tid == 0) {  // exclusive scan from the highest cost down: bucket start offsets
        int acc = 0;
        for (int c = a.hist_len - 1; c >= 0; --c) {
            const int n = a.hist[c];
            a.hist[c] = acc;
            acc += n;
        }
    }
    __syncthreads();
    for (int p = tid; p < ntiles; p += nthr) {
        const int b = find_sample(a.prefix, a.num_seqs, p);
        const int tile = p - a.prefix[b];
        const int s = a.cu[b], e = a.cu[b + 1];
        int cost = a.bwd ? bwd_item_cost(tile, s, e, a.causal, a.group) : fwd_item_cost(tile, s, e, a.causal);
        cost = cost < 0 ? 0 : (cost >= a.hist_len ? a.hist_len - 1 : cost);
        const int pos = atomicAdd(&a.hist[cost], 1);
        for (int h = 0; h < a.heads; ++h) {
            WorkItem w;
            w.head = h;
            w.seq = b;
            w.tile = tile;
            w.cost = cost;
            a.items[(int64_t)pos * a.heads + h] = w;
        }
    }
    if (tid == 0) {
        a.hdr->status = USP_OK;
        if (a.bwd) a.hdr->bwd_count = ntiles * a.heads;
        else a.hdr->fwd_count = ntiles * a.heads;
    }
}

cudaError_t launch_schedule(const SchedArgs& a, cudaStream_t s) {
    schedule_kernel<<<1, 1024, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace usp
