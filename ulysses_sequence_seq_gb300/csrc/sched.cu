// Varlen work scheduler: validates cu_seqlens on the device and builds the list of
// attention work items.
//
// Order: samples longest first (a counting sort over their tile counts, histogram in
// shared memory, block-wide scans), and within a sample head by head, each head's
// tiles heaviest first. CTAs started close together then work on the tiles of one or a
// few (sample, head) pairs and walk the same key/value blocks (forward) or query blocks
// (backward), so the blocks they share stay in L2 instead of being fetched once per
// tile; the grid's tail is made of the cheapest tiles of the shortest samples. Heads
// sharing a key/value head are adjacent.
#include <cuda_runtime.h>

#include "common.cuh"
#include "ptx.cuh"
#include "sched.cuh"
#include "tiles.cuh"

namespace usp {

// Cost histograms up to this many buckets (48 KB) live in shared memory.
constexpr int kSchedSmemHist = 12288;

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

// In-place exclusive prefix sum of data[0..n) by the whole CTA (data in shared or global
// memory); with `rev` the sum runs from the last element down. Returns the total.
__device__ int block_exclusive_scan(int* data, int n, bool rev, int* warp_sums) {
    const int tid = threadIdx.x, nthr = blockDim.x;
    const int per = (n + nthr - 1) / nthr;
    const int b0 = tid * per;
    const int b1 = (b0 + per < n) ? b0 + per : n;
    int local = 0;
    for (int i = b0; i < b1; ++i) local += data[rev ? n - 1 - i : i];
    const int lane = tid & 31, wid = tid >> 5, nwarps = nthr >> 5;
    int x = local;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, off);
        if (lane >= off) x += y;
    }
    if (lane == 31) warp_sums[wid] = x;
    __syncthreads();
    if (wid == 0) {
        int w = lane < nwarps ? warp_sums[lane] : 0;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, w, off);
            if (lane >= off) w += y;
        }
        warp_sums[lane] = w;
    }
    __syncthreads();
    int acc = x - local + (wid > 0 ? warp_sums[wid - 1] : 0);
    const int total = warp_sums[nwarps - 1];
    for (int i = b0; i < b1; ++i) {
        const int idx = rev ? n - 1 - i : i;
        const int v = data[idx];
        data[idx] = acc;
        acc += v;
    }
    __syncthreads();
    return total;
}

__device__ __forceinline__ void fail_schedule(const SchedArgs& a) {
    a.hdr->status = USP_ERR_DEVICE_CHECK;
    if (a.bwd) a.hdr->bwd_count = 0;
    else a.hdr->fwd_count = 0;
}

// The whole work list and the call's header: its status, the item count and the counter
// the persistent attention CTAs take their items from (zeroed here).
__device__ void schedule_body(const SchedArgs& a) {
    extern __shared__ int hist_smem[];
    __shared__ int bad;
    __shared__ int warp_sums[32];
    const int tid = threadIdx.x;
    const int nthr = blockDim.x;
    int* hist = a.hist_len <= kSchedSmemHist ? hist_smem : a.hist;
    if (tid == 0) bad = 0;
    for (int c = tid; c < a.hist_len; c += nthr) hist[c] = 0;
    __syncthreads();
    if (tid == 0 && (a.cu[0] != 0 || (int64_t)a.cu[a.num_seqs] != a.T)) bad = 1;
    for (int b = tid; b < a.num_seqs; b += nthr)
        if (a.cu[b + 1] < a.cu[b]) bad = 1;
    __syncthreads();
    if (bad) {
        if (tid == 0) fail_schedule(a);
        return;
    }
    const int rows = a.bwd ? kBwdRowsPerItem : a.fwd_rows;
    // tiles per sample, then their exclusive prefix sum (prefix[num_seqs] = total)
    for (int b = tid; b <= a.num_seqs; b += nthr)
        a.prefix[b] = b < a.num_seqs ? (a.cu[b + 1] - a.cu[b] + rows - 1) / rows : 0;
    __syncthreads();
    const int ntiles = block_exclusive_scan(a.prefix, a.num_seqs + 1, false, warp_sums);
    if ((int64_t)ntiles * a.heads > a.max_items) {  // cannot happen for valid cu_seqlens
        if (tid == 0) fail_schedule(a);
        return;
    }
    // samples by tile count, longest first: bucket c holds samples of c tiles, and its
    // share of the work order is (samples in it) x c tiles
    for (int b = tid; b < a.num_seqs; b += nthr) {
        const int nt = a.prefix[b + 1] - a.prefix[b];
        atomicAdd(&hist[nt < a.hist_len ? nt : a.hist_len - 1], 1);
    }
    __syncthreads();
    for (int c = tid; c < a.hist_len; c += nthr) hist[c] *= c;
    __syncthreads();
    block_exclusive_scan(hist, a.hist_len, true, warp_sums);
    for (int b = tid; b < a.num_seqs; b += nthr) {
        const int nt = a.prefix[b + 1] - a.prefix[b];
        a.sbase[b] = atomicAdd(&hist[nt < a.hist_len ? nt : a.hist_len - 1], nt);
    }
    __syncthreads();
    // within a sample, tiles heaviest first (the forward's last query tiles see the most
    // key/value blocks, the backward's first key/value tiles see the most query blocks):
    // head by head for long samples, whose shared blocks would not stay in L2 otherwise;
    // rank by rank across all heads for short ones, whose blocks all fit in L2 and whose
    // heaviest tiles should start first
    for (int p = tid; p < ntiles; p += nthr) {
        const int b = find_sample(a.prefix, a.num_seqs, p);
        const int tile = p - a.prefix[b];
        const int nt = a.prefix[b + 1] - a.prefix[b];
        const int s = a.cu[b], e = a.cu[b + 1];
        const int cost = a.bwd ? bwd_item_cost(tile, s, e, a.causal, a.group) : fwd_item_cost(tile, s, e, a.causal, a.fwd_rows);
        const int rank = a.bwd ? tile : nt - 1 - tile;
        const bool head_major = e - s >= a.head_major_from;
        for (int h = 0; h < a.heads; ++h) {
            WorkItem w;
            w.head = h;
            w.seq = b;
            w.tile = tile;
            w.cost = cost;
            const int64_t pos = head_major ? (int64_t)h * nt + rank : (int64_t)rank * a.heads + h;
            a.items[(int64_t)a.sbase[b] * a.heads + pos] = w;
        }
    }
    if (tid == 0) {
        a.hdr->status = USP_OK;
        a.hdr->max_cost = 0;
        if (a.bwd) {
            a.hdr->bwd_count = ntiles * a.heads;
            a.hdr->bwd_next = 0;
        } else {
            a.hdr->fwd_count = ntiles * a.heads;
            a.hdr->fwd_next = 0;
        }
    }
}

__global__ void __launch_bounds__(1024) schedule_kernel(SchedArgs a) {
    // the attention kernel after this one may be launched now; it waits for this kernel to
    // complete before it reads the work list
    ptx::pdl_trigger();
    schedule_body(a);
    // launched after the backward's operand conversion, this kernel may have started before
    // that one finished: it completes only once the conversion has (which itself waited for
    // the stats kernel), so the attention kernel's wait covers all of them
    ptx::pdl_wait();
}

cudaError_t launch_schedule(const SchedArgs& a, cudaStream_t s, bool after_prep) {
    const size_t smem = a.hist_len <= kSchedSmemHist ? sizeof(int) * (size_t)a.hist_len : 0;
    return launch_kernel(schedule_kernel, dim3(1), dim3(1024), smem, s, after_prep, a);
}

}  // namespace usp
