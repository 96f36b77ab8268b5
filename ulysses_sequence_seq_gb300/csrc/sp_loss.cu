// Bookkeeping around the attention of Ulysses sequence parallelism, on the device so
// that a training step needs no host round trip between the data and the attention:
//
//   * sample boundaries (cu_seqlens) from packed position_ids, and back;
//   * the label shift inside packed samples, with each SP rank's count of tokens whose
//     shifted label is not -100 ("good tokens");
//   * the loss over the SP ranks as the good-token weighted mean of the ranks' losses,
//     leaving out ranks without good tokens.
//
// HF Transformers "Ulysses sequence parallelism" guide (section on the Accelerate
// configuration file: position_ids, label shift and loss aggregation over SP ranks);
// jianying88 article on DeepSpeed Ulysses in Transformers, section
// "3. 跨 rank 的加权 loss 聚合" (the weighted aggregation and the good-token count).
//
// All of it is HBM-bound and tiny next to the attention (8-16 bytes per token).
#include <cuda_runtime.h>

#include <cstdint>

#include "common.cuh"
#include "usp.h"

namespace usp {
namespace {

constexpr int kThreads = 256;
constexpr int kPerThread = 8;
constexpr int kChunk = kThreads * kPerThread;  // position ids per CTA
constexpr int64_t kIgnore = -100;

// Workspace of usp_position_ids_to_cu_seqlens: the status word (read by
// usp_get_device_status), the sample count, then one count per CTA chunk.
struct PosHeader {
    int status;
    int num_seqs;
    int overflow;  // more samples than max_seqs
};
constexpr size_t kPosCountsOffset = 256;

__device__ __forceinline__ int warp_incl_scan(int x) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, off);
        if (lane >= off) x += y;
    }
    return x;
}

// Exclusive scan of one int per thread over the CTA; returns the CTA total in *total.
template <int NT>
__device__ __forceinline__ int block_excl_scan(int x, int* warp_sums, int* total) {
    constexpr int kWarps = NT / 32;
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    const int incl = warp_incl_scan(x);
    if (lane == 31) warp_sums[wid] = incl;
    __syncthreads();
    if (wid == 0) {
        const int w = lane < kWarps ? warp_sums[lane] : 0;
        const int wi = warp_incl_scan(w);
        if (lane < kWarps) warp_sums[lane] = wi;
    }
    __syncthreads();
    const int base = wid > 0 ? warp_sums[wid - 1] : 0;
    *total = warp_sums[kWarps - 1];
    __syncthreads();  // warp_sums may be reused by the caller
    return base + incl - x;
}

// A token starts a sample where its position id is 0; anywhere else the id must be the
// previous token's id + 1. Counts the starts of each chunk and flags malformed ids.
__global__ void __launch_bounds__(kThreads) pos_count_kernel(const int64_t* __restrict__ pos, int64_t T,
                                                             int* __restrict__ counts, PosHeader* hdr) {
    __shared__ int warp_sums[kThreads / 32];
    const int64_t base = (int64_t)blockIdx.x * kChunk;
    int starts = 0;
    bool bad = false;
#pragma unroll
    for (int j = 0; j < kPerThread; ++j) {
        const int64_t t = base + j * kThreads + threadIdx.x;
        if (t < T) {
            const int64_t p = pos[t];
            if (p == 0) ++starts;
            else if (t == 0 || p != pos[t - 1] + 1) bad = true;
        }
    }
    if (bad) hdr->status = USP_ERR_DEVICE_CHECK;
    int total;
    block_excl_scan<kThreads>(starts, warp_sums, &total);
    if (threadIdx.x == 0) counts[blockIdx.x] = total;
}

// Exclusive prefix sum of the chunk counts (one CTA, running carry over 1024-wide
// passes); the grand total is the number of samples.
__global__ void __launch_bounds__(1024) pos_scan_kernel(int* __restrict__ counts, int nblocks, int max_seqs,
                                                        PosHeader* hdr) {
    __shared__ int warp_sums[32];
    int carry = 0;
    for (int i0 = 0; i0 < nblocks; i0 += 1024) {
        const int i = i0 + threadIdx.x;
        const int x = i < nblocks ? counts[i] : 0;
        int total;
        const int ex = block_excl_scan<1024>(x, warp_sums, &total);
        if (i < nblocks) counts[i] = carry + ex;
        carry += total;
    }
    if (threadIdx.x == 0) {
        hdr->num_seqs = carry;
        if (carry > max_seqs && hdr->status == 0) {
            hdr->status = USP_ERR_DEVICE_CHECK;
            hdr->overflow = 1;
        }
    }
}

// Writes the start of sample b to cu[b] (chunk offset + rank of the start in its chunk),
// pads cu[n..max_seqs] with T, and reports n. Nothing is written to cu when the ids were
// malformed or the samples do not fit (n is still reported in the second case).
__global__ void __launch_bounds__(kThreads) pos_scatter_kernel(const int64_t* __restrict__ pos, int64_t T,
                                                               const int* __restrict__ offsets,
                                                               int32_t* __restrict__ cu, int max_seqs,
                                                               int32_t* num_seqs_out, const PosHeader* hdr) {
    __shared__ int warp_sums[kThreads / 32];
    const int status = hdr->status;
    const int n = hdr->num_seqs;
    // the count is reported when the ids are well formed, even if it exceeds max_seqs
    if (blockIdx.x == 0 && threadIdx.x == 0 && num_seqs_out && (status == 0 || hdr->overflow))
        *num_seqs_out = n;
    if (status != 0) return;
    const int64_t base = (int64_t)blockIdx.x * kChunk;
    int rank = offsets[blockIdx.x];
    // starts in chunk order: each pass of kThreads tokens is scanned, ranks continue
#pragma unroll 1
    for (int j = 0; j < kPerThread; ++j) {
        const int64_t t = base + j * kThreads + threadIdx.x;
        const int is_start = (t < T && pos[t] == 0) ? 1 : 0;
        int total;
        const int ex = block_excl_scan<kThreads>(is_start, warp_sums, &total);
        if (is_start) cu[rank + ex] = (int32_t)t;
        rank += total;
    }
    // padding: cu[n..max_seqs] = T (empty samples), by all threads of the grid
    const int64_t stride = (int64_t)gridDim.x * kThreads;
    for (int64_t i = (int64_t)blockIdx.x * kThreads + threadIdx.x + n; i <= max_seqs; i += stride)
        cu[i] = (int32_t)T;
}

// Largest b in [0, num_seqs) with cu[b] <= t: the sample holding token t (empty samples,
// whose cu[b] == cu[b+1], are passed over).
__device__ __forceinline__ int sample_of(const int32_t* __restrict__ cu, int num_seqs, int64_t t) {
    int lo = 0, hi = num_seqs - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if ((int64_t)__ldg(cu + mid) <= t) lo = mid;
        else hi = mid - 1;
    }
    return lo;
}

__global__ void __launch_bounds__(kThreads) cu_to_pos_kernel(const int32_t* __restrict__ cu, int num_seqs, int64_t T,
                                                             int64_t* __restrict__ pos) {
    const int64_t stride = (int64_t)gridDim.x * kThreads;
    for (int64_t t = (int64_t)blockIdx.x * kThreads + threadIdx.x; t < T; t += stride)
        pos[t] = t - __ldg(cu + sample_of(cu, num_seqs, t));
}

// shift[t] = labels[t+1] inside a sample, -100 on a sample's last token; good[r] counts
// the tokens of rank r's shard (S = T/sp tokens) whose shifted label is not -100.
__global__ void __launch_bounds__(kThreads) shift_labels_kernel(const int64_t* __restrict__ labels,
                                                                const int32_t* __restrict__ cu, int num_seqs,
                                                                int64_t T, int64_t S,
                                                                int64_t* __restrict__ shift,
                                                                unsigned long long* __restrict__ good) {
    const int64_t stride = (int64_t)gridDim.x * kThreads;
    const int64_t t_end = (T + kThreads - 1) / kThreads * kThreads;  // whole warps stay in the loop
    for (int64_t t = (int64_t)blockIdx.x * kThreads + threadIdx.x; t < t_end; t += stride) {
        int is_good = 0;
        int rank = -1;
        if (t < T) {
            const int b = sample_of(cu, num_seqs, t);
            const int64_t end = __ldg(cu + b + 1);
            const int64_t v = (t + 1 < end && t + 1 < T) ? labels[t + 1] : kIgnore;
            shift[t] = v;
            is_good = v != kIgnore;
            rank = (int)(t / S);
        }
        // one atomic per rank present in the warp
        const unsigned peers = __match_any_sync(0xffffffffu, rank);
        const int n = __popc(__ballot_sync(0xffffffffu, is_good) & peers);
        const int leader = __ffs(peers) - 1;
        if (rank >= 0 && (int)(threadIdx.x & 31) == leader && n) atomicAdd(good + rank, (unsigned long long)n);
    }
}

// loss = sum_{r: good_r > 0} loss_r * good_r / sum_r good_r  (0 when no rank has a good
// token), accumulated in float64 by one warp.
__global__ void __launch_bounds__(32) weighted_loss_kernel(const float* __restrict__ rank_loss,
                                                           const int64_t* __restrict__ good, int sp,
                                                           float* __restrict__ out) {
    double num = 0.0, den = 0.0;
    for (int r = threadIdx.x; r < sp; r += 32) {
        const int64_t g = good[r];
        if (g > 0) {
            num += (double)rank_loss[r] * (double)g;
            den += (double)g;
        }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        num += __shfl_xor_sync(0xffffffffu, num, off);
        den += __shfl_xor_sync(0xffffffffu, den, off);
    }
    if (threadIdx.x == 0) *out = den > 0.0 ? (float)(num / den) : 0.0f;
}

bool aligned(const void* p, uintptr_t a) { return ((uintptr_t)p & (a - 1)) == 0; }

int grid_1d(int64_t n) {
    const int64_t want = (n + kThreads - 1) / kThreads;
    const int sms = device_sm_count();
    const int64_t cap = (int64_t)(sms > 0 ? sms : 148) * 8;  // 8 CTAs of 256 threads per SM; grid-stride beyond
    return (int)(want < 1 ? 1 : (want < cap ? want : cap));
}

}  // namespace
}  // namespace usp

using namespace usp;

extern "C" size_t usp_position_ids_workspace_size(int64_t total_tokens) {
    if (total_tokens < 0) return 0;
    const int64_t blocks = (total_tokens + kChunk - 1) / kChunk;
    return kPosCountsOffset + (size_t)blocks * sizeof(int);
}

extern "C" usp_status usp_position_ids_to_cu_seqlens(const int64_t* position_ids, int64_t total_tokens,
                                                     int32_t* cu_seqlens, int max_seqs, int32_t* num_seqs,
                                                     void* workspace, size_t workspace_bytes, void* stream) {
    if (total_tokens < 0 || total_tokens > INT32_MAX || max_seqs < 1) return USP_ERR_INVALID_ARG;
    if (!cu_seqlens || !workspace || !aligned(cu_seqlens, 4) || !aligned(workspace, 16)) return USP_ERR_INVALID_ARG;
    if (num_seqs && !aligned(num_seqs, 4)) return USP_ERR_INVALID_ARG;
    if (workspace_bytes < usp_position_ids_workspace_size(total_tokens)) return USP_ERR_WORKSPACE;
    cudaStream_t s = (cudaStream_t)stream;
    PosHeader* hdr = (PosHeader*)workspace;
    if (cudaMemsetAsync(hdr, 0, sizeof(PosHeader), s) != cudaSuccess) return USP_ERR_CUDA;
    if (total_tokens == 0) {  // no samples: cu = {0, 0, ...}
        if (cudaMemsetAsync(cu_seqlens, 0, sizeof(int32_t) * ((size_t)max_seqs + 1), s) != cudaSuccess)
            return USP_ERR_CUDA;
        if (num_seqs && cudaMemsetAsync(num_seqs, 0, sizeof(int32_t), s) != cudaSuccess) return USP_ERR_CUDA;
        return USP_OK;
    }
    if (!position_ids || !aligned(position_ids, 8)) return USP_ERR_INVALID_ARG;
    const int blocks = (int)((total_tokens + kChunk - 1) / kChunk);
    int* counts = (int*)((uint8_t*)workspace + kPosCountsOffset);
    pos_count_kernel<<<blocks, kThreads, 0, s>>>(position_ids, total_tokens, counts, hdr);
    pos_scan_kernel<<<1, 1024, 0, s>>>(counts, blocks, max_seqs, hdr);
    pos_scatter_kernel<<<blocks, kThreads, 0, s>>>(position_ids, total_tokens, counts, cu_seqlens, max_seqs,
                                                   num_seqs, hdr);
    return cudaGetLastError() == cudaSuccess ? USP_OK : USP_ERR_CUDA;
}

extern "C" usp_status usp_cu_seqlens_to_position_ids(const int32_t* cu_seqlens, int num_seqs, int64_t total_tokens,
                                                     int64_t* position_ids, void* stream) {
    if (total_tokens < 0 || total_tokens > INT32_MAX) return USP_ERR_INVALID_ARG;
    if (total_tokens == 0) return USP_OK;
    if (num_seqs < 1 || !cu_seqlens || !position_ids || !aligned(cu_seqlens, 4) || !aligned(position_ids, 8))
        return USP_ERR_INVALID_ARG;
    cudaStream_t s = (cudaStream_t)stream;
    cu_to_pos_kernel<<<grid_1d(total_tokens), kThreads, 0, s>>>(cu_seqlens, num_seqs, total_tokens, position_ids);
    return cudaGetLastError() == cudaSuccess ? USP_OK : USP_ERR_CUDA;
}

extern "C" usp_status usp_shift_labels(const int64_t* labels, const int32_t* cu_seqlens, int num_seqs,
                                       int64_t total_tokens, int sp, int64_t* shift_labels, int64_t* good_tokens,
                                       void* stream) {
    if (total_tokens < 0 || total_tokens > INT32_MAX || sp < 1 || total_tokens % sp) return USP_ERR_INVALID_ARG;
    if (!good_tokens || !aligned(good_tokens, 8)) return USP_ERR_INVALID_ARG;
    cudaStream_t s = (cudaStream_t)stream;
    if (cudaMemsetAsync(good_tokens, 0, sizeof(int64_t) * (size_t)sp, s) != cudaSuccess) return USP_ERR_CUDA;
    if (total_tokens == 0) return USP_OK;
    if (num_seqs < 1 || !labels || !cu_seqlens || !shift_labels || !aligned(labels, 8) || !aligned(cu_seqlens, 4) ||
        !aligned(shift_labels, 8))
        return USP_ERR_INVALID_ARG;
    const int64_t lo = (int64_t)(uintptr_t)labels, hi = lo + 8 * total_tokens;
    const int64_t so = (int64_t)(uintptr_t)shift_labels;
    if (so < hi && lo < so + 8 * total_tokens) return USP_ERR_INVALID_ARG;  // in place would race
    shift_labels_kernel<<<grid_1d(total_tokens), kThreads, 0, s>>>(labels, cu_seqlens, num_seqs, total_tokens,
                                                                   total_tokens / sp, shift_labels,
                                                                   (unsigned long long*)good_tokens);
    return cudaGetLastError() == cudaSuccess ? USP_OK : USP_ERR_CUDA;
}

extern "C" usp_status usp_sp_weighted_loss(const float* rank_loss, const int64_t* good_tokens, int sp, float* loss,
                                           void* stream) {
    if (sp < 1 || !rank_loss || !good_tokens || !loss) return USP_ERR_INVALID_ARG;
    if (!aligned(rank_loss, 4) || !aligned(good_tokens, 8) || !aligned(loss, 4)) return USP_ERR_INVALID_ARG;
    weighted_loss_kernel<<<1, 32, 0, (cudaStream_t)stream>>>(rank_loss, good_tokens, sp, loss);
    return cudaGetLastError() == cudaSuccess ? USP_OK : USP_ERR_CUDA;
}
