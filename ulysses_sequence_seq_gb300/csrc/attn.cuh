// Launch interfaces of the attention kernels (attn_fwd.cu, attn_bwd.cu).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "common.cuh"

namespace usp {

struct FwdArgs {
    const int32_t* cu;
    const WorkItem* items;
    WsHeader* hdr;
    uint16_t* o;        // 16-bit [hq][T][D] (head-major) or [T][hq][D] (token_major)
    float* lse;         // [hq][T], natural log
    int64_t T;
    int hq;
    int group;          // hq / hkv
    int causal;
    int token_major;    // q, k, v, o in the seq-sharded [T][H][D] layout
    float scale_log2;   // softmax scale * log2(e)
    int f16;            // 16-bit inputs and outputs are fp16 (else bf16)
};

// o: the output map (make_activation_map over o) for whole-tile stores. grid: the work-item
// upper bound; min(grid, SM count) persistent CTAs are launched, as a programmatic
// dependent of the scheduler launched just before on s.
cudaError_t launch_attn_fwd(int head_dim, const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                            const CUtensorMap& o, const FwdArgs& a, int grid, cudaStream_t s);

struct BwdArgs {
    const int32_t* cu;
    const WorkItem* items;
    WsHeader* hdr;
    const float* lse;    // [hq][T]
    const float* delta;  // [hq][T]
    float* dq_acc;       // [hq][T][D] fp32 accumulator (atomic adds)
    void* dk;            // [hkv][T][D] (head-major) or [T][hkv][D] (token_major)
    void* dv;            // same layout as dk
    int grad_fp32;       // 1: dk/dv written as fp32, 0: in the input's 16-bit type
    int f16;             // 16-bit inputs and outputs are fp16 (else bf16)
    int64_t T;
    int hq;
    int hkv;
    int token_major;     // q, k, v, o, dO, dk, dv in the seq-sharded [T][H][D] layout
    int dq_token_major;  // dq_acc is the caller's fp32 dq in the [T][hq][D] layout
    int group;
    int causal;
    float scale;         // softmax scale
    float scale_log2;    // softmax scale * log2(e)
};

// dk, dv: 16-bit gradient maps (make_activation_map) for whole-tile stores; not read for
// fp32 gradients. grid: as for launch_attn_fwd.
cudaError_t launch_attn_bwd(int head_dim, const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                            const CUtensorMap& dout, const CUtensorMap& dq, const CUtensorMap& dk, const CUtensorMap& dv,
                            const BwdArgs& a, int grid, cudaStream_t s);

// Delta_i = dO_i . O_i (fp32, [hq][T]) for every query row, and zeroes the dQ accumulator.
// o / dout are head-major or token-major (token_major); the accumulator is head-major
// unless dq_token_major.
// o / dout are bf16, or fp16 when f16.
cudaError_t launch_bwd_prep(const void* o, const void* dout, float* delta, float* dq_acc, int64_t T, int hq,
                            int head_dim, int token_major, int dq_token_major, int f16, cudaStream_t s);

// dq (16-bit, head-major or token-major) = the head-major fp32 accumulator rounded to bf16,
// or to fp16 when f16. Launched as a programmatic dependent of the backward kernel.
cudaError_t launch_dq_convert(const float* dq_acc, void* dq, int64_t T, int hq, int head_dim, int token_major,
                              int f16, cudaStream_t s);

// TMA tensor map over a 16-bit activation (bf16 or fp16: the copy moves bytes), head-major [heads][T][D] or token-major
// [T][heads][D]: boxes of 64 columns x 128 rows of one head, 128-byte swizzle.
bool make_activation_map(CUtensorMap* map, const void* base, int64_t T, int heads, int D, int token_major);
// fp32 dQ accumulator ([heads][T][D] or [T][heads][D]) in 32-column x 32-row boxes with the
// 128-byte swizzle, the target of the backward's bulk tensor reductions.
bool make_dq_accum_map(CUtensorMap* map, float* base, int64_t T, int heads, int D, int token_major);

// Records `code` in the status word after a kernel that waits on an mbarrier nothing arrives on.
cudaError_t launch_debug_timeout(WsHeader* hdr, uint64_t limit_ns, cudaStream_t s);

}  // namespace usp
