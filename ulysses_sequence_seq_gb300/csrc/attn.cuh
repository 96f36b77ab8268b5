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
    uint16_t* o_res;    // NULL, or the rounding residual of o in the same type and layout:
                        // o_res = round16(O - o) for the fp32 result O, so o + o_res ~ O
    float* lse;         // [hq][T], natural log
    int64_t T;
    int hq;
    int group;          // hq / hkv
    int causal;
    int token_major;    // q, k, v, o in the seq-sharded [T][H][D] layout
    float scale_log2;   // softmax scale * log2(e)
    int f16;            // 16-bit inputs and outputs are fp16 (else bf16)
};

// o, o_res: the output maps (make_activation_map over o and o_res; o_res is not read when
// a.o_res is NULL) for whole-tile stores; k: boxes of fwd_k_box_rows(head_dim) rows.
// grid: the work-item upper bound; persistent CTAs (one per SM; pairs of them for head_dim
// 128, as many as can be resident) are launched, as a programmatic dependent of the
// scheduler launched just before on s.
cudaError_t launch_attn_fwd(int head_dim, const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                            const CUtensorMap& o, const CUtensorMap& o_res, const FwdArgs& a, int grid,
                            cudaStream_t s);

// The backward runs its tensor-core products on fp16 copies of q, k, v and dO, each scaled
// by a power of two per key/value group so that its largest magnitude lies in [8, 16):
// P and dS are then rounded to fp16 (11 significant bits) instead of bf16 (8), which the
// tolerance on short samples needs, and the scaling keeps small gradients (dO of a real
// loss) and large activations inside fp16's range. The exponent of a group follows from
// the largest magnitude alone (range_exponent), so every kernel derives it the same way.
enum { kAmaxQ = 0, kAmaxK = 1, kAmaxV = 2, kAmaxDO = 3 };

// e such that amax * 2^e lies in [8, 16); 0 for zero, subnormal or non-finite amax; clamped
// to [-24, 24] so that every product of the scales below stays a normal float.
__host__ __device__ __forceinline__ int range_exponent(uint32_t amax_bits) {
    const int E = (int)((amax_bits >> 23) & 0xffu);
    if (E == 0 || E == 255) return 0;
    int e = 130 - E;
    return e < -24 ? -24 : (e > 24 ? 24 : e);
}
__host__ __device__ __forceinline__ float exp2i(int e) {   // 2^e for e in [-126, 127]
#ifdef __CUDA_ARCH__
    return __int_as_float((e + 127) << 23);
#else
    union { uint32_t u; float f; } c;
    c.u = (uint32_t)(e + 127) << 23;
    return c.f;
#endif
}
// Exponent applied to dS before its fp16 rounding: |dS| is at most 2 D 16^2 scale on the
// scaled operands, and 2^ds_exp brings that bound to at most 2^15.
int ds_exponent(int head_dim, float scale);

struct BwdArgs {
    const int32_t* cu;
    const WorkItem* items;
    WsHeader* hdr;
    const float* lse;       // [hq][T]
    const float* delta;     // [hq][T], Delta_i = dO_i . O_i unscaled
    const uint32_t* amax;   // [4][hkv] float bits: largest |q|, |k|, |v|, |dO| of each key/value group
    float* dq_acc;          // [hq][T][D] fp32 accumulator of dQ' (bulk reductions), head-major
    void* dk;               // [hkv][T][D] (head-major) or [T][hkv][D] (token_major)
    void* dv;               // same layout as dk
    int grad_fp32;          // 1: dk/dv written as fp32, 0: 16-bit (out_f16 picks the type)
    int out_f16;            // 16-bit gradients are fp16 (else bf16)
    int64_t T;
    int hq;
    int hkv;
    int token_major;        // dk, dv in the seq-sharded [T][H][D] layout (the operands are head-major copies)
    int group;
    int causal;
    float scale;            // softmax scale
    float scale_log2;       // softmax scale * log2(e)
    int ds_exp;             // ds_exponent(D, scale)
};

// q, k, v, dout: maps over the scaled fp16 copies (head-major). dk, dv: 16-bit gradient
// maps (make_activation_map) for whole-tile stores; not read for fp32 gradients. grid: as
// for launch_attn_fwd.
cudaError_t launch_attn_bwd(int head_dim, const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                            const CUtensorMap& dout, const CUtensorMap& dq, const CUtensorMap& dk, const CUtensorMap& dv,
                            const BwdArgs& a, int grid, cudaStream_t s);

// First kernel of a backward call: Delta_i = dO_i . (O_i + O_res_i) in fp32 ([hq][T]) for
// every query row, zeroes the dQ accumulator, and the largest magnitude of q, k, v and dO of
// every key/value group into amax ([4][hkv] float bits, zeroed before the launch).
// Activations are 16-bit (fp16 when f16, else bf16), head-major or token-major; o_res may
// be NULL. The accumulator is head-major.
struct BwdStatsArgs {
    const uint16_t *q, *k, *v, *o, *o_res, *dout;
    float* delta;
    float* dq_acc;
    uint32_t* amax;
    int64_t T;
    int hq, hkv, group, token_major, f16;
};
cudaError_t launch_bwd_stats(int head_dim, const BwdStatsArgs& a, cudaStream_t s);

// Second kernel: q, k, v, dO as fp16 copies scaled by 2^range_exponent(amax of the group),
// written head-major into the workspace. Launched as a programmatic dependent of the stats.
struct BwdConvertArgs {
    const uint16_t* src[4];   // q, k, v, dO in the call's layout and type
    uint16_t* dst[4];         // head-major fp16 copies
    const uint32_t* amax;     // [4][hkv]
    int64_t T;
    int hq, hkv, group, token_major, f16;
};
cudaError_t launch_bwd_convert(int head_dim, const BwdConvertArgs& a, cudaStream_t s);

// dq (out_dt: USP_BF16, USP_FP16 or USP_FP32; head-major or token-major) = the head-major
// fp32 accumulator of scaled dQ' times its group's 2^-(ev+edo+ds_exp+ek). Launched as a
// programmatic dependent of the backward kernel.
cudaError_t launch_dq_convert(const float* dq_acc, void* dq, const uint32_t* amax, int64_t T, int hq, int hkv,
                              int head_dim, int token_major, int out_dt, int ds_exp, cudaStream_t s);

// TMA tensor map over a 16-bit activation (bf16 or fp16: the copy moves bytes), head-major [heads][T][D] or token-major
// [T][heads][D]: boxes of 64 columns x box_rows rows of one head, 128-byte swizzle.
bool make_activation_map(CUtensorMap* map, const void* base, int64_t T, int heads, int D, int token_major,
                         int box_rows = kTileM);
// Rows of the forward's K boxes: a CTA pair (head_dim 128) loads half of each key block per CTA.
inline int fwd_k_box_rows(int head_dim) { return head_dim == 128 ? kBlockN / 2 : kBlockN; }
// fp32 dQ accumulator ([heads][T][D] or [T][heads][D]) in 32-column x 32-row boxes with the
// 128-byte swizzle, the target of the backward's bulk tensor reductions.
bool make_dq_accum_map(CUtensorMap* map, float* base, int64_t T, int heads, int D, int token_major);

// Records `code` in the status word after a kernel that waits on an mbarrier nothing arrives on.
cudaError_t launch_debug_timeout(WsHeader* hdr, uint64_t limit_ns, cudaStream_t s);

}  // namespace usp
