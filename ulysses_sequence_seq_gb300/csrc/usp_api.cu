// C ABI of the attention calls: argument validation, workspace carving, TMA tensor
// maps and the launch sequence (scheduler -> attention kernels).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <climits>
#include <cmath>
#include <cstdint>
#include <mutex>

#include "attn.cuh"
#include "common.cuh"
#include "sched.cuh"

namespace usp {
namespace {

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = (EncodeTiledFn)p;
    });
    return fn;
}

bool aligned16(const void* p) { return ((uintptr_t)p & 15) == 0; }

// T == 0: nothing to compute and the data pointers may be NULL (empty tensors); the
// status word of a workspace, if one is given, is reset to USP_OK.
usp_status reset_status_if_any(void* workspace, size_t ws_bytes, cudaStream_t s) {
    if (!workspace || ws_bytes < sizeof(WsHeader)) return USP_OK;
    if (!aligned16(workspace)) return USP_ERR_INVALID_ARG;
    return cudaMemsetAsync(workspace, 0, sizeof(WsHeader), s) == cudaSuccess ? USP_OK : USP_ERR_CUDA;
}

}  // namespace

// Tensor map over a bf16 activation, 64-column x box_rows-row boxes of one head, 128-byte
// swizzled (the layout the tensor-core descriptors expect). Head-major [heads][T][D] maps
// are (D, T, heads); token-major [T][heads][D] maps are (D, heads, T), so the strides grow.
bool make_activation_map(CUtensorMap* map, const void* base, int64_t T, int heads, int D, int token_major,
                         int box_rows) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    const cuuint64_t row = (cuuint64_t)D * 2;
    cuuint64_t dims[3], strides[2];
    cuuint32_t box[3];
    if (token_major) {
        dims[0] = (cuuint64_t)D; dims[1] = (cuuint64_t)heads; dims[2] = (cuuint64_t)T;
        strides[0] = row; strides[1] = row * (cuuint64_t)heads;
        box[0] = 64; box[1] = 1; box[2] = (cuuint32_t)box_rows;
    } else {
        dims[0] = (cuuint64_t)D; dims[1] = (cuuint64_t)T; dims[2] = (cuuint64_t)heads;
        strides[0] = row; strides[1] = row * (cuuint64_t)T;
        box[0] = 64; box[1] = (cuuint32_t)box_rows; box[2] = 1;
    }
    cuuint32_t es[3] = {1, 1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_dq_accum_map(CUtensorMap* map, float* base, int64_t T, int heads, int D, int token_major) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    const cuuint64_t row = (cuuint64_t)D * 4;
    cuuint64_t dims[3], strides[2];
    cuuint32_t box[3];
    if (token_major) {
        dims[0] = (cuuint64_t)D; dims[1] = (cuuint64_t)heads; dims[2] = (cuuint64_t)T;
        strides[0] = row; strides[1] = row * (cuuint64_t)heads;
        box[0] = 32; box[1] = 1; box[2] = 32;
    } else {
        dims[0] = (cuuint64_t)D; dims[1] = (cuuint64_t)T; dims[2] = (cuuint64_t)heads;
        strides[0] = row; strides[1] = row * (cuuint64_t)T;
        box[0] = 32; box[1] = 32; box[2] = 1;
    }
    cuuint32_t es[3] = {1, 1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, base, dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace usp

using namespace usp;

extern "C" size_t usp_attn_workspace_size(int64_t total_tokens, int num_seqs, int hq, int hkv, int head_dim,
                                          int bwd) {
    if (total_tokens < 0 || num_seqs < 0 || hq < 1 || hkv < 1 || head_dim < 1) return 0;
    return ws_layout(total_tokens, num_seqs, hq, hkv, head_dim, bwd ? 1 : 0).total;
}

namespace usp {
namespace {

usp_status attn_fwd_impl(const void* q, const void* k, const void* v, void* o, void* o_res, float* lse,
                         const int32_t* cu_seqlens,
                         int num_seqs, int64_t total_tokens, int hq, int hkv, int head_dim, float softmax_scale,
                         int causal, void* workspace, size_t ws_bytes, cudaStream_t s, int token_major,
                         usp_dtype dt = USP_BF16) {
    usp_status st = check_attn_sizes(total_tokens, num_seqs, hq, hkv, head_dim, cu_seqlens);
    if (st != USP_OK) return st;
    if (dt != USP_BF16 && dt != USP_FP16) return dt == USP_FP32 ? USP_ERR_UNSUPPORTED : USP_ERR_INVALID_ARG;
    if (total_tokens == 0) return reset_status_if_any(workspace, ws_bytes, s);
    if (!q || !k || !v || !o || !lse || !workspace) return USP_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse) || !aligned16(workspace) ||
        !aligned16(o_res))
        return USP_ERR_INVALID_ARG;
    const WsLayout w = ws_layout(total_tokens, num_seqs, hq, hkv, head_dim, 0);
    if (ws_bytes < w.total) return USP_ERR_WORKSPACE;
    uint8_t* ws = (uint8_t*)workspace;
    WsHeader* hdr = (WsHeader*)ws;   // written by the scheduler: status, item count, item counter

    SchedArgs sa{};
    sa.cu = cu_seqlens;
    sa.num_seqs = num_seqs;
    sa.T = total_tokens;
    sa.heads = hq;
    sa.bwd = 0;
    sa.fwd_rows = fwd_rows_per_item(head_dim);
    sa.causal = causal ? 1 : 0;
    sa.group = hq / hkv;
    sa.hist_len = w.hist_len;
    sa.max_items = w.max_items;
    sa.hdr = hdr;
    sa.hist = (int*)(ws + w.hist);
    sa.prefix = (int*)(ws + w.prefix);
    sa.sbase = (int*)(ws + w.sbase);
    sa.head_major_from = head_major_from_tokens(hkv, head_dim, sa.bwd);
    sa.items = (WorkItem*)(ws + w.items);
    if (launch_schedule(sa, s, false) != cudaSuccess) return USP_ERR_CUDA;

    CUtensorMap mq, mk, mv, mo, mores;
    if (!make_activation_map(&mq, q, total_tokens, hq, head_dim, token_major) ||
        !make_activation_map(&mk, k, total_tokens, hkv, head_dim, token_major, fwd_k_box_rows(head_dim)) ||
        !make_activation_map(&mv, v, total_tokens, hkv, head_dim, token_major) ||
        !make_activation_map(&mo, o, total_tokens, hq, head_dim, token_major) ||
        !make_activation_map(&mores, o_res ? o_res : o, total_tokens, hq, head_dim, token_major))
        return USP_ERR_CUDA;
    FwdArgs fa{};
    fa.cu = cu_seqlens;
    fa.items = sa.items;
    fa.hdr = hdr;
    fa.o = (uint16_t*)o;
    fa.o_res = (uint16_t*)o_res;
    fa.f16 = dt == USP_FP16 ? 1 : 0;
    fa.lse = lse;
    fa.T = total_tokens;
    fa.hq = hq;
    fa.group = hq / hkv;
    fa.causal = sa.causal;
    fa.token_major = token_major;
    fa.scale_log2 = resolve_softmax_scale(softmax_scale, head_dim) * 1.4426950408889634f;
    if (launch_attn_fwd(head_dim, mq, mk, mv, mo, mores, fa, w.max_items, s) != cudaSuccess) return USP_ERR_CUDA;
    return USP_OK;
}

usp_status attn_bwd_impl(const void* q, const void* k, const void* v, const void* o, const void* o_res,
                         const float* lse, const void* d_o, void* dq, void* dk, void* dv, usp_dtype grad_dt,
                         const int32_t* cu_seqlens, int num_seqs, int64_t total_tokens, int hq, int hkv, int head_dim,
                         float softmax_scale, int causal, void* workspace, size_t ws_bytes, cudaStream_t s,
                         int token_major, usp_dtype dt = USP_BF16) {
    usp_status st = check_attn_sizes(total_tokens, num_seqs, hq, hkv, head_dim, cu_seqlens);
    if (st != USP_OK) return st;
    if (dt != USP_BF16 && dt != USP_FP16) return dt == USP_FP32 ? USP_ERR_UNSUPPORTED : USP_ERR_INVALID_ARG;
    // gradients in the inputs' 16-bit type or in fp32
    if (grad_dt != dt && grad_dt != USP_FP32)
        return (grad_dt == USP_BF16 || grad_dt == USP_FP16) ? USP_ERR_UNSUPPORTED : USP_ERR_INVALID_ARG;
    if (total_tokens == 0) return reset_status_if_any(workspace, ws_bytes, s);
    if (!q || !k || !v || !o || !lse || !d_o || !dq || !dk || !dv || !workspace) return USP_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse) || !aligned16(d_o) ||
        !aligned16(dq) || !aligned16(dk) || !aligned16(dv) || !aligned16(workspace) || !aligned16(o_res))
        return USP_ERR_INVALID_ARG;
    const WsLayout w = ws_layout(total_tokens, num_seqs, hq, hkv, head_dim, 1);
    if (ws_bytes < w.total) return USP_ERR_WORKSPACE;
    uint8_t* ws = (uint8_t*)workspace;
    WsHeader* hdr = (WsHeader*)ws;   // written by the scheduler: status, item count, item counter
    const bool fp32_grads = grad_dt == USP_FP32;
    float* delta = (float*)(ws + w.delta);
    // dQ' accumulates in the head-major workspace accumulator; a final pass scales it back
    // and writes dq in grad_dt and the caller's layout
    float* dq_acc = (float*)(ws + w.dq_acc);
    const int f16 = dt == USP_FP16 ? 1 : 0;
    uint32_t* amax = (uint32_t*)(ws + w.amax);
    uint16_t* q16 = (uint16_t*)(ws + w.q16);
    uint16_t* k16 = (uint16_t*)(ws + w.k16);
    uint16_t* v16 = (uint16_t*)(ws + w.v16);
    uint16_t* do16 = (uint16_t*)(ws + w.do16);

    // Delta, the zeroed dQ accumulator and the per-group magnitudes; then the scaled fp16
    // operand copies; the scheduler runs alongside them
    if (cudaMemsetAsync(amax, 0, sizeof(uint32_t) * 4 * (size_t)hkv, s) != cudaSuccess) return USP_ERR_CUDA;
    BwdStatsArgs sta{};
    sta.q = (const uint16_t*)q;
    sta.k = (const uint16_t*)k;
    sta.v = (const uint16_t*)v;
    sta.o = (const uint16_t*)o;
    sta.o_res = (const uint16_t*)o_res;
    sta.dout = (const uint16_t*)d_o;
    sta.delta = delta;
    sta.dq_acc = dq_acc;
    sta.amax = amax;
    sta.T = total_tokens;
    sta.hq = hq;
    sta.hkv = hkv;
    sta.group = hq / hkv;
    sta.token_major = token_major;
    sta.f16 = f16;
    if (launch_bwd_stats(head_dim, sta, s) != cudaSuccess) return USP_ERR_CUDA;
    BwdConvertArgs cva{};
    cva.src[kAmaxQ] = (const uint16_t*)q;
    cva.src[kAmaxK] = (const uint16_t*)k;
    cva.src[kAmaxV] = (const uint16_t*)v;
    cva.src[kAmaxDO] = (const uint16_t*)d_o;
    cva.dst[kAmaxQ] = q16;
    cva.dst[kAmaxK] = k16;
    cva.dst[kAmaxV] = v16;
    cva.dst[kAmaxDO] = do16;
    cva.amax = amax;
    cva.T = total_tokens;
    cva.hq = hq;
    cva.hkv = hkv;
    cva.group = hq / hkv;
    cva.token_major = token_major;
    cva.f16 = f16;
    if (launch_bwd_convert(head_dim, cva, s) != cudaSuccess) return USP_ERR_CUDA;

    SchedArgs sa{};
    sa.cu = cu_seqlens;
    sa.num_seqs = num_seqs;
    sa.T = total_tokens;
    sa.heads = hkv;
    sa.bwd = 1;
    sa.causal = causal ? 1 : 0;
    sa.group = hq / hkv;
    sa.hist_len = w.hist_len;
    sa.max_items = w.max_items;
    sa.hdr = hdr;
    sa.hist = (int*)(ws + w.hist);
    sa.prefix = (int*)(ws + w.prefix);
    sa.sbase = (int*)(ws + w.sbase);
    sa.head_major_from = head_major_from_tokens(hkv, head_dim, sa.bwd);
    sa.items = (WorkItem*)(ws + w.items);
    if (launch_schedule(sa, s, true) != cudaSuccess) return USP_ERR_CUDA;

    CUtensorMap mq, mk, mv, mdo, mdq, mdk, mdv;
    if (!make_activation_map(&mq, q16, total_tokens, hq, head_dim, 0) ||
        !make_activation_map(&mk, k16, total_tokens, hkv, head_dim, 0) ||
        !make_activation_map(&mv, v16, total_tokens, hkv, head_dim, 0) ||
        !make_activation_map(&mdo, do16, total_tokens, hq, head_dim, 0) ||
        !make_dq_accum_map(&mdq, dq_acc, total_tokens, hq, head_dim, 0))
        return USP_ERR_CUDA;
    // 16-bit dK/dV leave as whole tiles through these maps; fp32 gradients are stored by rows
    if (fp32_grads) {
        mdk = mk;
        mdv = mv;
    } else if (!make_activation_map(&mdk, dk, total_tokens, hkv, head_dim, token_major) ||
               !make_activation_map(&mdv, dv, total_tokens, hkv, head_dim, token_major)) {
        return USP_ERR_CUDA;
    }
    BwdArgs ba{};
    ba.cu = cu_seqlens;
    ba.items = sa.items;
    ba.hdr = hdr;
    ba.lse = lse;
    ba.delta = delta;
    ba.amax = amax;
    ba.dq_acc = dq_acc;
    ba.dk = dk;
    ba.dv = dv;
    ba.grad_fp32 = fp32_grads ? 1 : 0;
    ba.out_f16 = f16;
    ba.T = total_tokens;
    ba.hq = hq;
    ba.hkv = hkv;
    ba.token_major = token_major;
    ba.group = hq / hkv;
    ba.causal = sa.causal;
    ba.scale = resolve_softmax_scale(softmax_scale, head_dim);
    ba.scale_log2 = ba.scale * 1.4426950408889634f;
    ba.ds_exp = ds_exponent(head_dim, ba.scale);
    if (launch_attn_bwd(head_dim, mq, mk, mv, mdo, mdq, mdk, mdv, ba, w.max_items, s) != cudaSuccess)
        return USP_ERR_CUDA;
    if (launch_dq_convert(dq_acc, dq, amax, total_tokens, hq, hkv, head_dim, token_major, (int)grad_dt, ba.ds_exp,
                          s) != cudaSuccess)
        return USP_ERR_CUDA;
    return USP_OK;
}

// sp simulated ranks: the head counts must divide over them and the sequence must be
// padded to a multiple of sp_size (HF guide, "Configurar").
usp_status check_sp(int sp, int64_t total_tokens, int hq, int hkv) {
    if (sp < 1 || hq < 1 || hkv < 1 || total_tokens < 0) return USP_ERR_INVALID_ARG;
    if (hq % sp != 0 || total_tokens % sp != 0) return USP_ERR_INVALID_ARG;
    // key/value heads either split over the ranks or, with fewer heads than ranks, each
    // replicated over sp / hkv ranks (the fused kernels read the shared head in place)
    if (hkv % sp != 0 && sp % hkv != 0) return USP_ERR_INVALID_ARG;
    return USP_OK;
}

}  // namespace
}  // namespace usp

extern "C" usp_status usp_attn_fwd_varlen(const void* q, const void* k, const void* v, void* o, void* o_res,
                                          float* lse, const int32_t* cu_seqlens, int num_seqs, int64_t total_tokens,
                                          int hq, int hkv, int head_dim, float softmax_scale, int causal,
                                          void* workspace, size_t ws_bytes, void* stream) {
    return attn_fwd_impl(q, k, v, o, o_res, lse, cu_seqlens, num_seqs, total_tokens, hq, hkv, head_dim, softmax_scale,
                         causal, workspace, ws_bytes, (cudaStream_t)stream, 0);
}

extern "C" usp_status usp_attn_bwd_varlen(const void* q, const void* k, const void* v, const void* o,
                                          const void* o_res, const float* lse, const void* d_o, void* dq, void* dk,
                                          void* dv, usp_dtype grad_dt, const int32_t* cu_seqlens, int num_seqs,
                                          int64_t total_tokens, int hq, int hkv, int head_dim, float softmax_scale,
                                          int causal, void* workspace, size_t ws_bytes, void* stream) {
    return attn_bwd_impl(q, k, v, o, o_res, lse, d_o, dq, dk, dv, grad_dt, cu_seqlens, num_seqs, total_tokens, hq,
                         hkv, head_dim, softmax_scale, causal, workspace, ws_bytes, (cudaStream_t)stream, 0);
}

extern "C" usp_status usp_ulysses_attn_fwd(const void* q, const void* k, const void* v, void* o, void* o_res,
                                           float* lse, const int32_t* cu_seqlens, int num_seqs, int64_t total_tokens,
                                           int sp, int hq, int hkv, int head_dim, float softmax_scale, int causal,
                                           usp_dtype dt, void* workspace, size_t ws_bytes, void* stream) {
    const usp_status st = check_sp(sp, total_tokens, hq, hkv);
    if (st != USP_OK) return st;
    return attn_fwd_impl(q, k, v, o, o_res, lse, cu_seqlens, num_seqs, total_tokens, hq, hkv, head_dim, softmax_scale,
                         causal, workspace, ws_bytes, (cudaStream_t)stream, 1, dt);
}

extern "C" usp_status usp_ulysses_attn_bwd(const void* q, const void* k, const void* v, const void* o,
                                           const void* o_res, const float* lse, const void* d_o, void* dq, void* dk,
                                           void* dv, usp_dtype grad_dt, const int32_t* cu_seqlens, int num_seqs,
                                           int64_t total_tokens, int sp, int hq, int hkv, int head_dim,
                                           float softmax_scale, int causal, usp_dtype dt, void* workspace,
                                           size_t ws_bytes, void* stream) {
    const usp_status st = check_sp(sp, total_tokens, hq, hkv);
    if (st != USP_OK) return st;
    return attn_bwd_impl(q, k, v, o, o_res, lse, d_o, dq, dk, dv, grad_dt, cu_seqlens, num_seqs, total_tokens, hq,
                         hkv, head_dim, softmax_scale, causal, workspace, ws_bytes, (cudaStream_t)stream, 1, dt);
}

extern "C" usp_status usp_get_device_status(const void* workspace, void* stream) {
    if (!workspace) return USP_ERR_INVALID_ARG;
    cudaStream_t s = (cudaStream_t)stream;
    if (cudaStreamSynchronize(s) != cudaSuccess) return USP_ERR_CUDA;
    int status = 0;
    if (cudaMemcpy(&status, workspace, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return USP_ERR_CUDA;
    return (usp_status)status;
}

extern "C" const char* usp_status_string(usp_status status) {
    switch (status) {
        case USP_OK: return "USP_OK";
        case USP_ERR_INVALID_ARG: return "USP_ERR_INVALID_ARG";
        case USP_ERR_UNSUPPORTED: return "USP_ERR_UNSUPPORTED";
        case USP_ERR_CUDA: return "USP_ERR_CUDA";
        case USP_ERR_WORKSPACE: return "USP_ERR_WORKSPACE";
        case USP_ERR_TIMEOUT: return "USP_ERR_TIMEOUT";
        case USP_ERR_DEVICE_CHECK: return "USP_ERR_DEVICE_CHECK";
    }
    return "USP_ERR_UNKNOWN";
}

extern "C" usp_status usp_debug_wait_timeout(void* workspace, size_t ws_bytes, uint64_t limit_ns, void* stream) {
    if (!workspace || ws_bytes < sizeof(WsHeader) || !aligned16(workspace)) return USP_ERR_INVALID_ARG;
    if (limit_ns < 1000) limit_ns = 1000;
    if (limit_ns > 5000000000ull) limit_ns = 5000000000ull;
    cudaStream_t s = (cudaStream_t)stream;
    if (cudaMemsetAsync(workspace, 0, sizeof(WsHeader), s) != cudaSuccess) return USP_ERR_CUDA;
    if (launch_debug_timeout((WsHeader*)workspace, limit_ns, s) != cudaSuccess) return USP_ERR_CUDA;
    return USP_OK;
}
