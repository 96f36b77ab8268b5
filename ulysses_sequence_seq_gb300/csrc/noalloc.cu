// Attention forward for callers that cannot allocate device memory.
//
// usp_attn_fwd_varlen needs a caller-provided workspace for its scratch data: the
// status word, the scheduler's cost histogram and prefix sums, and the varlen work
// list. Some callers have no way to provide one: code inside a framework whose
// caching allocator owns all device memory and does not tolerate raw
// cudaMalloc/cudaFree next to it, real-time or embedded hosts that reserve a fixed
// memory budget up front and must not allocate per call, and plug-in code called
// through a hook with no allocator handle and nowhere to keep a workspace between
// calls. This entry point serves them: its scratch is a fixed array in the
// library's own device memory.
//
// The array is a file-scope `static __device__` object of kNoAllocScratchBytes
// (1 MiB). Every GPU that loads the library keeps it until the process exits, and
// every call shares it, so calls that overlap on the GPU (e.g. on two streams, or
// from two host threads without ordering) race on it and must be serialised by the
// caller. The array keeps the previous call's contents; the parts that must start
// at zero (status word and item count) are cleared by each call.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <mutex>

#include "attn.cuh"
#include "common.cuh"
#include "sched.cuh"

namespace usp {
namespace {

constexpr size_t kNoAllocScratchBytes = size_t(1) << 20;

// In host code this name is only a host-side stand-in for the device object; its
// device address must be obtained with cudaGetSymbolAddress on each device.
static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_setup_mutex;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device, looked up once per device
// (the first call may load the library's device code onto that device).
cudaError_t scratch_on_current_device(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (!g_scratch_ptr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return cudaSuccess;
}

}  // namespace
}  // namespace usp

using namespace usp;

extern "C" usp_status usp_attn_fwd_varlen_noalloc(const void* q, const void* k, const void* v, void* o, float* lse,
                                                  const int32_t* cu_seqlens, int num_seqs, int64_t total_tokens,
                                                  int hq, int hkv, int head_dim, float softmax_scale, int causal,
                                                  int32_t* status, void* stream) {
    const usp_status st = check_attn_sizes(total_tokens, num_seqs, hq, hkv, head_dim, cu_seqlens);
    if (st != USP_OK) return st;
    if (status && ((uintptr_t)status & 3)) return USP_ERR_INVALID_ARG;
    cudaStream_t s = (cudaStream_t)stream;
    if (total_tokens == 0) {
        if (status && cudaMemsetAsync(status, 0, sizeof(int32_t), s) != cudaSuccess) return USP_ERR_CUDA;
        return USP_OK;
    }
    if (!q || !k || !v || !o || !lse) return USP_ERR_INVALID_ARG;
    const uintptr_t mis = (uintptr_t)q | (uintptr_t)k | (uintptr_t)v | (uintptr_t)o | (uintptr_t)lse;
    if (mis & 15) return USP_ERR_INVALID_ARG;
    // the scratch holds the forward's work list: it bounds tokens, samples and heads together
    if (total_tokens > ((int64_t)1 << 30)) return USP_ERR_WORKSPACE;
    const WsLayout w = ws_layout(total_tokens, num_seqs, hq, hkv, head_dim, 0);
    if (w.total > kNoAllocScratchBytes) return USP_ERR_WORKSPACE;

    void* scratch = nullptr;
    if (scratch_on_current_device(&scratch) != cudaSuccess) return USP_ERR_CUDA;
    uint8_t* ws = (uint8_t*)scratch;
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

    CUtensorMap mq, mk, mv, mo;   // o doubles as the (unused) residual map: fa.o_res is NULL
    if (!make_activation_map(&mq, q, total_tokens, hq, head_dim, 0) ||
        !make_activation_map(&mk, k, total_tokens, hkv, head_dim, 0, fwd_k_box_rows(head_dim)) ||
        !make_activation_map(&mv, v, total_tokens, hkv, head_dim, 0) ||
        !make_activation_map(&mo, o, total_tokens, hq, head_dim, 0))
        return USP_ERR_CUDA;
    FwdArgs fa{};
    fa.cu = cu_seqlens;
    fa.items = sa.items;
    fa.hdr = hdr;
    fa.o = (uint16_t*)o;
    fa.lse = lse;
    fa.T = total_tokens;
    fa.hq = hq;
    fa.group = hq / hkv;
    fa.causal = sa.causal;
    fa.scale_log2 = resolve_softmax_scale(softmax_scale, head_dim) * 1.4426950408889634f;
    if (launch_attn_fwd(head_dim, mq, mk, mv, mo, mo, fa, w.max_items, s) != cudaSuccess) return USP_ERR_CUDA;
    // device-side outcome (USP_OK, USP_ERR_DEVICE_CHECK or USP_ERR_TIMEOUT) for the caller
    if (status && cudaMemcpyAsync(status, &hdr->status, sizeof(int32_t), cudaMemcpyDeviceToDevice, s) != cudaSuccess)
        return USP_ERR_CUDA;
    return USP_OK;
}
