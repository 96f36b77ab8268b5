// Shared definitions of the library: workspace layout, work items, limits.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cmath>
#include <mutex>

#include <cuda_runtime.h>

#include "usp.h"

namespace usp {

// Rows of one attention tile (tensor-core M) and of one key/value block (N).
constexpr int kTileM = 128;
constexpr int kBlockN = 128;
// A forward work item is four query tiles (512 rows) for head_dim 128, run by a pair of CTAs
// sharing each MMA, and two (256 rows) for head_dim 64, run by one CTA; a backward item is
// one key/value tile.
__host__ __device__ constexpr int fwd_rows_per_item(int head_dim) { return head_dim == 128 ? 4 * kTileM : 2 * kTileM; }
constexpr int kFwdRowsMax = 4 * kTileM;
constexpr int kBwdRowsPerItem = kTileM;

// Wall-clock limit of every bounded wait inside the attention kernels, and of the
// teardown waits for copies and MMAs already in flight.
constexpr uint64_t kWaitLimitNs = 2000000000ull;
constexpr uint64_t kDrainLimitNs = 200000000ull;

// A unit of work: (head, sample, tile index within the sample). `head` is a query
// head for the forward and a key/value head for the backward.
struct WorkItem {
    int head;
    int seq;
    int tile;
    int cost;
};

// Workspace layout (all offsets 256-byte aligned):
//   [0, 256)         header: status word, forward item count, backward item count
//   hist             int32[hist_len]   scheduler cost histogram / bucket cursors
//   tiles_prefix     int32[num_seqs+1] tiles per sample, prefix-summed
//   sample_base      int32[num_seqs+1] backward: first tile of each sample in the work order
//   items            WorkItem[max_items]
//   delta            fp32[hq][T]       backward only: Delta_i = dO_i . O_i
//   dq_acc           fp32[hq][T][D]    backward only: dQ accumulator
//   amax             u32[4][hkv]       backward only: largest |q|, |k|, |v|, |dO| per key/value group
//   q16, k16, v16, do16                backward only: scaled fp16 operand copies, head-major
struct WsHeader {
    int status;
    int fwd_count;
    int bwd_count;
    int max_cost;
    int bwd_next;  // backward work items handed out past the first one of each CTA
    int fwd_next;  // the same for the forward
};

struct WsLayout {
    size_t hist, prefix, sbase, items, delta, dq_acc, amax, q16, k16, v16, do16, total;
    int hist_len;
    int max_items;
};

// Row (of head_dim elements) holding token t of head h: head-major [H][T][D] (the
// head-sharded layout) or token-major [T][H][D] (the seq-sharded layout of all ranks).
__host__ __device__ __forceinline__ int64_t act_row(int h, int64_t t, int64_t T, int H, int token_major) {
    return token_major ? t * H + h : (int64_t)h * T + t;
}

// Host-side checks shared by every attention entry point: sizes, head counts and the
// limits of the work-list indexing (item counts and offsets stay within int).
inline usp_status check_attn_sizes(int64_t T, int num_seqs, int hq, int hkv, int D, const int32_t* cu) {
    if (T < 0 || hq < 1 || hkv < 1 || hq % hkv != 0) return USP_ERR_INVALID_ARG;
    if (T > 0 && (num_seqs < 1 || !cu)) return USP_ERR_INVALID_ARG;
    if (T > (int64_t)2147483647 - 2 * kFwdRowsMax || num_seqs > (1 << 24)) return USP_ERR_UNSUPPORTED;
    if (D != 64 && D != 128) return USP_ERR_UNSUPPORTED;
    if ((int64_t)hq * (T / kTileM + num_seqs + 1) > (int64_t)2147483647 / 2) return USP_ERR_UNSUPPORTED;
    return USP_OK;
}

// softmax_scale <= 0 selects 1/sqrt(D).
inline float resolve_softmax_scale(float softmax_scale, int D) {
    return softmax_scale > 0.f ? softmax_scale : 1.0f / sqrtf((float)D);
}

inline size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

inline int64_t ceil_div64(int64_t a, int64_t b) { return (a + b - 1) / b; }

inline WsLayout ws_layout(int64_t T, int num_seqs, int hq, int hkv, int D, int bwd) {
    WsLayout w{};
    const int64_t rows_per_item = bwd ? kBwdRowsPerItem : fwd_rows_per_item(D);
    const int64_t heads = bwd ? hkv : hq;
    const int64_t tiles = ceil_div64(T, rows_per_item) + num_seqs;
    // costs are counted in key/value blocks (x query heads per kv head for the backward)
    const int64_t max_cost = 2 * (ceil_div64(T, kBlockN) + 2) * (bwd ? (hq / (hkv > 0 ? hkv : 1)) : 1) + 8;
    w.hist_len = (int)max_cost;
    w.max_items = (int)(tiles * heads);
    size_t off = 256;
    w.hist = off;
    off = align256(off + sizeof(int) * (size_t)w.hist_len);
    w.prefix = off;
    off = align256(off + sizeof(int) * (size_t)(num_seqs + 1));
    w.sbase = off;
    off = align256(off + sizeof(int) * (size_t)(num_seqs + 1));
    w.items = off;
    off = align256(off + sizeof(WorkItem) * (size_t)w.max_items);
    w.delta = off;
    if (bwd) off = align256(off + sizeof(float) * (size_t)hq * (size_t)T);
    w.dq_acc = off;
    if (bwd) off = align256(off + sizeof(float) * (size_t)hq * (size_t)T * (size_t)D);
    const size_t qbytes = 2 * (size_t)hq * (size_t)T * (size_t)D, kvbytes = 2 * (size_t)hkv * (size_t)T * (size_t)D;
    w.amax = off;
    if (bwd) off = align256(off + sizeof(uint32_t) * 4 * (size_t)hkv);
    w.q16 = off;
    if (bwd) off = align256(off + qbytes);
    w.k16 = off;
    if (bwd) off = align256(off + kvbytes);
    w.v16 = off;
    if (bwd) off = align256(off + kvbytes);
    w.do16 = off;
    if (bwd) off = align256(off + qbytes);
    w.total = off;
    return w;
}

constexpr int kMaxDevices = 64;

// SM count of the current device, read once per device (thread-safe); 0 if it cannot be read.
inline int device_sm_count() {
    static std::mutex mu;
    static int sms[kMaxDevices] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
    std::lock_guard<std::mutex> lock(mu);
    if (sms[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
        sms[dev] = n;
    }
    return sms[dev];
}

// One-time set-up of a persistent kernel on the current device: raises the dynamic shared-
// memory limit of `Kernel` to `smem` (once per device and kernel -- the flags are per template
// instance, so per kernel -- under a lock, so concurrent first calls from several host threads
// and calls on several devices of one process are safe) and returns the device's SM count in *sms.
template <auto Kernel>
cudaError_t persistent_setup(size_t smem, int* sms) {
    static std::mutex mu;
    static bool done[kMaxDevices] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    {
        std::lock_guard<std::mutex> lock(mu);
        if (!done[dev]) {
            e = cudaFuncSetAttribute(Kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
            if (e != cudaSuccess) return e;
            done[dev] = true;
        }
    }
    *sms = device_sm_count();
    return *sms > 0 ? cudaSuccess : cudaErrorInvalidDevice;
}

// persistent_setup for a kernel launched in clusters of `cluster_x` CTAs: *units is how many
// clusters can be resident at once on the device (a cluster's CTAs share one GPC, so an SM
// count alone can overstate it), computed once per device.
template <auto Kernel>
cudaError_t persistent_cluster_setup(size_t smem, int threads, int cluster_x, int* units) {
    static std::mutex mu;
    static int clusters[kMaxDevices] = {};
    int sms = 0;
    cudaError_t e = persistent_setup<Kernel>(smem, &sms);
    if (e != cudaSuccess) return e;
    int dev = 0;
    e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lock(mu);
    if (clusters[dev] == 0) {
        cudaLaunchAttribute attr;
        attr.id = cudaLaunchAttributeClusterDimension;
        attr.val.clusterDim.x = (unsigned)cluster_x;
        attr.val.clusterDim.y = 1;
        attr.val.clusterDim.z = 1;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)(sms / cluster_x * cluster_x));
        cfg.blockDim = dim3((unsigned)threads);
        cfg.dynamicSmemBytes = smem;
        cfg.attrs = &attr;
        cfg.numAttrs = 1;
        int n = 0;
        e = cudaOccupancyMaxActiveClusters(&n, Kernel, &cfg);
        if (e != cudaSuccess) return e;
        if (n < 1) return cudaErrorInvalidConfiguration;
        clusters[dev] = n;
    }
    *units = clusters[dev];
    return cudaSuccess;
}

// Launches `kernel` on stream s; with `programmatic` the launch may overlap the end of the
// previous kernel in the stream, and the kernel must call pdl_wait() before it reads
// anything that kernel (or one before it) wrote.
template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                          bool programmatic, Args... args) {
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cfg.attrs = programmatic ? &attr : nullptr;
    cfg.numAttrs = programmatic ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// launch_kernel for clusters of `cluster_x` CTAs along x (gridDim.x a multiple of it).
template <typename... KArgs, typename... Args>
cudaError_t launch_kernel_cluster(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                                  bool programmatic, int cluster_x, Args... args) {
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)cluster_x;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = programmatic ? 2 : 1;
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}

}  // namespace usp
