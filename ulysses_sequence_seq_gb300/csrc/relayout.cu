// The two all-to-alls of Ulysses sequence parallelism as device-local permutations.
//
// With sp simulated ranks stored as shards of one buffer, the seq-sharded tensor
// [sp][T/sp][H][D] has the bytes of a token-major [T][H][D] tensor and the
// head-sharded tensor [sp][H/sp][T][D] those of a head-major [H][T][D] tensor
// (token t = r_s*S + s and head h = r*Hl + hl). So on one device both swaps are a
// (token, head) transpose of whole D-element rows, and sp only enters through the
// validation (HF Transformers "Ulysses sequence parallelism" guide: layout figure,
// and "Configurar" for the divisibility and padding rules).
//
// The kernel is a pure bandwidth copy: every thread moves 16-byte chunks, a row of
// D elements is copied by CPR consecutive threads, so both the reads and the writes
// of a warp cover whole contiguous rows (256 bytes at D = 128, bf16).
#include <cuda_runtime.h>

#include <climits>
#include <cstdint>

#include "common.cuh"

namespace usp {
namespace {

__device__ __forceinline__ uint4 ld_stream(const uint4* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// CPR: 16-byte chunks per row (a power of two). to_head: seq-sharded -> head-sharded.
template <int CPR>
__global__ void __launch_bounds__(256) relayout_rows_kernel(const uint4* __restrict__ in, uint4* __restrict__ out,
                                                            int T, int H, int to_head) {
    constexpr int kRowsPerPass = (256 / CPR) > 0 ? (256 / CPR) : 1;
    constexpr int kThreadsPerRow = CPR < 256 ? CPR : 256;
    constexpr int kUnroll = 4;
    const int h = blockIdx.y;
    const int lr = threadIdx.x / kThreadsPerRow;
    const int c0 = threadIdx.x % kThreadsPerRow;
    const int64_t step = (int64_t)gridDim.x * kRowsPerPass * kUnroll;
    for (int64_t t0 = (int64_t)blockIdx.x * kRowsPerPass * kUnroll; t0 < T; t0 += step) {
#pragma unroll 1
        for (int c = c0; c < CPR; c += kThreadsPerRow) {
            uint4 v[kUnroll];
            int64_t dst[kUnroll];
            bool ok[kUnroll];
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                const int64_t t = t0 + (int64_t)u * kRowsPerPass + lr;
                ok[u] = t < T;
                const int64_t head_row = (int64_t)h * T + t;  // [H][T] row
                const int64_t seq_row = t * H + h;             // [T][H] row
                const int64_t src = to_head ? seq_row : head_row;
                dst[u] = to_head ? head_row : seq_row;
                if (ok[u]) v[u] = ld_stream(in + src * CPR + c);
            }
#pragma unroll
            for (int u = 0; u < kUnroll; ++u)
                if (ok[u]) out[dst[u] * CPR + c] = v[u];
        }
    }
}

// Rows whose byte size is a multiple of 16 but whose chunk count is not a power of two.
__global__ void __launch_bounds__(256) relayout_rows_generic_kernel(const uint4* __restrict__ in,
                                                                    uint4* __restrict__ out, int T, int H, int cpr,
                                                                    int to_head) {
    const int h = blockIdx.y;
    const int64_t total = (int64_t)T * cpr;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t t = i / cpr;
        const int c = (int)(i - t * cpr);
        const int64_t head_row = (int64_t)h * T + t;
        const int64_t seq_row = t * H + h;
        const int64_t src = to_head ? seq_row : head_row;
        const int64_t dst = to_head ? head_row : seq_row;
        out[dst * cpr + c] = in[src * cpr + c];
    }
}

int num_sms_cached() {
    static int sms = 0;
    if (sms == 0) {
        int dev = 0, n = 0;
        if (cudaGetDevice(&dev) == cudaSuccess &&
            cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && n > 0)
            sms = n;
        else
            return 148;
    }
    return sms;
}

usp_status relayout(const void* in, void* out, int sp, int64_t T, int heads, int head_dim, usp_dtype dt,
                    void* stream, int to_head) {
    if (sp < 1 || T < 0 || heads < 1 || head_dim < 1) return USP_ERR_INVALID_ARG;
    if (heads % sp != 0 || T % sp != 0) return USP_ERR_INVALID_ARG;
    if (T == 0) return USP_OK;  // empty buffers may have NULL addresses
    if (!in || !out) return USP_ERR_INVALID_ARG;
    if (((uintptr_t)in & 15) || ((uintptr_t)out & 15)) return USP_ERR_INVALID_ARG;
    size_t esize;
    switch (dt) {
        case USP_BF16:
        case USP_FP16: esize = 2; break;
        case USP_FP32: esize = 4; break;
        default: return USP_ERR_INVALID_ARG;
    }
    if (T > INT_MAX || heads > 65535) return USP_ERR_UNSUPPORTED;
    const size_t row_bytes = esize * (size_t)head_dim;
    if (row_bytes % 16 != 0) return USP_ERR_UNSUPPORTED;
    const size_t bytes = row_bytes * (size_t)heads * (size_t)T;
    const uintptr_t a = (uintptr_t)in, b = (uintptr_t)out;
    if (bytes > 0 && a < b + bytes && b < a + bytes) return USP_ERR_INVALID_ARG;
    const int cpr = (int)(row_bytes / 16);
    cudaStream_t s = (cudaStream_t)stream;
    // Enough CTAs to keep every SM streaming: ~16 CTAs of 256 threads per SM in total.
    const int64_t want = (int64_t)num_sms_cached() * 16;
    int gx = (int)((want + heads - 1) / heads);
    const int rows_per_cta = 4 * (cpr <= 256 ? (256 / (cpr < 256 ? cpr : 256)) : 1);
    const int64_t max_gx = (T + rows_per_cta - 1) / rows_per_cta;
    if (gx > max_gx) gx = (int)max_gx;
    if (gx < 1) gx = 1;
    dim3 grid(gx, heads);
    const uint4* src = (const uint4*)in;
    uint4* dst = (uint4*)out;
    const int t = (int)T;
    switch (cpr) {
        case 1: relayout_rows_kernel<1><<<grid, 256, 0, s>>>(src, dst, t, heads, to_head); break;
        case 2: relayout_rows_kernel<2><<<grid, 256, 0, s>>>(src, dst, t, heads, to_head); break;
        case 4: relayout_rows_kernel<4><<<grid, 256, 0, s>>>(src, dst, t, heads, to_head); break;
        case 8: relayout_rows_kernel<8><<<grid, 256, 0, s>>>(src, dst, t, heads, to_head); break;
        case 16: relayout_rows_kernel<16><<<grid, 256, 0, s>>>(src, dst, t, heads, to_head); break;
        case 32: relayout_rows_kernel<32><<<grid, 256, 0, s>>>(src, dst, t, heads, to_head); break;
        case 64: relayout_rows_kernel<64><<<grid, 256, 0, s>>>(src, dst, t, heads, to_head); break;
        default: {
            dim3 g2((unsigned)((want + heads - 1) / heads), heads);
            relayout_rows_generic_kernel<<<g2, 256, 0, s>>>(src, dst, t, heads, cpr, to_head);
        }
    }
    return cudaGetLastError() == cudaSuccess ? USP_OK : USP_ERR_CUDA;
}

}  // namespace
}  // namespace usp

extern "C" usp_status usp_seq_to_head(const void* in, void* out, int sp, int64_t total_tokens, int heads,
                                      int head_dim, usp_dtype dt, void* stream) {
    return usp::relayout(in, out, sp, total_tokens, heads, head_dim, dt, stream, 1);
}

extern "C" usp_status usp_head_to_seq(const void* in, void* out, int sp, int64_t total_tokens, int heads,
                                      int head_dim, usp_dtype dt, void* stream) {
    return usp::relayout(in, out, sp, total_tokens, heads, head_dim, dt, stream, 0);
}
