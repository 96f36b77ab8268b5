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
// The grid's y index is the head-sharded head; with rep > 1 (key/value heads replicated
// over the ranks, seq -> head only) it reads seq-sharded head y / rep.
template <int CPR>
__global__ void __launch_bounds__(256) relayout_rows_kernel(const uint4* __restrict__ in, uint4* __restrict__ out,
                                                            int T, int H, int to_head, int rep) {
    constexpr int kRowsPerPass = (256 / CPR) > 0 ? (256 / CPR) : 1;
    constexpr int kThreadsPerRow = CPR < 256 ? CPR : 256;
    constexpr int kUnroll = 4;
    const int hy = blockIdx.y;          // head-sharded head
    const int h = hy / rep;             // seq-sharded head
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
                const int64_t head_row = (int64_t)hy * T + t;  // [H*rep][T] row
                const int64_t seq_row = t * H + h;              // [T][H] row
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
                                                                    int to_head, int rep) {
    const int hy = blockIdx.y;
    const int h = hy / rep;
    const int64_t total = (int64_t)T * cpr;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t t = i / cpr;
        const int c = (int)(i - t * cpr);
        const int64_t head_row = (int64_t)hy * T + t;
        const int64_t seq_row = t * H + h;
        const int64_t src = to_head ? seq_row : head_row;
        const int64_t dst = to_head ? head_row : seq_row;
        out[dst * cpr + c] = in[src * cpr + c];
    }
}

// Gradient of a replicated key/value head: out[t][g] = sum over its rep replicas
// in[g*rep + i][t], accumulated in fp32 in replica order and rounded once. Eight bf16
// (or four fp32) elements per thread.
template <bool kBf16>
__global__ void __launch_bounds__(256) sum_replicas_kernel(const uint4* __restrict__ in, uint4* __restrict__ out,
                                                           int64_t T, int H, int cpr, int rep) {
    const int g = blockIdx.y;
    const int64_t total = T * cpr;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t t = i / cpr;
        const int c = (int)(i - t * cpr);
        float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        for (int r = 0; r < rep; ++r) {
            const uint4 v = ld_stream(in + (((int64_t)g * rep + r) * T + t) * cpr + c);
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
            if (kBf16) {
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    acc[2 * j] += __uint_as_float(w[j] << 16);
                    acc[2 * j + 1] += __uint_as_float(w[j] & 0xffff0000u);
                }
            } else {
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[j] += __uint_as_float(w[j]);
            }
        }
        uint4 o;
        if (kBf16) {
            uint32_t w[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                uint32_t pr;
                asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(pr) : "f"(acc[2 * j + 1]), "f"(acc[2 * j]));
                w[j] = pr;
            }
            o = make_uint4(w[0], w[1], w[2], w[3]);
        } else {
            o = make_uint4(__float_as_uint(acc[0]), __float_as_uint(acc[1]), __float_as_uint(acc[2]),
                           __float_as_uint(acc[3]));
        }
        out[(t * H + g) * cpr + c] = o;
    }
}

int num_sms_cached() {
    const int sms = device_sm_count();
    return sms > 0 ? sms : 148;
}

// rep > 1: seq -> head with every seq-sharded head copied to rep consecutive
// head-sharded heads (heads * rep == sp).
usp_status relayout(const void* in, void* out, int sp, int64_t T, int heads, int head_dim, usp_dtype dt,
                    void* stream, int to_head, int rep = 1) {
    if (sp < 1 || T < 0 || heads < 1 || head_dim < 1) return USP_ERR_INVALID_ARG;
    if ((heads * rep) % sp != 0 || T % sp != 0) return USP_ERR_INVALID_ARG;
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
    const size_t in_bytes = row_bytes * (size_t)heads * (size_t)T;
    const size_t out_bytes = in_bytes * (size_t)rep;
    const uintptr_t a = (uintptr_t)in, b = (uintptr_t)out;
    if (in_bytes > 0 && a < b + out_bytes && b < a + in_bytes) return USP_ERR_INVALID_ARG;
    const int cpr = (int)(row_bytes / 16);
    cudaStream_t s = (cudaStream_t)stream;
    // Enough CTAs to keep every SM streaming: ~16 CTAs of 256 threads per SM in total.
    const int64_t want = (int64_t)num_sms_cached() * 16;
    const int ys = heads * rep;   // grid rows: head-sharded heads
    int gx = (int)((want + ys - 1) / ys);
    const int rows_per_cta = 4 * (cpr <= 256 ? (256 / (cpr < 256 ? cpr : 256)) : 1);
    const int64_t max_gx = (T + rows_per_cta - 1) / rows_per_cta;
    if (gx > max_gx) gx = (int)max_gx;
    if (gx < 1) gx = 1;
    dim3 grid(gx, ys);
    const uint4* src = (const uint4*)in;
    uint4* dst = (uint4*)out;
    const int t = (int)T;
    switch (cpr) {
        case 1: relayout_rows_kernel<1><<<grid, 256, 0, s>>>(src, dst, t, heads, to_head, rep); break;
        case 2: relayout_rows_kernel<2><<<grid, 256, 0, s>>>(src, dst, t, heads, to_head, rep); break;
        case 4: relayout_rows_kernel<4><<<grid, 256, 0, s>>>(src, dst, t, heads, to_head, rep); break;
        case 8: relayout_rows_kernel<8><<<grid, 256, 0, s>>>(src, dst, t, heads, to_head, rep); break;
        case 16: relayout_rows_kernel<16><<<grid, 256, 0, s>>>(src, dst, t, heads, to_head, rep); break;
        case 32: relayout_rows_kernel<32><<<grid, 256, 0, s>>>(src, dst, t, heads, to_head, rep); break;
        case 64: relayout_rows_kernel<64><<<grid, 256, 0, s>>>(src, dst, t, heads, to_head, rep); break;
        default: {
            dim3 g2((unsigned)((want + ys - 1) / ys), ys);
            relayout_rows_generic_kernel<<<g2, 256, 0, s>>>(src, dst, t, heads, cpr, to_head, rep);
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

// Key/value heads over sp ranks. With hkv % sp == 0 these are the plain swaps. With
// hkv < sp (sp % hkv == 0) every rank holds one key/value head, kv head r * hkv / sp, so
// each head is replicated sp / hkv times on the way in, and the gradients of the
// replicas are summed on the way out.
namespace usp {
namespace {
usp_status kv_rep(int sp, int hkv, int* rep) {
    if (sp < 1 || hkv < 1) return USP_ERR_INVALID_ARG;
    if (hkv % sp == 0) { *rep = 1; return USP_OK; }
    if (sp % hkv == 0) { *rep = sp / hkv; return USP_OK; }
    return USP_ERR_INVALID_ARG;
}
}  // namespace
}  // namespace usp

extern "C" usp_status usp_seq_to_head_kv(const void* in, void* out, int sp, int64_t total_tokens, int hkv,
                                         int head_dim, usp_dtype dt, void* stream) {
    int rep = 1;
    const usp_status st = usp::kv_rep(sp, hkv, &rep);
    if (st != USP_OK) return st;
    return usp::relayout(in, out, sp, total_tokens, hkv, head_dim, dt, stream, 1, rep);
}

extern "C" usp_status usp_head_to_seq_kv_grad(const void* in, void* out, int sp, int64_t total_tokens, int hkv,
                                              int head_dim, usp_dtype dt, void* stream) {
    int rep = 1;
    usp_status st = usp::kv_rep(sp, hkv, &rep);
    if (st != USP_OK) return st;
    if (rep == 1) return usp::relayout(in, out, sp, total_tokens, hkv, head_dim, dt, stream, 0);
    if (total_tokens < 0 || head_dim < 1 || total_tokens % sp != 0) return USP_ERR_INVALID_ARG;
    if (total_tokens == 0) return USP_OK;
    if (!in || !out || ((uintptr_t)in & 15) || ((uintptr_t)out & 15)) return USP_ERR_INVALID_ARG;
    if (dt != USP_BF16 && dt != USP_FP32) return USP_ERR_UNSUPPORTED;
    const size_t esize = dt == USP_FP32 ? 4 : 2;
    const size_t row_bytes = esize * (size_t)head_dim;
    if (row_bytes % 16 != 0 || total_tokens > INT_MAX || hkv > 65535) return USP_ERR_UNSUPPORTED;
    const size_t out_bytes = row_bytes * (size_t)hkv * (size_t)total_tokens, in_bytes = out_bytes * (size_t)rep;
    const uintptr_t a = (uintptr_t)in, b = (uintptr_t)out;
    if (a < b + out_bytes && b < a + in_bytes) return USP_ERR_INVALID_ARG;
    const int cpr = (int)(row_bytes / 16);
    const int64_t want = (int64_t)usp::num_sms_cached() * 16;
    dim3 grid((unsigned)((want + hkv - 1) / hkv), hkv);
    cudaStream_t s = (cudaStream_t)stream;
    if (dt == USP_BF16)
        usp::sum_replicas_kernel<true><<<grid, 256, 0, s>>>((const uint4*)in, (uint4*)out, total_tokens, hkv, cpr, rep);
    else
        usp::sum_replicas_kernel<false><<<grid, 256, 0, s>>>((const uint4*)in, (uint4*)out, total_tokens, hkv, cpr, rep);
    return cudaGetLastError() == cudaSuccess ? USP_OK : USP_ERR_CUDA;
}
