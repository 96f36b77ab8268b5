// Ring-attention steps built from the attention calls: merging partial results through
// their log-sum-exp, the final rounding of the merged output, and fp32 accumulation of
// gradient shares.
//
// In ring attention every rank keeps a chunk of the queries while the key/value chunks go
// around the ring; each step attends the local queries to the visiting chunk, and the
// partial outputs are combined through their log-sum-exp (ColossalAI sequence parallelism
// tutorial, the ring-attention plugin set-up and its closing comparison of Ulysses and ring
// attention). With equal chunks of one (packed, evenly split) sequence, the causal mask on
// global positions makes every step either unmasked (an earlier key chunk), causal (the
// query chunk's own keys) or empty (a later one), so a step is one attention call of the
// library with causal 0 or 1; these kernels do the rest. All three are HBM-bound.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "common.cuh"
#include "ptx.cuh"

namespace usp {
namespace {

using namespace ptx;

// 8 elements per thread. Row (h, t) of a [T][H][D] (token-major) or [H][T][D] tensor.
template <bool F16>
__global__ void __launch_bounds__(256) lse_merge_kernel(float* __restrict__ o_acc, float* __restrict__ lse_acc,
                                                        const uint16_t* __restrict__ o_part,
                                                        const uint16_t* __restrict__ o_part_res,
                                                        const float* __restrict__ lse_part, int64_t T, int H, int D,
                                                        int token_major, int init) {
    const int per_row = D / 8;
    const int64_t total = T * H * per_row;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
        const int c = (int)(i % per_row);
        const int64_t row = i / per_row;            // h * T + t
        const int h = (int)(row / T);
        const int64_t t = row - (int64_t)h * T;
        const int64_t off = act_row(h, t, T, H, token_major) * D + 8 * c;
        const uint4 pv = __ldg((const uint4*)(o_part + off));
        const uint4 rv = o_part_res ? __ldg((const uint4*)(o_part_res + off)) : make_uint4(0, 0, 0, 0);
        const uint32_t pw[4] = {pv.x, pv.y, pv.z, pv.w}, rw[4] = {rv.x, rv.y, rv.z, rv.w};
        float x[8];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float2 a = unpack2<F16>(pw[j]), b = unpack2<F16>(rw[j]);
            x[2 * j] = a.x + b.x;
            x[2 * j + 1] = a.y + b.y;
        }
        const float lb = __ldg(lse_part + row);
        float4* acc = (float4*)(o_acc + off);
        float la = -INFINITY;
        float wa = 0.f, wb = 1.f, lnew = lb;
        if (!init) {
            la = lse_acc[row];
            // log(e^la + e^lb), with -inf sides contributing nothing
            const float m = fmaxf(la, lb);
            if (m == -INFINITY) {
                wa = 0.f;
                wb = 0.f;
                lnew = -INFINITY;
            } else {
                const float ea = expf(la - m), eb = expf(lb - m);
                const float s = ea + eb;
                lnew = m + logf(s);
                wa = ea / s;
                wb = eb / s;
            }
        }
        float4 a0 = make_float4(0.f, 0.f, 0.f, 0.f), a1 = a0;
        if (!init && wa != 0.f) {
            a0 = acc[0];
            a1 = acc[1];
        }
        if (lb == -INFINITY) wb = 0.f;   // the part saw no key (its output is 0)
        acc[0] = make_float4(wa * a0.x + wb * x[0], wa * a0.y + wb * x[1], wa * a0.z + wb * x[2], wa * a0.w + wb * x[3]);
        acc[1] = make_float4(wa * a1.x + wb * x[4], wa * a1.y + wb * x[5], wa * a1.z + wb * x[6], wa * a1.w + wb * x[7]);
        // one thread per row writes the merged log-sum-exp, after every thread of the row
        // has read the old one (the row's threads are in one warp: per_row <= 16)
        __syncwarp(__activemask());   // a row's lanes are all active or all done
        if (c == 0) lse_acc[row] = lnew;
    }
}

// o = round16(o_acc), o_res = round16(o_acc - o) (NULL: not written).
template <bool F16>
__global__ void __launch_bounds__(256) o_finalize_kernel(const float4* __restrict__ o_acc, uint2* __restrict__ o,
                                                         uint2* __restrict__ o_res, int64_t n4) {
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n4; i += (int64_t)gridDim.x * blockDim.x) {
        const float4 v = o_acc[i];
        const uint32_t h0 = pack2<F16>(v.x, v.y), h1 = pack2<F16>(v.z, v.w);
        o[i] = make_uint2(h0, h1);
        if (o_res) {
            const float2 a = unpack2<F16>(h0), b = unpack2<F16>(h1);
            o_res[i] = make_uint2(pack2<F16>(v.x - a.x, v.y - a.y), pack2<F16>(v.z - b.x, v.w - b.y));
        }
    }
}

__global__ void __launch_bounds__(256) accumulate_f32_kernel(float4* __restrict__ acc, const float4* __restrict__ part,
                                                             int64_t n4) {
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n4; i += (int64_t)gridDim.x * blockDim.x) {
        const float4 a = acc[i], b = __ldg(part + i);
        acc[i] = make_float4(a.x + b.x, a.y + b.y, a.z + b.z, a.w + b.w);
    }
}

int grid_1d(int64_t n) {
    const int sms = device_sm_count();
    const int64_t cap = (int64_t)(sms > 0 ? sms : 148) * 16;
    int64_t g = (n + 255) / 256;
    return (int)(g < 1 ? 1 : (g > cap ? cap : g));
}

bool a16(const void* p) { return ((uintptr_t)p & 15) == 0; }

}  // namespace
}  // namespace usp

using namespace usp;

extern "C" usp_status usp_lse_merge(float* o_acc, float* lse_acc, const void* o_part, const void* o_part_res,
                                    const float* lse_part, int64_t total_tokens, int heads, int head_dim,
                                    int token_major, usp_dtype dt, int init, void* stream) {
    if (total_tokens < 0 || heads < 1 || (head_dim != 64 && head_dim != 128)) return USP_ERR_INVALID_ARG;
    if (dt != USP_BF16 && dt != USP_FP16) return USP_ERR_INVALID_ARG;
    if (total_tokens == 0) return USP_OK;
    if (!o_acc || !lse_acc || !o_part || !lse_part) return USP_ERR_INVALID_ARG;
    if (!a16(o_acc) || !a16(lse_acc) || !a16(o_part) || !a16(o_part_res) || !a16(lse_part)) return USP_ERR_INVALID_ARG;
    const int64_t n = total_tokens * heads * (head_dim / 8);
    cudaStream_t s = (cudaStream_t)stream;
    if (dt == USP_FP16)
        lse_merge_kernel<true><<<grid_1d(n), 256, 0, s>>>(o_acc, lse_acc, (const uint16_t*)o_part,
                                                          (const uint16_t*)o_part_res, lse_part, total_tokens, heads,
                                                          head_dim, token_major ? 1 : 0, init ? 1 : 0);
    else
        lse_merge_kernel<false><<<grid_1d(n), 256, 0, s>>>(o_acc, lse_acc, (const uint16_t*)o_part,
                                                           (const uint16_t*)o_part_res, lse_part, total_tokens, heads,
                                                           head_dim, token_major ? 1 : 0, init ? 1 : 0);
    return cudaGetLastError() == cudaSuccess ? USP_OK : USP_ERR_CUDA;
}

extern "C" usp_status usp_o_finalize(const float* o_acc, void* o, void* o_res, int64_t elements, usp_dtype dt,
                                     void* stream) {
    if (elements < 0 || elements % 4 != 0) return USP_ERR_INVALID_ARG;
    if (dt != USP_BF16 && dt != USP_FP16) return USP_ERR_INVALID_ARG;
    if (elements == 0) return USP_OK;
    if (!o_acc || !o || !a16(o_acc) || !a16(o) || !a16(o_res)) return USP_ERR_INVALID_ARG;
    const int64_t n4 = elements / 4;
    cudaStream_t s = (cudaStream_t)stream;
    if (dt == USP_FP16)
        o_finalize_kernel<true><<<grid_1d(n4), 256, 0, s>>>((const float4*)o_acc, (uint2*)o, (uint2*)o_res, n4);
    else
        o_finalize_kernel<false><<<grid_1d(n4), 256, 0, s>>>((const float4*)o_acc, (uint2*)o, (uint2*)o_res, n4);
    return cudaGetLastError() == cudaSuccess ? USP_OK : USP_ERR_CUDA;
}

extern "C" usp_status usp_accumulate_f32(float* acc, const float* part, int64_t elements, void* stream) {
    if (elements < 0 || elements % 4 != 0) return USP_ERR_INVALID_ARG;
    if (elements == 0) return USP_OK;
    if (!acc || !part || !a16(acc) || !a16(part)) return USP_ERR_INVALID_ARG;
    const int64_t n4 = elements / 4;
    accumulate_f32_kernel<<<grid_1d(n4), 256, 0, (cudaStream_t)stream>>>((float4*)acc, (const float4*)part, n4);
    return cudaGetLastError() == cudaSuccess ? USP_OK : USP_ERR_CUDA;
}
