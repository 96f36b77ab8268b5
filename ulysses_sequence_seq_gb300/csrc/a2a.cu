// The local halves of Ulysses' all-to-all exchange between real ranks.
//
// Before attention rank r holds its S = T/sp consecutive tokens with all H heads; the
// exchange gives it all T tokens of its H/sp heads (HF Transformers "Ulysses sequence
// parallelism" guide, opening paragraph and layout figure; congresoia365 article, "Cómo
// Funciona Ulysses", steps 3 and 5). A collective that moves equal contiguous blocks
// (all_to_all_single) does that once every rank has laid out what it sends as one block
// per destination:
//
//   pack    out[r][s][j] = in[s][r*Hl + head0 + j]   block r goes to rank r
//
// After the collective, block r' of the receive buffer holds rank r' tokens of this
// rank's heads, so the receive buffer [sp][S][nh][D] is already the token-major
// [T][nh][D] the fused attention kernels read. The way back needs no packing (the
// token-major output's block r' is the tokens of rank r'); the receiver unpacks:
//
//   unpack  out[s][r*Hl + head0 + j] = in[r][s][j]
//
// With fewer key/value heads than ranks (sp % H == 0) every rank needs the one head
// its query heads read, head r*H/sp: pack sends that head to each rank (replication)
// and unpack sums the sp/H replicas' gradients in fp32 (head g: ranks g*rep .. g*rep+rep-1).
// head0 and nh select a chunk of each rank's heads, so that the exchange of one chunk
// can overlap the attention of another.
//
// Rows (head_dim elements) move as 16-byte chunks, one per thread, whole rows per warp.
#include <cuda_runtime.h>

#include <climits>
#include <cstdint>

#include "common.cuh"

namespace usp {
namespace {

struct A2aGeom {
    int64_t S;     // tokens per rank
    int sp, H, Hl, head0, nh, rep, cpr;   // rep > 1: replicated heads (H < sp); cpr: 16-byte chunks per row
};

// index of the in/out rows: packed buffer [sp][S][nh] and the shard [S][H]
__device__ __forceinline__ void a2a_rows(const A2aGeom& g, int64_t i, int64_t& packed_row, int64_t& shard_row,
                                         int& r) {
    const int j = (int)(i % g.nh);
    const int64_t rs = i / g.nh;
    const int64_t s = rs % g.S;
    r = (int)(rs / g.S);
    packed_row = i;
    const int h = g.rep > 1 ? r / g.rep : r * g.Hl + g.head0 + j;
    shard_row = s * g.H + h;
}

__global__ void __launch_bounds__(256) a2a_pack_kernel(const uint4* __restrict__ in, uint4* __restrict__ out,
                                                       const A2aGeom g) {
    const int64_t total = (int64_t)g.sp * g.S * g.nh * g.cpr;
    for (int64_t k = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; k < total; k += (int64_t)gridDim.x * blockDim.x) {
        const int64_t i = k / g.cpr;
        const int c = (int)(k - i * g.cpr);
        int64_t prow, srow;
        int r;
        a2a_rows(g, i, prow, srow, r);
        out[prow * g.cpr + c] = __ldg(in + srow * g.cpr + c);
    }
}

__global__ void __launch_bounds__(256) a2a_unpack_kernel(const uint4* __restrict__ in, uint4* __restrict__ out,
                                                         const A2aGeom g) {
    const int64_t total = (int64_t)g.sp * g.S * g.nh * g.cpr;
    for (int64_t k = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; k < total; k += (int64_t)gridDim.x * blockDim.x) {
        const int64_t i = k / g.cpr;
        const int c = (int)(k - i * g.cpr);
        int64_t prow, srow;
        int r;
        a2a_rows(g, i, prow, srow, r);
        out[srow * g.cpr + c] = __ldg(in + prow * g.cpr + c);
    }
}

// Replicated heads: out[s][h] = sum over its rep replicas (ranks h*rep + i) of in[r][s][0],
// accumulated in fp32 in rank order and rounded once (bf16) or kept (fp32).
template <bool kBf16>
__global__ void __launch_bounds__(256) a2a_unpack_sum_kernel(const uint4* __restrict__ in, uint4* __restrict__ out,
                                                             const A2aGeom g) {
    const int64_t total = g.S * g.H * g.cpr;
    for (int64_t k = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; k < total; k += (int64_t)gridDim.x * blockDim.x) {
        const int64_t row = k / g.cpr;   // shard row s * H + h
        const int c = (int)(k - row * g.cpr);
        const int h = (int)(row % g.H);
        const int64_t s = row / g.H;
        float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        for (int i = 0; i < g.rep; ++i) {
            const int r = h * g.rep + i;
            const uint4 v = __ldg(in + ((int64_t)r * g.S + s) * g.cpr + c);
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
            if (kBf16) {
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    acc[2 * q] += __uint_as_float(w[q] << 16);
                    acc[2 * q + 1] += __uint_as_float(w[q] & 0xffff0000u);
                }
            } else {
#pragma unroll
                for (int q = 0; q < 4; ++q) acc[q] += __uint_as_float(w[q]);
            }
        }
        uint4 o;
        if (kBf16) {
            uint32_t w[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                uint32_t pr;
                asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(pr) : "f"(acc[2 * q + 1]), "f"(acc[2 * q]));
                w[q] = pr;
            }
            o = make_uint4(w[0], w[1], w[2], w[3]);
        } else {
            o = make_uint4(__float_as_uint(acc[0]), __float_as_uint(acc[1]), __float_as_uint(acc[2]),
                           __float_as_uint(acc[3]));
        }
        out[k] = o;
    }
}

usp_status a2a_geometry(int sp, int64_t S, int heads, int head_dim, int head0, int nheads, usp_dtype dt,
                        A2aGeom* g) {
    if (sp < 1 || S < 0 || heads < 1 || head_dim < 1) return USP_ERR_INVALID_ARG;
    size_t esize;
    switch (dt) {
        case USP_BF16:
        case USP_FP16: esize = 2; break;
        case USP_FP32: esize = 4; break;
        default: return USP_ERR_INVALID_ARG;
    }
    g->S = S;
    g->sp = sp;
    g->H = heads;
    if (heads % sp == 0) {
        g->Hl = heads / sp;
        g->rep = 1;
        if (head0 < 0 || nheads < 1 || head0 + nheads > g->Hl) return USP_ERR_INVALID_ARG;
    } else if (sp % heads == 0) {
        g->Hl = 1;
        g->rep = sp / heads;
        if (head0 != 0 || nheads != 1) return USP_ERR_INVALID_ARG;
    } else {
        return USP_ERR_INVALID_ARG;   // heads must divide over sp_size or divide it
    }
    g->head0 = head0;
    g->nh = nheads;
    const size_t row = esize * (size_t)head_dim;
    if (row % 16 != 0) return USP_ERR_UNSUPPORTED;
    g->cpr = (int)(row / 16);
    return USP_OK;
}

int a2a_grid(int64_t chunks) {
    const int sms = device_sm_count();
    const int64_t cap = (int64_t)(sms > 0 ? sms : 148) * 16;
    int64_t g = (chunks + 255) / 256;
    if (g > cap) g = cap;
    return (int)(g < 1 ? 1 : g);
}

bool overlap(const void* a, size_t an, const void* b, size_t bn) {
    const uintptr_t x = (uintptr_t)a, y = (uintptr_t)b;
    return an > 0 && bn > 0 && x < y + bn && y < x + an;
}

}  // namespace
}  // namespace usp

using namespace usp;

extern "C" usp_status usp_a2a_pack(const void* in, void* out, int sp, int64_t shard_tokens, int heads, int head_dim,
                                   int head0, int nheads, usp_dtype dt, void* stream) {
    A2aGeom g{};
    const usp_status st = a2a_geometry(sp, shard_tokens, heads, head_dim, head0, nheads, dt, &g);
    if (st != USP_OK) return st;
    if (shard_tokens == 0) return USP_OK;
    if (!in || !out || ((uintptr_t)in & 15) || ((uintptr_t)out & 15)) return USP_ERR_INVALID_ARG;
    const size_t row = (size_t)g.cpr * 16;
    if (overlap(in, row * (size_t)heads * (size_t)shard_tokens, out, row * (size_t)sp * (size_t)shard_tokens * nheads))
        return USP_ERR_INVALID_ARG;
    const int64_t chunks = (int64_t)sp * shard_tokens * nheads * g.cpr;
    a2a_pack_kernel<<<a2a_grid(chunks), 256, 0, (cudaStream_t)stream>>>((const uint4*)in, (uint4*)out, g);
    return cudaGetLastError() == cudaSuccess ? USP_OK : USP_ERR_CUDA;
}

extern "C" usp_status usp_a2a_unpack(const void* in, void* out, int sp, int64_t shard_tokens, int heads,
                                     int head_dim, int head0, int nheads, usp_dtype dt, void* stream) {
    A2aGeom g{};
    const usp_status st = a2a_geometry(sp, shard_tokens, heads, head_dim, head0, nheads, dt, &g);
    if (st != USP_OK) return st;
    if (g.rep > 1 && dt == USP_FP16) return USP_ERR_UNSUPPORTED;   // replica sums: bf16 or fp32
    if (shard_tokens == 0) return USP_OK;
    if (!in || !out || ((uintptr_t)in & 15) || ((uintptr_t)out & 15)) return USP_ERR_INVALID_ARG;
    const size_t row = (size_t)g.cpr * 16;
    if (overlap(in, row * (size_t)sp * (size_t)shard_tokens * nheads, out, row * (size_t)heads * (size_t)shard_tokens))
        return USP_ERR_INVALID_ARG;
    cudaStream_t s = (cudaStream_t)stream;
    if (g.rep > 1) {
        const int64_t chunks = shard_tokens * heads * g.cpr;
        if (dt == USP_BF16)
            a2a_unpack_sum_kernel<true><<<a2a_grid(chunks), 256, 0, s>>>((const uint4*)in, (uint4*)out, g);
        else
            a2a_unpack_sum_kernel<false><<<a2a_grid(chunks), 256, 0, s>>>((const uint4*)in, (uint4*)out, g);
    } else {
        const int64_t chunks = (int64_t)sp * shard_tokens * nheads * g.cpr;
        a2a_unpack_kernel<<<a2a_grid(chunks), 256, 0, s>>>((const uint4*)in, (uint4*)out, g);
    }
    return cudaGetLastError() == cudaSuccess ? USP_OK : USP_ERR_CUDA;
}
