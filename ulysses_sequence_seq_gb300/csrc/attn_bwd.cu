// Backward of the local attention step on sm_103a: dQ, dK, dV of causal,
// sample-boundary-masked softmax attention from the saved logsumexp.
//
//   P_ij  = exp(s_ij - lse_i)           dP_ij = dO_i . v_j        Delta_i = dO_i . O_i
//   dS_ij = scale * P_ij (dP_ij - Delta_i)
//   dV_j  = sum_i P_ij dO_i     dK_j = sum_i dS_ij q_i     dQ_i = sum_j dS_ij k_j
//
// One CTA owns a 128-row key/value tile of one sample and one key/value head and
// walks every query block that sees it (from the diagonal on when causal), for all
// query heads of its GQA group, so dK and dV accumulate in tensor memory and are
// written once. dQ partial tiles are added into an fp32 accumulator by TMA bulk
// reductions. Everything is computed transposed (key rows on TMEM lanes) so that P^T
// feeds the dV MMA straight from TMEM.
//
// Each query block is processed as two independent halves of 64 query columns: S, dP,
// dV and dK are issued per half, so the tensor cores run one half's MMAs while the
// warps of the other half compute P or dS. Only dQ waits for both halves.
//
// Warp roles (448 threads):
//   warps 0-3  compute half A: thread = key row, query columns 0-63 of the block
//   warps 4-7  compute half B: thread = key row, query columns 64-127
//              (at the end half A writes dV and half B writes dK)
//   warps 8-11 dQ group: thread = query row; moves each dQ tile from TMEM into its own
//              128-byte-swizzled staging buffers and adds it to the accumulator with
//              bulk tensor reductions (whole 128-byte lines, no per-thread atomics)
//   warp  12   TMA producer: K, V once, then Q blocks into a 2-stage ring, dO blocks
//              into one buffer (dO is consumed early in a step)
//   warp  13   MMA issuer and TMEM owner
// Tensor memory: [0,128) holds S^T, then bf16 P^T, then dP^T: half A in [0,64) and half
// B in [64,128), each with its bf16 P^T at the start of its range; dQ [128,256); dV
// [256,256+D); dK [384,384+D). dS lives only in shared memory, where dK reads it K-major
// and dQ MN-major.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>

#include "attn.cuh"
#include "common.cuh"
#include "ptx.cuh"
#include "tiles.cuh"

namespace usp {
namespace {

using namespace ptx;

constexpr int kHalfCols = kBlockN / 2;           // query columns per half
constexpr int kComputeWarps = 8;                 // two warpgroups, one per half
constexpr int kDqWarp0 = kComputeWarps;          // 4 warps
constexpr int kProducerWarp = kComputeWarps + 4;
constexpr int kMmaWarp = kComputeWarps + 5;
constexpr int kBwdThreads = 32 * (kComputeWarps + 6);
constexpr int kDqChunkBytes = 32 * 32 * 4;       // one warp's 32 query rows x 32 fp32 columns

template <int D>
struct BwdSmem {
    static constexpr int kPanels = D / 64;
    static constexpr int kTileBytes = kTileM * D * 2;
    static constexpr int kK = 0;
    static constexpr int kV = kTileBytes;
    static constexpr int kQ = 2 * kTileBytes;        // + stage * kTileBytes
    static constexpr int kDO = 4 * kTileBytes;
    static constexpr int kDS = 5 * kTileBytes;       // [128 key rows][128 query cols] bf16, two 64-col panels
    static constexpr int kStage = kDS + kTileM * kBlockN * 2;   // dQ staging: one chunk per warp
    static constexpr int kLse = kStage + 4 * kDqChunkBytes;     // fp32[2][64]: -lse (log2 units), one half each
    static constexpr int kDelta = kLse + 512;                   // fp32[2][64]: -Delta
    static constexpr int kBars = kDelta + 512;
    // bKvEmpty: the item's last MMA has run (K and V free, dK and dV final); bItem: 4-slot ring
    static constexpr int bKvFull = 0, bQFull = 1, bQEmpty = 3, bDoFull = 5, bDoEmpty = 6, bSFull = 7, bPFull = 9,
                         bDpFull = 11, bDsFull = 13, bDqFull = 15, bDqEmpty = 16, bDrain = 17, bKvEmpty = 18,
                         bAccEmpty = 19, bItem = 20, kNumBars = 24;
    static constexpr int kItemRing = kBars + 8 * kNumBars;        // int[4]: work item of each slot
    static constexpr int kTmemSlot = kItemRing + 16;
    static constexpr int kAbort = kTmemSlot + 8;
    static constexpr int kBytes = kAbort + 8;
    static constexpr int kAlloc = kBytes + 1024;
};
static_assert(BwdSmem<128>::kAlloc <= 232448, "backward shared memory exceeds the per-CTA limit");
static_assert(BwdSmem<128>::kStage % 1024 == 0, "dQ staging must keep the 128-byte swizzle atoms aligned");

// Optional clock64 timeline of the first kTlSteps steps of every CTA (compile with
// -DUSP_TIMELINE; the default build has none of it). Events: MMA thread 0-4 (both halves'
// P ready, both halves' dS ready, dQ issued), compute half h 5+5h..8+5h (S ready, P
// stored, dP ready, dS stored), dQ drain 14-15 (dQ ready, TMEM released), MMA thread 16
// (dO arrived), producer 17-18 (dO load issued, Q load issued). Read back with
// usp_debug_timeline.
#ifdef USP_TIMELINE
constexpr int kTlSteps = 48, kTlEvents = 20, kTlCtas = 160;
static __device__ long long g_timeline[kTlCtas][kTlSteps][kTlEvents];
#define USP_TL(step, ev)                                                                        \
    do {                                                                                        \
        if ((step) < kTlSteps && blockIdx.x < kTlCtas) g_timeline[blockIdx.x][(step)][(ev)] = clock64(); \
    } while (0)
#else
#define USP_TL(step, ev) \
    do {                 \
    } while (0)
#endif

// One backward work item: a key/value tile of one sample and one key/value head, and the
// query blocks (of every query head of its GQA group) that see it.
struct BwdItem {
    int g, s, e, kv0, i0, nq, nsteps;
    // first row of the query block of step k: query head g * group + k / nq, blocks walked
    // from the sample's last one down to the diagonal, so CTAs that start together share
    // their query blocks
    __device__ __forceinline__ int q0(int k) const { return s + (i0 + nq - 1 - k % nq) * kTileM; }
};
__device__ __forceinline__ BwdItem bwd_item(const BwdArgs& a, int idx) {
    const WorkItem it = a.items[idx];
    BwdItem b;
    b.g = it.head;
    b.s = a.cu[it.seq];
    b.e = a.cu[it.seq + 1];
    b.kv0 = b.s + it.tile * kBlockN;
    b.i0 = first_query_block_for_kv_block(it.tile, a.causal);
    b.nq = query_blocks_in_sample(b.s, b.e) - b.i0;
    b.nsteps = b.nq * a.group;
    return b;
}

// Scale factors of one key/value group's fp16 operands (see BwdArgs): the products run on
// q' = q 2^eq, k' = k 2^ek, v' = v 2^ev, dO' = dO 2^edo, and dS is rounded as dS 2^(ev+edo+ds_exp).
struct GroupScale {
    float sl2;      // scale * log2(e) * 2^-(eq+ek): turns the scaled S' into log2 units
    float sc;       // scale * 2^ds_exp: the factor of dS
    float dsc;      // 2^(ev+edo) * sc: Delta on the scale of dP', times the factor of dS
    float dv_un;    // 2^-edo: dV' -> dV
    float dk_un;    // 2^-(ev+edo+ds_exp+eq): dK' -> dK
    float dq_un;    // 2^-(ev+edo+ds_exp+ek): dQ' -> dQ
};
__device__ __forceinline__ GroupScale group_scale(const BwdArgs& a, int g) {
    const int eq = range_exponent(__ldg(a.amax + kAmaxQ * a.hkv + g));
    const int ek = range_exponent(__ldg(a.amax + kAmaxK * a.hkv + g));
    const int ev = range_exponent(__ldg(a.amax + kAmaxV * a.hkv + g));
    const int edo = range_exponent(__ldg(a.amax + kAmaxDO * a.hkv + g));
    GroupScale r;
    r.sl2 = a.scale_log2 * exp2i(-(eq + ek));
    r.sc = a.scale * exp2i(a.ds_exp);
    r.dsc = exp2i(ev + edo) * r.sc;
    r.dv_un = exp2i(-edo);
    r.dk_un = exp2i(-(ev + edo + a.ds_exp + eq));
    r.dq_un = exp2i(-(ev + edo + a.ds_exp + ek));
    return r;
}

// The CTA's j-th work item, published by the producer in a 4-slot ring; false when the
// wait gave up (abort). No role runs more than two items behind the producer, so a
// slot is never rewritten while a reader still needs it.
__device__ __forceinline__ bool read_item(uint64_t* item_bars, volatile int* ring, int j, volatile int* abort_flag,
                                          int& idx) {
    if (!mbar_wait(&item_bars[j & 3], (j >> 2) & 1, abort_flag, kWaitLimitNs)) return false;
    idx = ring[j & 3];
    return true;
}

// 448 threads = 14 warps, one CTA per SM; two of the four SM sub-partitions hold four
// warps, so 16384 registers per sub-partition cap a thread at 128.
template <int D, bool F16>
__global__ void __launch_bounds__(kBwdThreads, 1)
    attn_bwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDO,
                    const __grid_constant__ CUtensorMap tmDQ, const __grid_constant__ CUtensorMap tmDK,
                    const __grid_constant__ CUtensorMap tmDV, const BwdArgs a) {
    using L = BwdSmem<D>;
    pdl_wait();   // the work list, Delta and the zeroed dQ accumulator come from the kernels before
    const int count = a.hdr->bwd_count;
    if ((int)blockIdx.x >= count) return;
    // once any CTA of this launch has timed out, the rest skip their work
    if (*(volatile int*)&a.hdr->status != (int)USP_OK) return;
    const int G = a.group;

    extern __shared__ uint8_t smem_raw[];
    // 1024-byte aligned base for the 128-byte swizzle atoms, derived from smem_raw by an
    // offset so the compiler keeps it in the shared window (LDS/STS, not generic accesses)
    uint8_t* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint64_t* bars = (uint64_t*)(sm + L::kBars);
    uint32_t* tmem_slot = (uint32_t*)(sm + L::kTmemSlot);
    volatile int* abort_flag = (volatile int*)(sm + L::kAbort);
    float* lse_s = (float*)(sm + L::kLse);
    float* delta_s = (float*)(sm + L::kDelta);
    volatile int* item_ring = (volatile int*)(sm + L::kItemRing);

    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x % 32;

    if (warp == kMmaWarp) {
        tmem_alloc(tmem_slot, 512);
        tmem_relinquish();
    }
    if (threadIdx.x == 0) {
        mbar_init(&bars[L::bKvFull], 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bars[L::bQFull + i], 1);
            mbar_init(&bars[L::bQEmpty + i], 1);   // released by the dQ group (see there)
            mbar_init(&bars[L::bSFull + i], 1);
            mbar_init(&bars[L::bPFull + i], 4);
            mbar_init(&bars[L::bDpFull + i], 1);
            mbar_init(&bars[L::bDsFull + i], 4);
        }
        mbar_init(&bars[L::bDoFull], 1);
        mbar_init(&bars[L::bDoEmpty], 1);   // released by compute half B (see there)
        mbar_init(&bars[L::bDqFull], 1);
        mbar_init(&bars[L::bDqEmpty], 4);
        mbar_init(&bars[L::bDrain], 1);
        mbar_init(&bars[L::bKvEmpty], 1);
        mbar_init(&bars[L::bAccEmpty], kComputeWarps);
        for (int i = 0; i < 4; ++i) mbar_init(&bars[L::bItem + i], 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = *tmem_slot;

    // Persistent CTAs: each one takes work items in the scheduler's order (heaviest first),
    // its first one by its index and the rest from a counter, until the list is done. Every
    // per-step barrier phase follows the CTA's running step count `gk` across items; the
    // per-item ones (K/V, dK/dV accumulators) follow the item count `j`.
    uint64_t* item_bars = &bars[L::bItem];
    if (warp == kProducerWarp) {
        // ------------------------------------------------------------------ TMA producer
        if (lane == 0) {
            prefetch_tmap(&tmQ);
            prefetch_tmap(&tmK);
            prefetch_tmap(&tmV);
            prefetch_tmap(&tmDO);
            bool ok = true;
            int gk = 0, q_total = 0, do_total = 0, kv_total = 0;
            int next_idx = (int)blockIdx.x;
            for (int j = 0; ok && next_idx >= 0; ++j) {
                const int idx = next_idx;
                next_idx = -1;
                item_ring[j & 3] = idx;
                mbar_arrive(&item_bars[j & 3]);   // release: the slot write is visible to its readers
                if (idx >= count) break;
                const BwdItem w = bwd_item(a, idx);
                for (int k = 0; k < w.nsteps; ++k, ++gk) {
                    const int st = gk & 1;
                    const int h = w.g * G + k / w.nq;
                    const int q0 = w.q0(k);
                    if (gk >= 2 && !mbar_wait(&bars[L::bQEmpty + st], ((gk >> 1) - 1) & 1, abort_flag, kWaitLimitNs)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&bars[L::bQFull + st], L::kTileBytes);
                    USP_TL(gk, 18);
                    for (int p = 0; p < L::kPanels; ++p)
                        tma_load_rows(sm + L::kQ + st * L::kTileBytes + p * (kTileM * 128), &tmQ,
                                      &bars[L::bQFull + st], p * 64, q0, h, 0);
                    ++q_total;
                    // the single dO buffer is free once both halves' dV and dP of the previous block are done
                    if (gk >= 1 && !mbar_wait(&bars[L::bDoEmpty], (gk - 1) & 1, abort_flag, kWaitLimitNs)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&bars[L::bDoFull], L::kTileBytes);
                    USP_TL(gk, 17);
                    for (int p = 0; p < L::kPanels; ++p)
                        tma_load_rows(sm + L::kDO + p * (kTileM * 128), &tmDO, &bars[L::bDoFull], p * 64, q0, h, 0);
                    ++do_total;
                    // The CTAs walk the same query blocks in near lockstep, so a block's first
                    // load goes to DRAM for all of them; pull Q and dO two steps ahead into L2
                    // (the next item's first two steps are pulled when it is reserved, below).
                    if (k + 2 < w.nsteps) {
                        const int k2 = k + 2, h2 = w.g * G + k2 / w.nq, q2 = w.q0(k2);
                        for (int p = 0; p < L::kPanels; ++p) {
                            tma_prefetch_rows(&tmQ, p * 64, q2, h2, 0);
                            tma_prefetch_rows(&tmDO, p * 64, q2, h2, 0);
                        }
                    }
                    if (k == 0) {  // K, V once the previous item's last MMA has read them
                        if (j > 0 && !mbar_wait(&bars[L::bKvEmpty], (j - 1) & 1, abort_flag, kWaitLimitNs)) {
                            ok = false;
                            break;
                        }
                        mbar_arrive_expect_tx(&bars[L::bKvFull], 2 * L::kTileBytes);
                        for (int p = 0; p < L::kPanels; ++p) {
                            tma_load_rows(sm + L::kK + p * (kTileM * 128), &tmK, &bars[L::bKvFull], p * 64, w.kv0,
                                          w.g, 0);
                            tma_load_rows(sm + L::kV + p * (kTileM * 128), &tmV, &bars[L::bKvFull], p * 64, w.kv0,
                                          w.g, 0);
                        }
                        ++kv_total;
                    }
                    // two blocks before the end, reserve the next item and pull its K and V
                    // into L2, so that its start does not wait on DRAM
                    if (k == (w.nsteps >= 2 ? w.nsteps - 2 : 0)) {
                        next_idx = (int)gridDim.x + atomicAdd(&a.hdr->bwd_next, 1);
                        if (next_idx < count) {
                            const BwdItem nw = bwd_item(a, next_idx);
                            for (int p = 0; p < L::kPanels; ++p) {
                                tma_prefetch_rows(&tmK, p * 64, nw.kv0, nw.g, 0);
                                tma_prefetch_rows(&tmV, p * 64, nw.kv0, nw.g, 0);
                                for (int k2 = 0; k2 < 2 && k2 < nw.nsteps; ++k2) {
                                    tma_prefetch_rows(&tmQ, p * 64, nw.q0(k2), nw.g * G + k2 / nw.nq, 0);
                                    tma_prefetch_rows(&tmDO, p * 64, nw.q0(k2), nw.g * G + k2 / nw.nq, 0);
                                }
                            }
                        }
                    }
                }
            }
            // let every copy in flight land before the CTA can exit
            if (kv_total > 0) mbar_wait_drain(&bars[L::bKvFull], (kv_total - 1) & 1, kDrainLimitNs);
            for (int q = q_total - 2 < 0 ? 0 : q_total - 2; q < q_total; ++q)
                mbar_wait_drain(&bars[L::bQFull + (q & 1)], (q >> 1) & 1, kDrainLimitNs);
            if (do_total > 0) mbar_wait_drain(&bars[L::bDoFull], (do_total - 1) & 1, kDrainLimitNs);
        }
    } else if (warp == kMmaWarp) {
        // ------------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idH = idesc_16b_f32(kBlockN, kHalfCols, false, false, F16);  // S^T, dP^T of one half
            constexpr uint32_t idDv = idesc_16b_f32(kBlockN, D, false, true, F16);         // dV (A in TMEM)
            constexpr uint32_t idDk = idesc_16b_f32(kBlockN, D, false, true, F16);         // dK (A = dS, K-major)
            constexpr uint32_t idDq = idesc_16b_f32(kTileM, D, true, true, F16);           // dQ (A, B MN-major)
            // 64-bit shared-memory descriptors are built once; a K step or a row offset only
            // adds a constant to the start-address field (addresses stay below 2^18, so the
            // field never carries).
            constexpr uint32_t kPanel = kTileM * 128;  // bytes of one 64-column panel of a tile
            const uint32_t sK = smem_u32(sm + L::kK), sV = smem_u32(sm + L::kV);
            const uint32_t sQ = smem_u32(sm + L::kQ), sDO = smem_u32(sm + L::kDO), sDS = smem_u32(sm + L::kDS);
            const uint64_t dK_kmaj = sdesc_sw128(sK, 0, 1024), dK_mn = sdesc_sw128(sK, kPanel, 1024);
            const uint64_t dV_kmaj = sdesc_sw128(sV, 0, 1024);
            const uint64_t dQ_kmaj = sdesc_sw128(sQ, 0, 1024), dQ_mn = sdesc_sw128(sQ, kPanel, 1024);
            const uint64_t dDO_kmaj = sdesc_sw128(sDO, 0, 1024), dDO_mn = sdesc_sw128(sDO, kPanel, 1024);
            const uint64_t dDS_kmaj = sdesc_sw128(sDS, 0, 1024), dDS_mn = sdesc_sw128(sDS, kBlockN * 128, 1024);
            constexpr uint64_t kStageQ = (uint64_t)(L::kTileBytes >> 4);
            constexpr uint64_t kHalfRows = (uint64_t)((kHalfCols * 128) >> 4);   // 64 rows of a K-major tile
            const uint32_t tS = tbase, tDQ = tbase + 128, tDV = tbase + 256, tDK = tbase + 384;
            // d[128 x 64] = A . B^T over K = D, both operands K-major (S^T and dP^T of one half)
            auto issue_half = [&](uint32_t d, uint64_t a_desc, uint64_t b_desc) {
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint64_t off = (uint64_t)((((kk / 4) * kPanel) + (kk % 4) * 32) >> 4);
                    mma_ss(d, a_desc + off, b_desc + off, idH, kk > 0);
                }
            };
            bool ok = true;
            int gk = 0;
            for (int j = 0; ok; ++j) {
                int idx;
                if (!read_item(item_bars, item_ring, j, abort_flag, idx)) break;
                if (idx >= count) break;
                const int nsteps = bwd_item(a, idx).nsteps;
                if (!mbar_wait2(&bars[L::bKvFull], j & 1, &bars[L::bQFull + (gk & 1)], (gk >> 1) & 1, abort_flag,
                                kWaitLimitNs))
                    break;
                tc_fence_after();
                for (int hf = 0; hf < 2; ++hf) {
                    issue_half(tS + hf * kHalfCols, dK_kmaj, dQ_kmaj + (gk & 1) * kStageQ + hf * kHalfRows);
                    mma_commit(&bars[L::bSFull + hf]);
                }
                // the epilogue of the previous item must have read dK and dV out of TMEM
                if (j > 0 && !mbar_wait(&bars[L::bAccEmpty], (j - 1) & 1, abort_flag, kWaitLimitNs)) break;
                // Per step k and half hf: dV += P^T.dO, dP^T = V.dO^T (after P), then S^T of the
                // next block and dK += dS^T.Q (after dS); dQ = dS.K once both halves wrote dS. The
                // tensor cores run in issue order, so the commit that releases a half's dP^T also
                // covers the previous block's dQ and dK reads of the dS buffer that half rewrites.
                // The issue queue of the tensor pipe is about one MMA deep, so each wait between
                // two batches leaves the pipe idle for its latency, and so does a commit right
                // behind another (it holds this thread until the first is delivered): per step
                // there are four gaps, each waiting on what its batch needs, two barriers at
                // once where possible, and the dO and Q buffers are released by the warps that
                // see their last readers complete instead of by commits.
                for (int k = 0; ok && k < nsteps; ++k, ++gk) {
                    const int st = gk & 1;
                    const bool next = k + 1 < nsteps;
                    // gap 1: this step's dO and half A's P^T
                    if (!mbar_wait2(&bars[L::bDoFull], gk & 1, &bars[L::bPFull + 0], gk & 1, abort_flag,
                                    kWaitLimitNs)) {
                        ok = false;
                        break;
                    }
                    USP_TL(gk, 16);
                    for (int hf = 0; ok && hf < 2; ++hf) {
                        // gap 2 (half B): its P^T
                        if (hf == 1 && !mbar_wait(&bars[L::bPFull + 1], gk & 1, abort_flag, kWaitLimitNs)) {
                            ok = false;
                            break;
                        }
                        USP_TL(gk, hf);
                        tc_fence_after();
#pragma unroll
                        for (int kk = 0; kk < kHalfCols / 16; ++kk)  // dV += P^T . dO over this half's queries
                            mma_ts(tDV, tS + hf * kHalfCols + 8 * kk,
                                   dDO_mn + (uint64_t)((((hf * kHalfCols) / 16 + kk) * 2048) >> 4), idDv,
                                   (k > 0 || hf > 0 || kk > 0) ? 1u : 0u);
                        issue_half(tS + hf * kHalfCols, dV_kmaj, dDO_kmaj + hf * kHalfRows);  // dP^T, after dV read P^T
                        mma_commit(&bars[L::bDpFull + hf]);
                    }
                    if (!ok) break;
                    for (int hf = 0; ok && hf < 2; ++hf) {
                        // gap 3 (half A): its dS and, for the next S^T, the next block's Q;
                        // gap 4 (half B): its dS and the dQ accumulator's tensor memory
                        uint64_t* other = nullptr;
                        uint32_t other_par = 0;
                        if (hf == 0 && next) {
                            other = &bars[L::bQFull + (st ^ 1)];
                            other_par = ((gk + 1) >> 1) & 1;
                        } else if (hf == 1 && gk > 0) {
                            other = &bars[L::bDqEmpty];
                            other_par = (gk - 1) & 1;
                        }
                        const bool got = other ? mbar_wait2(&bars[L::bDsFull + hf], gk & 1, other, other_par, abort_flag,
                                                            kWaitLimitNs)
                                               : mbar_wait(&bars[L::bDsFull + hf], gk & 1, abort_flag, kWaitLimitNs);
                        if (!got) {
                            ok = false;
                            break;
                        }
                        USP_TL(gk, 2 + hf);
                        tc_fence_after();
                        if (next) {  // S^T of the next block first: it heads this half's next step
                            issue_half(tS + hf * kHalfCols, dK_kmaj, dQ_kmaj + (st ^ 1) * kStageQ + hf * kHalfRows);
                            mma_commit(&bars[L::bSFull + hf]);
                        }
#pragma unroll
                        for (int kk = 0; kk < kHalfCols / 16; ++kk)  // dK += dS^T . Q over this half's queries
                            mma_ss(tDK, dDS_kmaj + (uint64_t)((hf * kBlockN * 128 + kk * 32) >> 4),
                                   dQ_mn + st * kStageQ + (uint64_t)((((hf * kHalfCols) / 16 + kk) * 2048) >> 4),
                                   idDk, (k > 0 || hf > 0 || kk > 0) ? 1u : 0u);
                    }
                    if (!ok) break;
#pragma unroll
                    for (int kk = 0; kk < kBlockN / 16; ++kk)  // dQ = dS . K
                        mma_ss(tDQ, dDS_mn + (uint64_t)((kk * 2048) >> 4), dK_mn + (uint64_t)((kk * 2048) >> 4), idDq,
                               kk > 0 ? 1u : 0u);
                    mma_commit(&bars[L::bDqFull]);
                    USP_TL(gk, 4);
                }
                if (!ok) break;
                mma_commit(&bars[L::bKvEmpty]);   // K and V read for the last time; dK and dV final
            }
            mma_commit(&bars[L::bDrain]);
            mbar_wait_drain(&bars[L::bDrain], 0, kDrainLimitNs);
        }
    } else if (warp < kComputeWarps) {
        // ------------------------------------------------------------------ compute halves (key rows)
        const int grp = warp >> 2;          // query columns [grp * kHalfCols, (grp + 1) * kHalfCols)
        const int r = (warp & 3) * 32 + lane;
        const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
        // this half's columns of the S^T / P^T / dP^T region
        const uint32_t tS = tbase + lane_off + grp * kHalfCols;
        float* lse_g = lse_s + grp * kHalfCols;
        float* delta_g = delta_s + grp * kHalfCols;
        bool ok = true;
        int gk = 0;
        // This half's query rows of a step, negated: -lse (log2 units) and -Delta; rows outside
        // the sample get -lse = -inf, which makes their P exactly zero. Loaded one step ahead
        // (the first step of the next item before this item's epilogue), so that their
        // global-memory latency stays off the critical path.
        float nl_next = -INFINITY, nd_next = 0.f;
        auto fetch_row_stats = [&](const BwdItem& it, int k, float dsc) {
            const int h = it.g * G + k / it.nq;
            const int q = it.q0(k) + grp * kHalfCols + r;
            const bool q_ok = r < kHalfCols && q < it.e;
            nl_next = q_ok ? -__ldg(a.lse + (int64_t)h * a.T + q) * 1.4426950408889634f : -INFINITY;
            nd_next = q_ok ? -__ldg(a.delta + (int64_t)h * a.T + q) * dsc : 0.f;   // -Delta' * sc
        };
        // The half's four warps leave their loops together: a warp that gave up on a bounded
        // wait skips ahead to the next vote (group_any) instead of leaving at once, so that no
        // warp is left waiting at one of the half's barriers for warps that have gone.
        int idx = count;
        if (!read_item(item_bars, item_ring, 0, abort_flag, idx)) ok = false;
        ok = !group_any(1 + grp, 128, !ok);
        if (ok && idx < count) {
            const BwdItem w0 = bwd_item(a, idx);
            fetch_row_stats(w0, 0, group_scale(a, w0.g).dsc);
        }
        for (int j = 0; ok && idx < count; ++j) {
            const BwdItem w = bwd_item(a, idx);
            float sl2, sc, dsc;
            {
                const GroupScale gs = group_scale(a, w.g);
                sl2 = gs.sl2;
                sc = gs.sc;
                dsc = gs.dsc;
            }
            const int kv = w.kv0 + r;
            const bool kv_ok = kv < w.e;
            for (int k = 0; k < w.nsteps; ++k, ++gk) {
                const int q0 = w.q0(k);
                if (group_any(1 + grp, 128, !ok)) {   // also: the previous step's reads of the row stats are done
                    ok = false;
                    break;
                }
                if (r < kHalfCols) {
                    lse_g[r] = nl_next;
                    delta_g[r] = nd_next;
                }
                named_bar_sync(1 + grp, 128);
                if (k + 1 < w.nsteps) fetch_row_stats(w, k + 1, dsc);
                // element masks are only needed on the diagonal block and on the sample's ragged
                // last key tile; there query column c (of 128) is visible to key row r iff c >= r
                const bool mask_blk = (a.causal && q0 == w.kv0) || (w.kv0 + kBlockN > w.e);
                const int vis_from = (a.causal && q0 == w.kv0) ? r - grp * kHalfCols : -1;
                // the warp agrees on every wait's outcome: its tcgen05 loads and stores are collective
                if (!__all_sync(0xffffffffu, mbar_wait(&bars[L::bSFull + grp], gk & 1, abort_flag, kWaitLimitNs))) {
                    ok = false;
                    continue;
                }
                if ((warp & 3) == 0 && lane == 0) USP_TL(gk, 5 + 5 * grp);
                tc_fence_after();
                // P for this row's query columns as packed bf16 pairs: the values the dV MMA
                // consumes, kept (half the registers of fp32) for dS
                uint32_t pkall[kHalfCols / 2];
                static_assert(kHalfCols == 64, "the P pass loads the half's two 32-column chunks at once");
                {
                    uint32_t sr[2][32];
                    tmem_ld32(tS, sr[0]);
                    tmem_ld32(tS + 32, sr[1]);
                    tmem_ld_wait(sr[0]);
                    reg_fence(sr[1]);
#pragma unroll
                    for (int c = 0; c < 2; ++c) {
#pragma unroll
                        for (int jj = 0; jj < 16; ++jj) {
                            const int c0 = 32 * c + 2 * jj;
                            const float2 nl = *(const float2*)(lse_g + c0);
                            const float2 x = fma2(make_float2(__uint_as_float(sr[c][2 * jj]), __uint_as_float(sr[c][2 * jj + 1])),
                                                  make_float2(sl2, sl2), nl);
                            float2 pp = make_float2(ex2_approx(x.x), ex2_approx(x.y));
                            if (mask_blk) {
                                if (!kv_ok || c0 < vis_from) pp.x = 0.f;
                                if (!kv_ok || c0 + 1 < vis_from) pp.y = 0.f;
                            }
                            pkall[16 * c + jj] = pack2<F16>(pp.x, pp.y);
                        }
                        uint32_t pk[16];
#pragma unroll
                        for (int jj = 0; jj < 16; ++jj) pk[jj] = pkall[16 * c + jj];
                        tmem_st16(tS + 16 * c, pk);
                    }
                }
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars[L::bPFull + grp]);
                if ((warp & 3) == 0 && lane == 0) USP_TL(gk, 6 + 5 * grp);

                // dP^T of this half; its commit also covers the previous block's reads of the dS buffer
                if (!__all_sync(0xffffffffu, mbar_wait(&bars[L::bDpFull + grp], gk & 1, abort_flag, kWaitLimitNs))) {
                    ok = false;
                    continue;
                }
                if ((warp & 3) == 0 && lane == 0) USP_TL(gk, 7 + 5 * grp);
                // half B's dP^T is the step's last MMA reading dO (they run in issue order): the
                // dO buffer is free for the next block
                if (grp == 1 && r == 0) mbar_arrive(&bars[L::bDoEmpty]);
                tc_fence_after();
                uint8_t* panel = sm + L::kDS + grp * (kBlockN * 128);
#pragma unroll
                for (int c = 0; c < kHalfCols / 32; ++c) {
                    uint32_t dr[32];
                    tmem_ld32(tS + 32 * c, dr);
                    float4 nd4[8];
#pragma unroll
                    for (int jj = 0; jj < 8; ++jj) nd4[jj] = *(const float4*)(delta_g + 32 * c + 4 * jj);
                    tmem_ld_wait(dr);
                    // dS = P * ((dP' - Delta') sc): the bracket in fp32 (one fma with -Delta' sc
                    // from shared memory), rounded to fp16, then multiplied by the fp16 P the dV
                    // MMA consumed (|(dP' - Delta') sc| <= 2^15 by the choice of ds_exp)
                    uint32_t pk[16];
#pragma unroll
                    for (int jj = 0; jj < 16; ++jj) {
                        const float4 d4 = nd4[jj >> 1];
                        const float2 nd = (jj & 1) ? make_float2(d4.z, d4.w) : make_float2(d4.x, d4.y);
                        const float2 d = fma2(make_float2(__uint_as_float(dr[2 * jj]), __uint_as_float(dr[2 * jj + 1])),
                                              make_float2(sc, sc), nd);
                        pk[jj] = hmul2(pack2<true>(d.x, d.y), pkall[16 * c + jj]);
                    }
                    // row r of the [key][query] dS operand (read K-major by dK, MN-major by dQ)
#pragma unroll
                    for (int jj = 0; jj < 4; ++jj) {
                        const uint32_t bytecol = (uint32_t)(c * 64 + jj * 16);
                        *(uint4*)(panel + sw128_offset(r, bytecol)) =
                            make_uint4(pk[4 * jj], pk[4 * jj + 1], pk[4 * jj + 2], pk[4 * jj + 3]);
                    }
                }
                fence_proxy_async_smem();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars[L::bDsFull + grp]);
                if ((warp & 3) == 0 && lane == 0) USP_TL(gk, 8 + 5 * grp);
            }
            // the next item, and its first step's row statistics, before this item's epilogue
            int idx_next = count;
            if (ok && !read_item(item_bars, item_ring, j + 1, abort_flag, idx_next)) ok = false;
            if (ok && idx_next < count) {
                const BwdItem wn = bwd_item(a, idx_next);
                fetch_row_stats(wn, 0, group_scale(a, wn.g).dsc);
            }
            idx = idx_next;
            if (ok) ok = mbar_wait(&bars[L::bKvEmpty], j & 1, abort_flag, kWaitLimitNs);   // dK, dV final
            if (group_any(1 + grp, 128, !ok)) break;
            tc_fence_after();
            // half A writes dV, half B writes dK; TMEM is handed back to the next item's MMAs as
            // soon as the last chunk has been read, before the global stores finish
            const uint32_t src = tbase + lane_off + (grp ? 384 : 256);
            const float un = grp ? group_scale(a, w.g).dk_un : group_scale(a, w.g).dv_un;   // exact powers of two
            const bool of16 = a.out_f16 != 0;
            auto pk_out = [&](float x0, float x1) { return of16 ? pack2<true>(x0 * un, x1 * un) : pack2<false>(x0 * un, x1 * un); };
            if (!a.grad_fp32 && w.kv0 + kBlockN <= w.e) {
                // Whole 16-bit tile: each half stages its accumulator through its own 64-column
                // dS panel, 64 columns per round, and writes each round with one TMA store, so
                // the rows leave as full lines instead of 16-byte pieces 256 bytes apart. The
                // second round is read and packed before the first store, so TMEM goes back to
                // the next item's MMAs at once; the panel is this half's own, so the next item's
                // dS needs no other half's store to finish.
                uint8_t* panel = sm + L::kDS + grp * (kBlockN * 128);
                uint32_t held[32 * (D / 64 - 1) + 1];   // columns 64..D-1, two per word (none for D = 64)
                static_assert(D == 64 || D == 128, "the epilogue holds at most one extra 64-column panel");
#pragma unroll
                for (int c = 0; c < D / 32; ++c) {
                    uint32_t o[32];
                    tmem_ld32(src + 32 * c, o);
                    tmem_ld_wait(o);
                    if (c + 1 == D / 32) {   // the accumulator has been read: TMEM back to the MMAs
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&bars[L::bAccEmpty]);
                    }
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const uint32_t p0 = pk_out(__uint_as_float(o[8 * q]), __uint_as_float(o[8 * q + 1]));
                        const uint32_t p1 = pk_out(__uint_as_float(o[8 * q + 2]), __uint_as_float(o[8 * q + 3]));
                        const uint32_t p2 = pk_out(__uint_as_float(o[8 * q + 4]), __uint_as_float(o[8 * q + 5]));
                        const uint32_t p3 = pk_out(__uint_as_float(o[8 * q + 6]), __uint_as_float(o[8 * q + 7]));
                        const int col = 32 * c + 8 * q;   // first of the 8 columns in this 16-byte chunk
                        if (col < 64) {
                            *(uint4*)(panel + sw128_offset(r, (uint32_t)(col * 2))) = make_uint4(p0, p1, p2, p3);
                        } else if (D > 64) {
                            const int i = (col - 64) / 2;
                            held[i] = p0;
                            held[i + 1] = p1;
                            held[i + 2] = p2;
                            held[i + 3] = p3;
                        }
                    }
                }
#pragma unroll 1
                for (int round = 0; round < D / 64; ++round) {
                    if (round > 0) {   // columns 64..127 into the panel the first store has released
#pragma unroll
                        for (int jj = 0; jj < 8; ++jj)
                            *(uint4*)(panel + sw128_offset(r, (uint32_t)(jj * 16))) =
                                make_uint4(held[4 * jj], held[4 * jj + 1], held[4 * jj + 2], held[4 * jj + 3]);
                    }
                    fence_proxy_async_smem();
                    named_bar_sync(1 + grp, 128);
                    if (r == 0) {
                        tma_store_rows(grp ? &tmDK : &tmDV, panel, round * 64, w.kv0, w.g, a.token_major);
                        bulk_commit_group();
                        bulk_wait_group_read<0>();
                    }
                    named_bar_sync(1 + grp, 128);
                }
                continue;
            }
            // fp32 gradients, or a sample's ragged last tile: row by row
            const int64_t row = act_row(w.g, kv, a.T, a.hkv, a.token_major);
            void* dst_base = grp ? a.dk : a.dv;
#pragma unroll 1
            for (int c = 0; c < D; c += 32) {
                uint32_t o[32];
                tmem_ld32(src + c, o);
                tmem_ld_wait(o);
                if (c + 32 == D) {
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&bars[L::bAccEmpty]);
                }
                if (!kv_ok) continue;
                if (a.grad_fp32) {
                    float4* dst = (float4*)((float*)dst_base + row * D + c);
#pragma unroll
                    for (int jj = 0; jj < 8; ++jj)
                        dst[jj] = make_float4(__uint_as_float(o[4 * jj]) * un, __uint_as_float(o[4 * jj + 1]) * un,
                                              __uint_as_float(o[4 * jj + 2]) * un, __uint_as_float(o[4 * jj + 3]) * un);
                } else {
                    uint4* dst = (uint4*)((uint16_t*)dst_base + row * D + c);
#pragma unroll
                    for (int jj = 0; jj < 4; ++jj)
                        dst[jj] = make_uint4(pk_out(__uint_as_float(o[8 * jj]), __uint_as_float(o[8 * jj + 1])),
                                             pk_out(__uint_as_float(o[8 * jj + 2]), __uint_as_float(o[8 * jj + 3])),
                                             pk_out(__uint_as_float(o[8 * jj + 4]), __uint_as_float(o[8 * jj + 5])),
                                             pk_out(__uint_as_float(o[8 * jj + 6]), __uint_as_float(o[8 * jj + 7])));
                }
            }
        }
        if (r == 0) bulk_wait_group<0>();   // the last tile stores have landed
    } else if (warp < kDqWarp0 + 4) {
        // ------------------------------------------------------------------ dQ group (query rows)
        // Each warp owns 32 query rows of the tile: per 32-column chunk it loads 32 x 32 fp32
        // from TMEM, writes them to its staging buffer in the 128-byte swizzle the dQ tensor
        // map expects, and one lane hands the box to the TMA unit, which adds it to the
        // accumulator at L2. Query rows past the sample end carry exact zeros (their P is
        // zero), so whole boxes can be added; rows past the tensor end are skipped by the TMA.
        // One buffer per warp, so at most one reduction per warp is in flight: measured
        // faster than two (the TMA unit also serves the next blocks' Q and dO loads).
        const int w4 = warp - kDqWarp0;
        const uint32_t tDQ = tbase + ((uint32_t)(w4 * 32) << 16) + 128;
        uint8_t* stage = sm + L::kStage + w4 * kDqChunkBytes;
        if (lane == 0) prefetch_tmap(&tmDQ);
        bool ok = true;
        int gk = 0;
        for (int j = 0; ok; ++j) {
            int idx;
            if (!read_item(item_bars, item_ring, j, abort_flag, idx)) break;
            if (idx >= count) break;
            const BwdItem w = bwd_item(a, idx);
            for (int k = 0; k < w.nsteps; ++k, ++gk) {
                const int h = w.g * G + k / w.nq;
                const int qrow0 = w.q0(k) + w4 * 32;   // first query row of this warp
                if (!__all_sync(0xffffffffu, mbar_wait(&bars[L::bDqFull], gk & 1, abort_flag, kWaitLimitNs))) {
                    ok = false;
                    break;
                }
                if (w4 == 0 && lane == 0) USP_TL(gk, 14);
                // this dQ follows the step's dK, the last MMA reading its Q block: Q's stage is free
                if (w4 == 0 && lane == 0) mbar_arrive(&bars[L::bQEmpty + (gk & 1)]);
                tc_fence_after();
                // chunk c+1 is read from TMEM while chunk c is staged
                uint32_t v[2][32];
                tmem_ld32(tDQ, v[0]);
                tmem_ld_wait(v[0]);
#pragma unroll
                for (int ci = 0; ci < D / 32; ++ci) {
                    const int c = ci * 32;
                    uint32_t (&cur)[32] = v[ci & 1];
                    if (ci + 1 < D / 32) {
                        tmem_ld32(tDQ + c + 32, v[(ci + 1) & 1]);
                    } else {  // the whole tile has left TMEM: its columns are free for the next dQ
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&bars[L::bDqEmpty]);
                        if (w4 == 0 && lane == 0) USP_TL(gk, 15);
                    }
                    uint8_t* buf = stage;
                    // the previous chunk's reduction must have read the buffer
                    if (lane == 0) bulk_wait_group_read<0>();
                    __syncwarp();
#pragma unroll
                    for (int jj = 0; jj < 8; ++jj)   // row `lane`, 16-byte chunk jj, XOR-swizzled by row
                        *(uint4*)(buf + lane * 128 + ((jj ^ (lane & 7)) << 4)) =
                            make_uint4(cur[4 * jj], cur[4 * jj + 1], cur[4 * jj + 2], cur[4 * jj + 3]);
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        tma_reduce_add_rows(&tmDQ, buf, c, qrow0, h, 0);
                        bulk_commit_group();
                    }
                    if (ci + 1 < D / 32) tmem_ld_wait(v[(ci + 1) & 1]);
                }
            }
        }
        if (lane == 0) bulk_wait_group<0>();
    }

    pdl_trigger();   // this CTA has no more items: dq_convert may start launching
    __syncwarp();
    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) tmem_dealloc(tbase, 512);
    if (threadIdx.x == 0 && *abort_flag) atomicCAS(&a.hdr->status, (int)USP_OK, (int)USP_ERR_TIMEOUT);
}

// Largest magnitude of the 8 16-bit values of v.
template <bool F16>
__device__ __forceinline__ float amax8(uint4 v) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    float m = 0.f;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const float2 x = unpack2<F16>(w[j]);
        m = fmax3(m, fabsf(x.x), fabsf(x.y));
    }
    return m;
}

// Block-wide max of `m` (every thread of the 256 calls it), then one atomicMax on the float
// bits, which order like the values for non-negative floats.
__device__ __forceinline__ void block_amax(float m, uint32_t* dst, float* red) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
    __syncthreads();   // `red` may still be read from the previous call
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
    __syncthreads();
    if (threadIdx.x == 0) {
        float b = red[0];
        for (int i = 1; i < 8; ++i) b = fmaxf(b, red[i]);
        atomicMax(dst, __float_as_uint(b));
    }
}

// Delta_i = dO_i . (O_i + O_res_i) in fp32, zero row i of the dQ accumulator, and the largest
// magnitudes of q, dO (of query head blockIdx.y) and of k, v (of key/value head blockIdx.y,
// when there is one). TPR threads per row, each owning 8 consecutive elements (16 bytes).
template <int D, bool F16>
__global__ void __launch_bounds__(256) bwd_stats_kernel(const BwdStatsArgs a) {
    constexpr int TPR = D / 8;   // threads per row, 8 elements (16 bytes) each
    pdl_trigger();   // the next kernel waits for this one's completion before it reads anything
    __shared__ float red[8];
    const int h = blockIdx.y;
    const int sub = threadIdx.x % TPR;
    const int64_t T = a.T;
    const bool kv_head = h < a.hkv;
    float mq = 0.f, mdo = 0.f, mk = 0.f, mv = 0.f;
    constexpr int64_t kRowsPerCta = 256 / TPR;
    // the loop bound is uniform across the CTA so that every lane reaches the shuffles
    for (int64_t base = (int64_t)blockIdx.x * kRowsPerCta; base < T; base += (int64_t)gridDim.x * kRowsPerCta) {
        const int64_t t = base + threadIdx.x / TPR;
        const bool valid = t < T;
        float acc = 0.f;
        if (valid) {
            const int64_t arow = act_row(h, t, T, a.hq, a.token_major);
            const uint4 ov = __ldg((const uint4*)(a.o + arow * D) + sub);
            const uint4 dv = __ldg((const uint4*)(a.dout + arow * D) + sub);
            const uint4 qv = __ldg((const uint4*)(a.q + arow * D) + sub);
            const uint4 rv = a.o_res ? __ldg((const uint4*)(a.o_res + arow * D) + sub) : make_uint4(0, 0, 0, 0);
            const uint32_t o2[4] = {ov.x, ov.y, ov.z, ov.w};
            const uint32_t r2[4] = {rv.x, rv.y, rv.z, rv.w};
            const uint32_t d2[4] = {dv.x, dv.y, dv.z, dv.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float2 x = unpack2<F16>(o2[j]);
                const float2 xr = unpack2<F16>(r2[j]);
                const float2 y = unpack2<F16>(d2[j]);
                acc = fmaf(x.x + xr.x, y.x, acc);
                acc = fmaf(x.y + xr.y, y.y, acc);
            }
            mq = fmaxf(mq, amax8<F16>(qv));
            mdo = fmaxf(mdo, amax8<F16>(dv));
            if (kv_head) {
                const int64_t krow = act_row(h, t, T, a.hkv, a.token_major);
                mk = fmaxf(mk, amax8<F16>(__ldg((const uint4*)(a.k + krow * D) + sub)));
                mv = fmaxf(mv, amax8<F16>(__ldg((const uint4*)(a.v + krow * D) + sub)));
            }
        }
#pragma unroll
        for (int off = TPR / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
        if (valid) {
            if (sub == 0) a.delta[(int64_t)h * T + t] = acc;
            float4* z = (float4*)(a.dq_acc + ((int64_t)h * T + t) * D) + 2 * sub;
            z[0] = make_float4(0.f, 0.f, 0.f, 0.f);
            z[1] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
    }
    const int g = h / a.group;
    block_amax(mq, a.amax + kAmaxQ * a.hkv + g, red);
    block_amax(mdo, a.amax + kAmaxDO * a.hkv + g, red);
    if (kv_head) {   // uniform over the CTA
        block_amax(mk, a.amax + kAmaxK * a.hkv + h, red);
        block_amax(mv, a.amax + kAmaxV * a.hkv + h, red);
    }
}

// The fp16 operand copies: tensor blockIdx.z (q, k, v, dO), head blockIdx.y, scaled by
// 2^range_exponent(amax of its key/value group) and written head-major. 8 elements per thread.
template <int D, bool F16>
__global__ void __launch_bounds__(256) bwd_convert_kernel(const BwdConvertArgs a) {
    constexpr int TPR = D / 8;
    pdl_wait();   // amax is final once the stats kernel has completed
    pdl_trigger();
    const int tz = blockIdx.z;
    const bool kv = tz == kAmaxK || tz == kAmaxV;
    const int H = kv ? a.hkv : a.hq;
    const int h = blockIdx.y;
    if (h >= H) return;
    const int g = kv ? h : h / a.group;
    const float sc = exp2i(range_exponent(__ldg(a.amax + tz * a.hkv + g)));
    // constant indices keep the parameter arrays out of local memory
    const uint16_t* src = tz == 0 ? a.src[0] : tz == 1 ? a.src[1] : tz == 2 ? a.src[2] : a.src[3];
    uint16_t* dst = (tz == 0 ? a.dst[0] : tz == 1 ? a.dst[1] : tz == 2 ? a.dst[2] : a.dst[3]) + (int64_t)h * a.T * D;
    const int sub = threadIdx.x % TPR;
    constexpr int64_t kRowsPerCta = 256 / TPR;
    for (int64_t t = (int64_t)blockIdx.x * kRowsPerCta + threadIdx.x / TPR; t < a.T;
         t += (int64_t)gridDim.x * kRowsPerCta) {
        const uint4 x = __ldg((const uint4*)(src + act_row(h, t, a.T, H, a.token_major) * D) + sub);
        const uint32_t w[4] = {x.x, x.y, x.z, x.w};
        uint32_t r[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float2 f = unpack2<F16>(w[j]);
            r[j] = pack2<true>(f.x * sc, f.y * sc);
        }
        ((uint4*)(dst + t * D))[sub] = make_uint4(r[0], r[1], r[2], r[3]);
    }
}

// The head-major fp32 accumulator, which holds dQ' = dQ 2^(ev+edo+ds_exp+ek) of each head's
// key/value group, scaled back and written as dq (bf16, fp16 or fp32; head-major or
// token-major). D4 (= D / 4, a power of two) threads per row, 4 elements each.
struct DqConvertArgs {
    const float4* src;
    void* dst;
    const uint32_t* amax;
    int64_t T;
    int H, hkv, group, token_major, out_dt, ds_exp;
};
template <int D4>
__global__ void __launch_bounds__(256) dq_convert_kernel(const DqConvertArgs a) {
    pdl_wait();   // the accumulator is final once the backward kernel has completed
    const int h = blockIdx.y;
    const int g = h / a.group;
    const int ek = range_exponent(__ldg(a.amax + kAmaxK * a.hkv + g));
    const int ev = range_exponent(__ldg(a.amax + kAmaxV * a.hkv + g));
    const int edo = range_exponent(__ldg(a.amax + kAmaxDO * a.hkv + g));
    const float un = exp2i(-(ev + edo + a.ds_exp + ek));   // exact power of two
    const float4* s_head = a.src + (int64_t)h * a.T * D4;
    const int64_t n = a.T * D4;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t t = i / D4;
        const int c = (int)(i % D4);
        const float4 v = s_head[i];
        const int64_t o = act_row(h, t, a.T, a.H, a.token_major) * D4 + c;
        if (a.out_dt == USP_FP32)
            ((float4*)a.dst)[o] = make_float4(v.x * un, v.y * un, v.z * un, v.w * un);
        else if (a.out_dt == USP_FP16)
            ((uint2*)a.dst)[o] = make_uint2(pack2<true>(v.x * un, v.y * un), pack2<true>(v.z * un, v.w * un));
        else
            ((uint2*)a.dst)[o] = make_uint2(pack2<false>(v.x * un, v.y * un), pack2<false>(v.z * un, v.w * un));
    }
}

__global__ void debug_timeout_kernel(WsHeader* hdr, uint64_t limit_ns) {
    __shared__ uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        abort_flag = 0;
        fence_barrier_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        // nothing ever arrives on `bar`: the bounded wait must give up and report it
        if (!mbar_wait(&bar, 0, &abort_flag, limit_ns)) atomicCAS(&hdr->status, (int)USP_OK, (int)USP_ERR_TIMEOUT);
    }
}

template <int D>
cudaError_t launch_bwd_impl(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v, const CUtensorMap& dout,
                            const CUtensorMap& dq, const CUtensorMap& dk, const CUtensorMap& dv, const BwdArgs& a,
                            int grid, cudaStream_t s) {
    using L = BwdSmem<D>;
    // persistent CTAs, one per SM (the shared-memory footprint allows no more)
    int sms = 0;
    const cudaError_t e = persistent_setup<attn_bwd_kernel<D, true>>((size_t)L::kAlloc, &sms);
    if (e != cudaSuccess) return e;
    if (grid > sms) grid = sms;
    return launch_kernel(attn_bwd_kernel<D, true>, dim3(grid), dim3(kBwdThreads), (size_t)L::kAlloc, s, true, q, k,
                         v, dout, dq, dk, dv, a);
}

// CTAs for `work_items` units at `per_cta` units each, capped so that all `ys` rows of the
// grid together keep about 16 CTAs per SM.
int grid_for(int64_t work_items, int per_cta, int ys = 1) {
    int64_t g = (work_items + per_cta - 1) / per_cta;
    const int sms = device_sm_count();
    const int64_t cap = ((sms > 0 ? sms : 148) * 16 + ys - 1) / ys;
    if (g > cap) g = cap;
    if (g < 1) g = 1;
    return (int)g;
}

}  // namespace

int ds_exponent(int head_dim, float scale) {
    // bound on |dS| for operands below 16: 2 * D * 16 * 16 * scale
    const double bound = 512.0 * (double)head_dim * (double)scale;
    int e = (int)std::floor(std::log2(32768.0 / bound));
    return e < -24 ? -24 : (e > 24 ? 24 : e);
}

cudaError_t launch_attn_bwd(int head_dim, const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                            const CUtensorMap& dout, const CUtensorMap& dq, const CUtensorMap& dk, const CUtensorMap& dv,
                            const BwdArgs& a, int grid, cudaStream_t s) {
    if (head_dim == 128) return launch_bwd_impl<128>(q, k, v, dout, dq, dk, dv, a, grid, s);
    return launch_bwd_impl<64>(q, k, v, dout, dq, dk, dv, a, grid, s);
}

cudaError_t launch_bwd_stats(int head_dim, const BwdStatsArgs& a, cudaStream_t s) {
    const int tpr = head_dim / 8;
    const dim3 grid(grid_for(a.T, 256 / tpr, a.hq), a.hq);
    if (head_dim == 128 && a.f16)
        bwd_stats_kernel<128, true><<<grid, 256, 0, s>>>(a);
    else if (head_dim == 128)
        bwd_stats_kernel<128, false><<<grid, 256, 0, s>>>(a);
    else if (a.f16)
        bwd_stats_kernel<64, true><<<grid, 256, 0, s>>>(a);
    else
        bwd_stats_kernel<64, false><<<grid, 256, 0, s>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_bwd_convert(int head_dim, const BwdConvertArgs& a, cudaStream_t s) {
    const int tpr = head_dim / 8;
    const int hmax = a.hq > a.hkv ? a.hq : a.hkv;
    const dim3 grid(grid_for(a.T, 256 / tpr, 2 * a.hq + 2 * a.hkv), hmax, 4);
    auto kernel = head_dim == 128 ? (a.f16 ? bwd_convert_kernel<128, true> : bwd_convert_kernel<128, false>)
                                  : (a.f16 ? bwd_convert_kernel<64, true> : bwd_convert_kernel<64, false>);
    return launch_kernel(kernel, grid, dim3(256), 0, s, true, a);
}

cudaError_t launch_dq_convert(const float* dq_acc, void* dq, const uint32_t* amax, int64_t T, int hq, int hkv,
                              int head_dim, int token_major, int out_dt, int ds_exp, cudaStream_t s) {
    const int D4 = head_dim / 4;
    const dim3 grid(grid_for(T * D4, 256, hq), hq);
    DqConvertArgs a{(const float4*)dq_acc, dq, amax, T, hq, hkv, hq / hkv, token_major, out_dt, ds_exp};
    // launched right after the backward kernel, whose completion it waits for on the device
    auto kernel = D4 == 32 ? dq_convert_kernel<32> : dq_convert_kernel<16>;
    return launch_kernel(kernel, grid, dim3(256), 0, s, true, a);
}

#ifdef USP_TIMELINE
// The backward's timeline (kTlCtas x kTlSteps x kTlEvents clock64 values) into host memory.
extern "C" int usp_debug_timeline(void* host_dst, size_t bytes) {
    if (bytes < sizeof(g_timeline)) return (int)USP_ERR_INVALID_ARG;
    return cudaMemcpyFromSymbol(host_dst, g_timeline, sizeof(g_timeline)) == cudaSuccess ? 0 : (int)USP_ERR_CUDA;
}
#endif

cudaError_t launch_debug_timeout(WsHeader* hdr, uint64_t limit_ns, cudaStream_t s) {
    debug_timeout_kernel<<<1, 32, 0, s>>>(hdr, limit_ns);
    return cudaGetLastError();
}

}  // namespace usp
