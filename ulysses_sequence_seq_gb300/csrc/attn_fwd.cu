// Forward of the local attention step of Ulysses sequence parallelism on sm_103a:
// causal, sample-boundary-masked softmax attention over the full packed sequence for
// the heads a rank owns, written FlashAttention-style (online softmax, O(n) memory,
// no materialised score matrix; congresoia365 article, "El Desafío del
// Entrenamiento de Secuencias Largas", and HF guide "Configurar" on packed samples).
//
// Two forms of one kernel, persistent and warp-specialised:
//  * head_dim 128 -- a pair of CTAs (a cluster of two, one per SM) shares every MMA
//    (tcgen05 cta_group::2, M = 256): each CTA holds 128 query rows of each of its two
//    256-row tiles and only half of each key/value block's operands (64 of its 128 keys of
//    K, 64 of the 128 columns of V). With one CTA per tile, each SM would take in 64 KB of K
//    and V per block and its MMAs would read both operands of every Q.K^T from its own
//    shared memory; that traffic, not the tensor core, set the pace. The pair halves both.
//    A work item is 512 query rows; the leader (rank 0) takes the items, issues the MMAs and
//    counts both CTAs' loads on its barriers; the halved operands leave room for a 4-stage
//    key/value ring.
//  * head_dim 64 -- one CTA per SM, two 128-row query tiles (256 rows) per item, a
//    2-stage ring.
// Pairs (or CTAs) take their first item by index and the rest from a counter, in schedule
// order, so the next item's Q, K, V loads and first Q.K^T overlap the softmax of the
// current one's last blocks and its output.
// Warp roles (384 threads per CTA, warp 11 idle):
//   warps 0-3  softmax group for query tile 0 (thread = one query row = one TMEM lane)
//   warps 4-7  softmax group for query tile 1
//   warp  8    TMA producer: Q tiles once, then K/V blocks (or this CTA's halves) into the ring
//   warp  9    MMA issuer of tile 0 (one thread; the pair's leader only) and TMEM owner
//   warp  10   MMA issuer of tile 1
// Tensor memory (512 columns): S0 [0,128), S1 [128,256), O0 [256,256+D), O1 [384,384+D).
// A whole output tile leaves through a 64-column shared-memory panel of its own, one TMA
// store per 64 columns; a sample's ragged last tile is written row by row. On request the
// rounding residual of O (the fp32 result minus its 16-bit rounding) leaves the same way,
// so that the backward can take Delta = dO . O from O to about 16 significant bits.
// P (bf16 or fp16, the input type) overwrites the first 64 columns of its S tile and feeds the P.V MMA
// straight from TMEM. The two tiles ping-pong: while one softmax group works on
// its S, the tensor core runs the other tile's P.V and next Q.K^T. Each tile has its own MMA
// thread, so that one thread's waits (for its P and the next K/V block) overlap the other's
// batch in the tensor pipe, whose issue queue is about one MMA deep; a turn passed between
// the two threads keeps the tiles half a period apart. The threads commit only S-ready and
// O-done: each tile's softmax group releases the ring stages and Q its MMAs have read.
// The O rescale is lazy: the running max is only moved when a row's max grows by
// more than 2^8, which is exact after the final division by the row sum.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "attn.cuh"
#include "common.cuh"
#include "ptx.cuh"
#include "tiles.cuh"

namespace usp {
namespace {

using namespace ptx;

constexpr int kFwdThreads = 384;  // 3 warpgroups: two softmax groups, one for load / MMA (2 warps idle)
// Register shares (per thread) after setmaxnreg: the softmax groups hold a 128-column score
// row each; the load/MMA warpgroup keeps the item ring, the block counters and both tiles'
// barrier phases across the persistent loop. Launched with kLaunchRegs per thread,
// 128 * (2 * kSoftmaxRegs + kAuxRegs) must not exceed kFwdThreads * kLaunchRegs.
constexpr int kLaunchRegs = 168;
constexpr int kSoftmaxRegs = 200;
constexpr int kAuxRegs = 104;
static_assert(128 * (2 * kSoftmaxRegs + kAuxRegs) <= kFwdThreads * kLaunchRegs, "register split exceeds the launch pool");
constexpr float kRescaleThreshold = 8.0f;  // log2 units
constexpr uint16_t kPairMask = 0x3;        // both CTAs of a pair

template <int D, bool PAIR>
struct FwdSmem {
    static_assert(!PAIR || D == 128, "the pair splits V into two 64-column panels");
    static constexpr int kPanels = D / 64;
    static constexpr int kTileBytes = kTileM * D * 2;          // one 128-row tile of 16-bit elements
    static constexpr int kStages = PAIR ? 4 : 2;               // key/value ring depth
    static constexpr int kKRows = PAIR ? kBlockN / 2 : kBlockN;   // keys of a block whose K this CTA holds
    static constexpr int kKPanel = kKRows * 128;               // one 64-column panel of them
    static constexpr int kKBytes = kKPanel * kPanels;
    static constexpr int kVPanels = PAIR ? kPanels / 2 : kPanels;   // 64-column panels of V this CTA holds
    static constexpr int kVBytes = kBlockN * 128 * kVPanels;
    static constexpr int kQ0 = 0;
    static constexpr int kQ1 = kTileBytes;
    static constexpr int kK = 2 * kTileBytes;                  // + stage * kKBytes
    static constexpr int kV = kK + kStages * kKBytes;          // + stage * kVBytes
    static constexpr int kStage = kV + kStages * kVBytes;      // O staging: one [128][64] panel per tile
    static constexpr int kBars = kStage + 2 * kTileM * 128;
    // barrier indices
    // bKvFull: a stage's K and V both landed (one barrier, so that an MMA thread checks a block once);
    // bDrain, bTurn: one per tile's MMA thread
    static constexpr int bQFull = 0, bKvFull = 1, bKvEmpty = bKvFull + kStages,
                         bSFull = bKvEmpty + kStages, bPFull = bSFull + 2, bODone = bPFull + 2, bDrain = bODone + 2,
                         bTurn = bDrain + 2, bQEmpty = bTurn + 2, bItem = bQEmpty + 1, bItemFree = bItem + 4,
                         kNumBars = bItemFree + 4;
    // bItem / bItemFree: published / read by every reader, one of each per slot of the 4-slot item ring
    static constexpr int kItemRing = kBars + 8 * kNumBars;   // int[4]: work item of each slot
    static constexpr int kTmemSlot = kItemRing + 16;
    static constexpr int kAbort = kTmemSlot + 8;
    static constexpr int kBytes = kAbort + 8;
    static constexpr int kAlloc = kBytes + 1024;  // slack for 1024-byte alignment of the base
    static_assert(kKBytes % 1024 == 0 && kVBytes % 1024 == 0, "ring stages must keep 1024-byte alignment");
};
static_assert(FwdSmem<128, true>::kAlloc <= 232448, "forward shared memory exceeds the per-CTA limit");
static_assert(FwdSmem<64, false>::kAlloc <= 232448, "forward shared memory exceeds the per-CTA limit");

// Optional clock64 timeline of the first kTlSteps key/value blocks of every CTA (compile with
// -DUSP_TIMELINE; the default build has none of it). Events by the CTA's running block count:
// MMA threads 15 (tile 0's block started), 1-2 (tile 0 / 1 P ready and turn taken), 3-4 (tile 0 / 1
// next S issued); softmax
// group t 5+4t (S ready), 6+4t (row max done), 8+4t (P stored), 7+4t (P-ready arrival made);
// producer 13-14 (K / V load issued). Read back with usp_debug_fwd_timeline.
#ifdef USP_TIMELINE
#ifndef USP_TIMELINE_FIRST
#define USP_TIMELINE_FIRST 0   // first recorded block (a later window shows the steady state)
#endif
constexpr int kFTlSteps = 48, kFTlEvents = 16, kFTlCtas = 160;
static __device__ long long g_fwd_timeline[kFTlCtas][kFTlSteps][kFTlEvents];
#define USP_FTL(step, ev)                                                                            \
    do {                                                                                             \
        const int s_ = (step) - USP_TIMELINE_FIRST;                                                  \
        if (s_ >= 0 && s_ < kFTlSteps && blockIdx.x < kFTlCtas) g_fwd_timeline[blockIdx.x][s_][(ev)] = clock64(); \
    } while (0)
#else
#define USP_FTL(step, ev) \
    do {                  \
    } while (0)
#endif

// Query rows of one forward work item (a multiple of both tiles' 128 rows).
template <bool PAIR>
__host__ __device__ constexpr int fwd_item_rows() {
    return PAIR ? 4 * kTileM : 2 * kTileM;
}

// One forward work item as this CTA sees it: query head h of the sample [s, e); this CTA's
// rows of query tiles 0 and 1 start at q00 and q01, and the tiles take nb0 and nb1 key/value
// blocks. In a pair, tile t is the 256 rows from base + 256 t (the leader holds the first 128,
// the peer the rest), and its block count is the pair's, so both CTAs walk the same blocks
// (a row that sees none of a block's keys has them all masked).
struct FwdItem {
    int h, s, e, q00, q01, nb0, nb1, nmax, kvh;
};
template <bool PAIR>
__device__ __forceinline__ FwdItem fwd_item(const FwdArgs& a, int idx, uint32_t rank) {
    const WorkItem it = a.items[idx];
    FwdItem f;
    f.h = it.head;
    f.s = a.cu[it.seq];
    f.e = a.cu[it.seq + 1];
    const int base = f.s + it.tile * fwd_item_rows<PAIR>();
    if constexpr (PAIR) {
        f.q00 = base + (int)rank * kTileM;
        f.q01 = f.q00 + 2 * kTileM;
        const int a0 = kv_blocks_for_query_tile(base, f.s, f.e, a.causal);
        const int a1 = kv_blocks_for_query_tile(base + kTileM, f.s, f.e, a.causal);
        const int b0 = kv_blocks_for_query_tile(base + 2 * kTileM, f.s, f.e, a.causal);
        const int b1 = kv_blocks_for_query_tile(base + 3 * kTileM, f.s, f.e, a.causal);
        f.nb0 = a0 > a1 ? a0 : a1;
        f.nb1 = b0 > b1 ? b0 : b1;
    } else {
        f.q00 = base;
        f.q01 = base + kTileM;
        f.nb0 = kv_blocks_for_query_tile(f.q00, f.s, f.e, a.causal);
        f.nb1 = kv_blocks_for_query_tile(f.q01, f.s, f.e, a.causal);
    }
    f.nmax = f.nb0 > f.nb1 ? f.nb0 : f.nb1;
    f.kvh = f.h / a.group;
    return f;
}

// Bounded wait on a per-block barrier. In a pair the other CTA's arrivals on it are MMA
// commits (for data the waiter reads through tcgen05 after tcgen05.fence::after_thread_sync)
// and P-ready signals (for P in tensor memory), so a CTA-scope acquire is enough.
template <bool PAIR>
__device__ __forceinline__ bool fwait(uint64_t* bar, uint32_t parity, volatile int* abort_flag) {
    return mbar_wait(bar, parity, abort_flag, kWaitLimitNs);
}
// Signal the barrier at `bar`'s offset in the pair's leader (this CTA's own otherwise).
template <bool PAIR>
__device__ __forceinline__ void arrive_leader(uint64_t* bar, uint32_t rank) {
    if (PAIR && rank != 0)
        mbar_arrive_remote_signal(mapa_shared(smem_u32(bar), 0));
    else
        mbar_arrive(bar);
}
// Release an item slot on the leader's free barrier: at cluster scope, since the leader then
// rewrites the slot in this CTA's shared memory with a generic store.
template <bool PAIR>
__device__ __forceinline__ void release_item_slot(uint64_t* bar, uint32_t rank) {
    if (PAIR && rank != 0)
        mbar_arrive_remote(mapa_shared(smem_u32(bar), 0));
    else
        mbar_arrive(bar);
}
// MMA commit to the barrier at `bar`'s offset in every CTA that waits on it.
template <bool PAIR>
__device__ __forceinline__ void commit_all(uint64_t* bar) {
    if constexpr (PAIR)
        mma_commit_pair_multicast(bar, kPairMask);
    else
        mma_commit(bar);
}

// The j-th work item from this CTA's 4-slot ring (false: the wait gave up), which the
// producer (in a pair, the leader's, in both CTAs) writes. Each reader then frees the slot on
// the leader's free barrier; the slot is rewritten only once every reader has, because a
// softmax group whose tile has no blocks in a run of items is not held back by the MMAs and
// may lag.
template <bool PAIR>
__device__ __forceinline__ bool fwd_read_item(uint64_t* item_bars, volatile int* ring, int j,
                                              volatile int* abort_flag, int& idx) {
    // the slot was written by the leader's producer, in a pair with a remote generic store
    const bool got = PAIR ? mbar_wait_cluster(&item_bars[j & 3], (j >> 2) & 1, abort_flag, kWaitLimitNs)
                          : mbar_wait(&item_bars[j & 3], (j >> 2) & 1, abort_flag, kWaitLimitNs);
    if (!got) return false;
    idx = ring[j & 3];
    return true;
}
// Readers of an item slot: the two MMA threads and the 8 softmax warps; in a pair the
// leader's MMA threads, both CTAs' softmax warps and the peer's producer.
template <bool PAIR>
__host__ __device__ constexpr int fwd_slot_readers() {
    return PAIR ? 2 + 2 * 8 + 1 : 2 + 8;
}

template <int D, bool F16, bool PAIR>
__global__ void __maxnreg__(kLaunchRegs)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO,
                    const __grid_constant__ CUtensorMap tmOres, const FwdArgs a) {
    using L = FwdSmem<D, PAIR>;
    constexpr int S = L::kStages;
    pdl_wait();   // the work list and the header come from the scheduler launched just before
    const int count = a.hdr->fwd_count;
    const uint32_t rank = PAIR ? cluster_ctarank() : 0;
    const int unit = PAIR ? (int)blockIdx.x >> 1 : (int)blockIdx.x;   // this pair (or CTA)
    const int units = PAIR ? (int)gridDim.x >> 1 : (int)gridDim.x;
    // the same answer in both CTAs of a pair (the count is final): they take the same path
    if (unit >= count) return;
    if constexpr (!PAIR) {
        // once any CTA of this launch has timed out, the rest skip their work (a pair's leader
        // checks before each item and ends both CTAs' work through the item ring)
        if (*(volatile int*)&a.hdr->status != (int)USP_OK) return;
    }

    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint64_t* bars = (uint64_t*)(sm + L::kBars);
    uint32_t* tmem_slot = (uint32_t*)(sm + L::kTmemSlot);
    volatile int* abort_flag = (volatile int*)(sm + L::kAbort);
    volatile int* item_ring = (volatile int*)(sm + L::kItemRing);
    uint64_t* item_bars = &bars[L::bItem];
    uint64_t* item_free = &bars[L::bItemFree];

    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x % 32;

    if (warp == 9) {
        if constexpr (PAIR) {
            tmem_alloc_pair(tmem_slot, 512);
            tmem_relinquish_pair();
        } else {
            tmem_alloc(tmem_slot, 512);
            tmem_relinquish();
        }
    }
    if (threadIdx.x == 0) {
        mbar_init(&bars[L::bQFull], 1);
        for (int i = 0; i < S; ++i) {
            mbar_init(&bars[L::bKvFull + i], 1);
            mbar_init(&bars[L::bKvEmpty + i], 2);   // one releasing softmax thread per tile
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bars[L::bSFull + i], 1);
            mbar_init(&bars[L::bPFull + i], PAIR ? 8 : 4);   // the tile's softmax warps (of both CTAs)
            mbar_init(&bars[L::bODone + i], 1);
            mbar_init(&bars[L::bDrain + i], 1);
            mbar_init(&bars[L::bTurn + i], 1);
        }
        mbar_init(&bars[L::bQEmpty], 2);
        for (int i = 0; i < 4; ++i) {
            mbar_init(&bars[L::bItem + i], 1);
            mbar_init(&bars[L::bItemFree + i], fwd_slot_readers<PAIR>());
        }
        *abort_flag = 0;
        fence_barrier_init();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = *tmem_slot;
    // the peer's barriers are initialised before any remote arrival or copy reaches them
    if constexpr (PAIR) cluster_sync_all();

    // Every per-block barrier phase follows a running count across items (the key/value
    // blocks for the ring, each tile's blocks for S and P); Q's follow the item count j, and a
    // tile's O-done the count of items in which that tile has blocks. Each phase of these
    // barriers needs its waiter to have passed the one before, so a waiter is never two
    // phases behind and parities cannot alias.
    if (warp == 11) {
        regs_decrease<kAuxRegs>();  // the idle warp of the load/MMA warpgroup
    } else if (warp == 8) {
        regs_decrease<kAuxRegs>();
        // ------------------------------------------------------------------ TMA producer
        if (lane == 0) {
            prefetch_tmap(&tmQ);
            prefetch_tmap(&tmK);
            prefetch_tmap(&tmV);
            // a load completes on the leader's barrier in a pair, on this CTA's otherwise
            auto load = [&](void* dst, const CUtensorMap* map, uint64_t* bar, int x, int row, int h) {
                if constexpr (PAIR)
                    tma_load_rows_pair(dst, map, mapa_shared(smem_u32(bar), 0), x, row, h, a.token_major);
                else
                    tma_load_rows(dst, map, bar, x, row, h, a.token_major);
            };
            const bool leader = rank == 0;
            bool ok = true;
            int gn = 0, q_loads = 0;
            int next_idx = unit;
            for (int j = 0; ok; ++j) {
                int idx;
                if (leader) {
                    idx = next_idx;
                    next_idx = -1;
                    // once any CTA of this launch has timed out, the rest end their work
                    if (PAIR && *(volatile int*)&a.hdr->status != (int)USP_OK) idx = count;
                    // every reader has taken the item this slot held four items ago
                    if (j >= 4 && !(PAIR ? mbar_wait_cluster(&item_free[j & 3], ((j >> 2) - 1) & 1, abort_flag,
                                                             kWaitLimitNs)
                                         : mbar_wait(&item_free[j & 3], ((j >> 2) - 1) & 1, abort_flag,
                                                     kWaitLimitNs)))
                        break;
                    item_ring[j & 3] = idx;
                    mbar_arrive(&item_bars[j & 3]);   // release: the slot write is visible to its readers
                    if constexpr (PAIR) {
                        st_cluster_u32(mapa_shared(smem_u32((const void*)&item_ring[j & 3]), 1), (uint32_t)idx);
                        mbar_arrive_remote(mapa_shared(smem_u32(&item_bars[j & 3]), 1));
                    }
                } else {
                    if (!fwd_read_item<PAIR>(item_bars, item_ring, j, abort_flag, idx)) break;
                    release_item_slot<PAIR>(&item_free[j & 3], rank);
                }
                if (idx >= count) break;
                const FwdItem f = fwd_item<PAIR>(a, idx, rank);
                // the Q buffers are free once the previous item's last Q.K^T has run
                if (j > 0 && !fwait<PAIR>(&bars[L::bQEmpty], (j - 1) & 1, abort_flag)) break;
                const int ntiles = f.nb1 > 0 ? 2 : 1;
                if (leader) mbar_arrive_expect_tx(&bars[L::bQFull], (PAIR ? 2 : 1) * ntiles * L::kTileBytes);
                for (int t = 0; t < ntiles; ++t)
                    for (int p = 0; p < L::kPanels; ++p)
                        load(sm + (t ? L::kQ1 : L::kQ0) + p * (kTileM * 128), &tmQ, &bars[L::bQFull], p * 64,
                             t ? f.q01 : f.q00, f.h);
                ++q_loads;
                for (int n = 0; n < f.nmax; ++n, ++gn) {
                    const int st = gn % S;
                    if (gn >= S && !fwait<PAIR>(&bars[L::bKvEmpty + st], ((gn / S) - 1) & 1, abort_flag)) {
                        ok = false;
                        break;
                    }
                    const int row = f.s + n * kBlockN;
                    const int krow = row + (int)rank * L::kKRows;   // this CTA's keys of the block
                    const int vcol = (int)rank * 64 * L::kVPanels;  // and its columns of V
                    if (leader) {
                        mbar_arrive_expect_tx(&bars[L::bKvFull + st], (PAIR ? 2 : 1) * (L::kKBytes + L::kVBytes));
                    }
                    USP_FTL(gn, 13);
                    for (int p = 0; p < L::kPanels; ++p)
                        load(sm + L::kK + st * L::kKBytes + p * L::kKPanel, &tmK, &bars[L::bKvFull + st], p * 64, krow,
                             f.kvh);
                    USP_FTL(gn, 14);
                    for (int p = 0; p < L::kVPanels; ++p)
                        load(sm + L::kV + st * L::kVBytes + p * (kBlockN * 128), &tmV, &bars[L::bKvFull + st],
                             vcol + p * 64, row, f.kvh);
                    // The CTAs walk the same key/value blocks in near lockstep, so a block's first
                    // load goes to DRAM for all of them: pull this CTA's share two blocks ahead into L2.
                    if (n + 2 < f.nmax) {
                        for (int p = 0; p < L::kPanels; ++p)
                            tma_prefetch_rows(&tmK, p * 64, krow + 2 * kBlockN, f.kvh, a.token_major);
                        for (int p = 0; p < L::kVPanels; ++p)
                            tma_prefetch_rows(&tmV, vcol + p * 64, row + 2 * kBlockN, f.kvh, a.token_major);
                    }
                    // two blocks before the end, reserve the next item and pull its Q into L2
                    if (leader && n == (f.nmax >= 2 ? f.nmax - 2 : 0)) {
                        next_idx = units + atomicAdd(&a.hdr->fwd_next, 1);
                        if (next_idx < count) {
                            const WorkItem nit = a.items[next_idx];
                            const int nbase = a.cu[nit.seq] + nit.tile * fwd_item_rows<PAIR>();
                            const int nend = a.cu[nit.seq + 1];
                            for (int r = 0; r < fwd_item_rows<PAIR>() && nbase + r < nend; r += kTileM)
                                for (int p = 0; p < L::kPanels; ++p)
                                    tma_prefetch_rows(&tmQ, p * 64, nbase + r, nit.head, a.token_major);
                        }
                    }
                }
                // (every item has blocks: its first tile starts inside its sample; kept for safety)
                if (leader && ok && next_idx < 0) next_idx = units + atomicAdd(&a.hdr->fwd_next, 1);
            }
            // Before the CTAs may exit, every copy must have landed. In a pair all of them
            // complete on the leader's barriers (the CTAs leave together, after both have
            // finished). The last use of each barrier is its final phase, so waiting on it is
            // always sound.
            if (leader) {
                if (q_loads > 0) mbar_wait_drain(&bars[L::bQFull], (q_loads - 1) & 1, kDrainLimitNs);
                for (int n = gn - S < 0 ? 0 : gn - S; n < gn; ++n) {
                    mbar_wait_drain(&bars[L::bKvFull + n % S], (n / S) & 1, kDrainLimitNs);
                }
            }
        }
    } else if (warp == 9 || warp == 10) {
        regs_decrease<kAuxRegs>();
        // ------------------------------------------------------------------ MMA issuers
        // One thread per query tile (the pair's leader only): tile t's thread issues its P.V
        // and Q.K^T. The tensor pipe's issue queue is about one MMA deep, so a thread that
        // waits between two batches leaves the pipe idle; with two threads, one waits (for its
        // tile's P, the next K/V block and its turn) while the other's batch runs. The turn
        // keeps the tiles half a period apart: per item there are 1 + nmax slots (the first
        // Q.K^T, then one per key/value block), tile 0 goes first in each and hands the turn
        // to tile 1 shortly before its batch's last MMAs, tile 1 hands it back. A tile with
        // nothing in a slot passes the turn on at once. Without the turn, two free-running
        // threads let the tiles fall into phase (both S ready together, both softmax groups
        // competing, then both batches).
        if (lane == 0 && rank == 0) {
            const int t = warp - 9;
            constexpr int M = PAIR ? 2 * kTileM : kTileM;
            constexpr uint32_t idS = idesc_16b_f32(M, kBlockN, false, false, F16);  // Q.K^T: both K-major
            constexpr uint32_t idO = idesc_16b_f32(M, D, false, true, F16);         // P.V: V is MN-major
            // The turn goes to the other tile this many MMAs before a batch ends (measured on the
            // 262,144-token slice: 0 -> 1516, 1 -> 1548-1560, 2 -> 1548, 3 -> 1545, 4 -> 1534 TFLOP/s).
            constexpr int kEarly = 1;
            // The 64-bit shared-memory descriptors are built once; a K step only adds a constant
            // to the start-address field (addresses stay below 2^18, so the field never carries).
            // Rebuilding them per MMA made the issuing thread, not the tensor core, the limit.
            const uint64_t dQt = sdesc_sw128(smem_u32(sm + (t ? L::kQ1 : L::kQ0)), 0, 1024);
            const uint64_t dK0 = sdesc_sw128(smem_u32(sm + L::kK), 0, 1024);
            const uint64_t dV0 = sdesc_sw128(smem_u32(sm + L::kV), kBlockN * 128, 1024);
            const uint32_t tS = tbase + t * 128, tO = tbase + 256 + t * 128;
            auto pass_turn = [&]() { mbar_arrive(&bars[L::bTurn + (t ^ 1)]); };
            // Q.K^T of this tile into its S region; `pass` hands the turn on inside the batch
            auto issue_s = [&](int st, bool pass) {
                const uint64_t bd = dK0 + (uint64_t)((st * L::kKBytes) >> 4);
#pragma unroll
                for (int k = 0; k < D / 16; ++k) {
                    const uint64_t aoff = (uint64_t)((((k / 4) * (kTileM * 128)) + (k % 4) * 32) >> 4);
                    const uint64_t boff = (uint64_t)((((k / 4) * L::kKPanel) + (k % 4) * 32) >> 4);
                    if constexpr (PAIR)
                        mma_ss_pair(tS, dQt + aoff, bd + boff, idS, k > 0);
                    else
                        mma_ss(tS, dQt + aoff, bd + boff, idS, k > 0);
                    if (pass && k == D / 16 - 1 - kEarly) pass_turn();
                }
                commit_all<PAIR>(&bars[L::bSFull + t]);
            };
            auto issue_pv = [&](int st, bool acc, bool pass) {
                const uint64_t bd = dV0 + (uint64_t)((st * L::kVBytes) >> 4);
#pragma unroll
                for (int k = 0; k < kBlockN / 16; ++k) {
                    if constexpr (PAIR)
                        mma_ts_pair(tO, tS + k * 8, bd + (uint64_t)((k * 2048) >> 4), idO, (acc || k > 0) ? 1u : 0u);
                    else
                        mma_ts(tO, tS + k * 8, bd + (uint64_t)((k * 2048) >> 4), idO, (acc || k > 0) ? 1u : 0u);
                    if (pass && k == kBlockN / 16 - 1 - kEarly) pass_turn();
                }
            };
            // This tile's turn for its next slot (tile 0's very first slot needs none).
            int slots = 0;
            auto take_turn = [&]() -> bool {
                if (t == 0) return slots == 0 || fwait<PAIR>(&bars[L::bTurn + 0], (slots - 1) & 1, abort_flag);
                return fwait<PAIR>(&bars[L::bTurn + 1], slots & 1, abort_flag);
            };
            // This thread commits only the S-ready and O-done signals of its tile: the softmax
            // releases the ring stages and Q (a commit right behind another one holds the
            // issuing thread until the first has been delivered).
            bool ok = true;
            int gn = 0, pb = 0;   // blocks of the ring and of this tile before this item
            for (int j = 0; ok; ++j) {
                int idx;
                if (!fwd_read_item<PAIR>(item_bars, item_ring, j, abort_flag, idx)) break;
                mbar_arrive(&item_free[j & 3]);
                if (idx >= count) break;
                const FwdItem f = fwd_item<PAIR>(a, idx, 0);
                const int nbt = t ? f.nb1 : f.nb0;
                if (!fwait<PAIR>(&bars[L::bQFull], j & 1, abort_flag)) break;
                // slot 0: the first Q.K^T (the S region is free: this thread issued the previous
                // item's last P.V, which read it, before)
                if (nbt > 0 && !fwait<PAIR>(&bars[L::bKvFull + gn % S], (gn / S) & 1, abort_flag)) break;
                if (!take_turn()) break;
                if (nbt > 0) {
                    tc_fence_after();
                    issue_s(gn % S, true);
                } else {
                    pass_turn();
                }
                ++slots;
                for (int n = 0; ok && n < f.nmax; ++n) {
                    const int gb = gn + n, st = gb % S, st1 = (gb + 1) % S;
                    const bool has = n < nbt, more = n + 1 < nbt;   // a next Q.K^T of this tile reads block n+1
                    const uint32_t pph = (pb + n) & 1;
                    if (t == 0) USP_FTL(gb, 15);
                    // this tile's P, the next block's K and V, and this tile's turn (the other
                    // thread hands it over shortly before its batch ends), tested together
                    if (has) {
                        ok = mbar_wait3(&bars[L::bPFull + t], pph, more ? &bars[L::bKvFull + st1] : nullptr,
                                        ((gb + 1) / S) & 1, t == 0 && slots == 0 ? nullptr : &bars[L::bTurn + t],
                                        (t == 0 ? slots - 1 : slots) & 1, abort_flag, kWaitLimitNs);
                    } else {
                        ok = take_turn();
                    }
                    if (!ok) break;
                    USP_FTL(gb, 1 + t);
                    if (has) {
                        tc_fence_after();
                        issue_pv(st, n > 0, !more);
                        if (more) {
                            issue_s(st1, true);
                            USP_FTL(gb, 3 + t);
                        } else {
                            commit_all<PAIR>(&bars[L::bODone + t]);
                        }
                    } else {
                        pass_turn();
                    }
                    ++slots;
                }
                if (!ok) break;
                gn += f.nmax;
                pb += nbt;
            }
            // Drain: this thread's MMAs have run before TMEM is released.
            commit_all<PAIR>(&bars[L::bDrain + t]);
            mbar_wait_drain(&bars[L::bDrain + t], 0, kDrainLimitNs);
        }
    } else {
        regs_increase<kSoftmaxRegs>();
        // ------------------------------------------------------------------ softmax groups
        const int t = warp >> 2;
        const int rq = (warp & 3) * 32 + lane;
        const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
        const uint32_t tS = tbase + lane_off + t * 128;
        const uint32_t tO = tbase + lane_off + 256 + t * 128;
        const float sl2 = a.scale_log2;
        int pb = 0;   // this tile's blocks before the current item
        int od = 0;   // items before the current one in which this tile has blocks
        int gq = 0;   // ring blocks before the current item
        for (int j = 0;; ++j) {
            int idx = count;
            bool ok = fwd_read_item<PAIR>(item_bars, item_ring, j, abort_flag, idx);
            __syncwarp();
            if (ok && lane == 0) release_item_slot<PAIR>(&item_free[j & 3], rank);
            const FwdItem f = fwd_item<PAIR>(a, ok && idx < count ? idx : 0, rank);
            const int s = f.s, e = f.e, h = f.h;
            const int q0 = t ? f.q01 : f.q00;
            const int nbt = (ok && idx < count) ? (t ? f.nb1 : f.nb0) : 0;
            const int i = q0 + rq;  // this thread's query row
            // Each tile releases what its own MMA thread's MMAs read: once the group has seen
            // S(n) complete, this tile's Q.K^T and P.V of block n-1 have run (one thread's MMAs
            // run in issue order); its O-done covers its last block, and its last S its Q. A
            // block or a Q the other tile does not read (tile 0 has fewer blocks when nb0 < nb1,
            // tile 1 none when its rows lie past the sample's end) is released for both.
            const bool releaser = rq == 0;
            const int other_nb = (ok && idx < count) ? (t ? f.nb0 : f.nb1) : 0;
            auto rel_count = [&](int blk) -> uint32_t { return blk < other_nb ? 1u : 2u; };
            float m = -INFINITY, l = 0.f;
            for (int n = 0; n < nbt; ++n) {
                // (the warp agrees on the outcome: its tcgen05 loads and stores below are collective)
                if (!__all_sync(0xffffffffu, fwait<PAIR>(&bars[L::bSFull + t], (pb + n) & 1, abort_flag))) {
                    ok = false;
                    break;
                }
                if (releaser) {
                    if (n > 0) mbar_arrive_cnt(&bars[L::bKvEmpty + (gq + n - 1) % S], rel_count(n - 1));   // block n-1
                    if (n == nbt - 1) mbar_arrive_cnt(&bars[L::bQEmpty], other_nb > 0 ? 1u : 2u);          // Q
                }
                if (rq == 0) USP_FTL(pb + n, 5 + 4 * t);
                tc_fence_after();
                uint32_t r0[32], r1[32], r2[32], r3[32];
                tmem_ld32(tS + 0, r0);
                tmem_ld32(tS + 32, r1);
                tmem_ld32(tS + 64, r2);
                tmem_ld32(tS + 96, r3);
                tmem_ld_wait();
                reg_fence(r0);
                reg_fence(r1);
                reg_fence(r2);
                reg_fence(r3);
                float sv[128];
    #pragma unroll
                for (int c = 0; c < 32; ++c) {
                    sv[c] = __uint_as_float(r0[c]);
                    sv[32 + c] = __uint_as_float(r1[c]);
                    sv[64 + c] = __uint_as_float(r2[c]);
                    sv[96 + c] = __uint_as_float(r3[c]);
                }
                const int kv0 = s + n * kBlockN;
                const bool need_mask = (a.causal && kv0 + kBlockN - 1 > q0) || (kv0 + kBlockN > e);
                if (need_mask) {
                    int lim = e - 1 - kv0;  // last visible column of this block
                    if (a.causal && i - kv0 < lim) lim = i - kv0;
    #pragma unroll
                    for (int c = 0; c < 128; ++c)
                        if (c > lim) sv[c] = -INFINITY;
                }
                // the block's row max (log2 units) over 8 independent chains of three-input max (a
                // single two-input chain would serialise 127 dependent ops)
                auto block_max = [&]() -> float {
                    float mx8[8];
    #pragma unroll
                    for (int q = 0; q < 8; ++q) mx8[q] = sv[q];
    #pragma unroll
                    for (int c = 8; c < 120; c += 16)
    #pragma unroll
                        for (int q = 0; q < 8; ++q) mx8[q] = fmax3(mx8[q], sv[c + q], sv[c + 8 + q]);
    #pragma unroll
                    for (int q = 0; q < 8; ++q) mx8[q] = fmaxf(mx8[q], sv[120 + q]);
                    return fmax3(fmax3(mx8[0], mx8[1], mx8[2]), fmax3(mx8[3], mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7])) * sl2;
                };
                // P = exp2(s sl2 - m) into the S columns; returns the partial row sums
                auto exponentials = [&](float m_used) -> float2 {
                    const float mu = (m_used == -INFINITY) ? 0.f : m_used;
                    const float2 sl2x2 = make_float2(sl2, sl2), nmu2 = make_float2(-mu, -mu);
                    float2 l4[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                                    make_float2(0.f, 0.f)};
    #pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        uint32_t pk[16];
    #pragma unroll
                        for (int q = 0; q < 16; ++q) {
                            const float2 x = fma2(make_float2(sv[32 * c + 2 * q], sv[32 * c + 2 * q + 1]), sl2x2, nmu2);
                            const float2 pp = make_float2(ex2_approx(x.x), ex2_approx(x.y));
                            l4[q & 3] = add2(l4[q & 3], pp);   // independent partial row sums
                            pk[q] = pack2<F16>(pp.x, pp.y);
                        }
                        tmem_st16(tS + 16 * c, pk);
                    }
                    return add2(add2(l4[0], l4[1]), add2(l4[2], l4[3]));
                };
                const float m_blk = block_max();
                if (rq == 0) USP_FTL(pb + n, 6 + 4 * t);
                if (n == 0) {
                    m = m_blk;
                } else {
                    // tcgen05.ld / st are warp-collective: when any row of the warp moves its max,
                    // the whole warp rescales, each row by its own factor (1 for rows that keep
                    // theirs, which leaves their O bit-identical)
                    const bool up = m_blk > m + kRescaleThreshold;
                    if (__any_sync(0xffffffffu, up)) {
                        const float f = up ? ex2_approx(m - m_blk) : 1.f;
                        l *= f;
    #pragma unroll 1
                        for (int c = 0; c < D; c += 32) {
                            uint32_t o[32];
                            tmem_ld32(tO + c, o);
                            tmem_ld_wait(o);
                            uint32_t lo[16], hi[16];
    #pragma unroll
                            for (int q = 0; q < 16; ++q) {
                                lo[q] = __float_as_uint(__uint_as_float(o[q]) * f);
                                hi[q] = __float_as_uint(__uint_as_float(o[16 + q]) * f);
                            }
                            tmem_st16(tO + c, lo);
                            tmem_st16(tO + c + 16, hi);
                        }
                        if (up) m = m_blk;
                    }
                }
                const float2 lsum = exponentials(m);
                l += lsum.x + lsum.y;
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (rq == 0) USP_FTL(pb + n, 8 + 4 * t);
                if (lane == 0) arrive_leader<PAIR>(&bars[L::bPFull + t], rank);   // P ready for the tile's MMA thread
                if (rq == 0) USP_FTL(pb + n, 7 + 4 * t);

            }
            if (ok && nbt > 0) ok = __all_sync(0xffffffffu, fwait<PAIR>(&bars[L::bODone + t], od & 1, abort_flag));
            if (ok && releaser && nbt > 0)   // this tile's last block
                mbar_arrive_cnt(&bars[L::bKvEmpty + (gq + nbt - 1) % S], rel_count(nbt - 1));
            // The group's warps leave together (a warp that gave up on a wait must not leave the
            // others at the epilogue's barriers); the ring's end marker ends every warp's loop.
            if (group_any(1 + t, 128, !ok) || idx >= count) break;
            if (nbt > 0) ++od;
            if (nbt > 0 && q0 + kTileM <= e) {
                // Whole tile: O leaves through this tile's 64-column staging panel, 64 columns
                // per round, each round one TMA store (full lines instead of 16-byte pieces 256
                // bytes apart); the second round is packed into registers first.
                tc_fence_after();
                const float inv_l = (l > 0.f) ? 1.f / l : 0.f;
                uint8_t* stage = sm + L::kStage + t * (kTileM * 128);
                uint32_t held[32 * (D / 64 - 1) + 1];   // columns 64..D-1, two per word (none for D = 64)
                static_assert(D == 64 || D == 128, "the epilogue holds at most one extra 64-column panel");
#pragma unroll
                for (int c = 0; c < D / 32; ++c) {
                    uint32_t o[32];
                    tmem_ld32(tO + 32 * c, o);
                    tmem_ld_wait(o);
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const uint32_t p0 = pack2<F16>(__uint_as_float(o[8 * q]) * inv_l, __uint_as_float(o[8 * q + 1]) * inv_l);
                        const uint32_t p1 = pack2<F16>(__uint_as_float(o[8 * q + 2]) * inv_l, __uint_as_float(o[8 * q + 3]) * inv_l);
                        const uint32_t p2 = pack2<F16>(__uint_as_float(o[8 * q + 4]) * inv_l, __uint_as_float(o[8 * q + 5]) * inv_l);
                        const uint32_t p3 = pack2<F16>(__uint_as_float(o[8 * q + 6]) * inv_l, __uint_as_float(o[8 * q + 7]) * inv_l);
                        const int col = 32 * c + 8 * q;   // first of the 8 columns in this 16-byte chunk
                        if (col < 64) {
                            *(uint4*)(stage + sw128_offset(rq, (uint32_t)(col * 2))) = make_uint4(p0, p1, p2, p3);
                        } else if (D > 64) {
                            const int hi = (col - 64) / 2;
                            held[hi] = p0;
                            held[hi + 1] = p1;
                            held[hi + 2] = p2;
                            held[hi + 3] = p3;
                        }
                    }
                }
#pragma unroll 1
                for (int round = 0; round < D / 64; ++round) {
                    if (round > 0) {   // columns 64..127 into the panel the first store has released
#pragma unroll
                        for (int jj = 0; jj < 8; ++jj)
                            *(uint4*)(stage + sw128_offset(rq, (uint32_t)(jj * 16))) =
                                make_uint4(held[4 * jj], held[4 * jj + 1], held[4 * jj + 2], held[4 * jj + 3]);
                    }
                    fence_proxy_async_smem();
                    named_bar_sync(1 + t, 128);
                    if (rq == 0) {
                        tma_store_rows(&tmO, stage, round * 64, q0, h, a.token_major);
                        bulk_commit_group();
                        bulk_wait_group_read<0>();
                    }
                    named_bar_sync(1 + t, 128);
                }
                if (a.o_res) {
                    // The rounding residual O - round16(O) in two more rounds through the same
                    // panel, reading O from TMEM again: it stays there until this group's next
                    // P.V, which the tile's MMA thread issues only after the group's next P.
#pragma unroll 1
                    for (int round = 0; round < D / 64; ++round) {
#pragma unroll
                        for (int c = 0; c < 2; ++c) {
                            uint32_t o[32];
                            tmem_ld32(tO + round * 64 + 32 * c, o);
                            tmem_ld_wait(o);
#pragma unroll
                            for (int q = 0; q < 4; ++q) {
                                uint32_t r4[4];
#pragma unroll
                                for (int u = 0; u < 4; ++u) {
                                    const float x0 = __uint_as_float(o[8 * q + 2 * u]) * inv_l;
                                    const float x1 = __uint_as_float(o[8 * q + 2 * u + 1]) * inv_l;
                                    const float2 hv = unpack2<F16>(pack2<F16>(x0, x1));
                                    r4[u] = pack2<F16>(x0 - hv.x, x1 - hv.y);
                                }
                                *(uint4*)(stage + sw128_offset(rq, (uint32_t)((32 * c + 8 * q) * 2))) =
                                    make_uint4(r4[0], r4[1], r4[2], r4[3]);
                            }
                        }
                        fence_proxy_async_smem();
                        named_bar_sync(1 + t, 128);
                        if (rq == 0) {
                            tma_store_rows(&tmOres, stage, round * 64, q0, h, a.token_major);
                            bulk_commit_group();
                            bulk_wait_group_read<0>();
                        }
                        named_bar_sync(1 + t, 128);
                    }
                }
                a.lse[(int64_t)h * a.T + i] = (m + __log2f(l)) * 0.69314718055994530942f;
            } else if (nbt > 0) {   // a sample's ragged last tile: row by row, rows past the end skipped
                tc_fence_after();
                const bool valid = i < e;
                const float inv_l = (l > 0.f) ? 1.f / l : 0.f;
                const int64_t orow_off = act_row(h, i, a.T, a.hq, a.token_major) * D;
                uint16_t* orow = a.o + orow_off;
#pragma unroll 1
                for (int c = 0; c < D; c += 32) {
                    uint32_t o[32];
                    tmem_ld32(tO + c, o);
                    tmem_ld_wait(o);
                    uint32_t pk[16], rk[16];
#pragma unroll
                    for (int jj = 0; jj < 16; ++jj) {
                        const float x0 = __uint_as_float(o[2 * jj]) * inv_l, x1 = __uint_as_float(o[2 * jj + 1]) * inv_l;
                        pk[jj] = pack2<F16>(x0, x1);
                        const float2 hv = unpack2<F16>(pk[jj]);
                        rk[jj] = pack2<F16>(x0 - hv.x, x1 - hv.y);
                    }
                    if (valid) {
                        uint4* dst = (uint4*)(orow + c);
#pragma unroll
                        for (int jj = 0; jj < 4; ++jj)
                            dst[jj] = make_uint4(pk[4 * jj], pk[4 * jj + 1], pk[4 * jj + 2], pk[4 * jj + 3]);
                        if (a.o_res) {
                            uint4* rdst = (uint4*)(a.o_res + orow_off + c);
#pragma unroll
                            for (int jj = 0; jj < 4; ++jj)
                                rdst[jj] = make_uint4(rk[4 * jj], rk[4 * jj + 1], rk[4 * jj + 2], rk[4 * jj + 3]);
                        }
                    }
                }
                if (valid) a.lse[(int64_t)h * a.T + i] = (m + __log2f(l)) * 0.69314718055994530942f;
            }
            pb += nbt;
            gq += f.nmax;
        }
        if (rq == 0) bulk_wait_group<0>();   // the last output stores have landed
    }

    __syncwarp();
    tc_fence_before();
    __syncthreads();
    if constexpr (PAIR) {
        // neither CTA leaves (or frees tensor memory the pair's MMAs write) while the other may
        // still copy into it, arrive on its barriers or run MMAs on it
        cluster_sync_all();
        if (warp == 9) tmem_dealloc_pair(tbase, 512);
    } else {
        if (warp == 9) tmem_dealloc(tbase, 512);
    }
    if (threadIdx.x == 0 && *abort_flag) atomicCAS(&a.hdr->status, (int)USP_OK, (int)USP_ERR_TIMEOUT);
}

#ifdef USP_TIMELINE
}  // namespace
// The forward's timeline (kFTlCtas x kFTlSteps x kFTlEvents clock64 values) into host memory.
extern "C" int usp_debug_fwd_timeline(void* host_dst, size_t bytes) {
    if (bytes < sizeof(g_fwd_timeline)) return (int)USP_ERR_INVALID_ARG;
    return cudaMemcpyFromSymbol(host_dst, g_fwd_timeline, sizeof(g_fwd_timeline)) == cudaSuccess ? 0
                                                                                                 : (int)USP_ERR_CUDA;
}
namespace {
#endif

template <int D, bool F16, bool PAIR>
cudaError_t launch_fwd_impl(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v, const CUtensorMap& o,
                            const CUtensorMap& ores, const FwdArgs& a, int grid, cudaStream_t s) {
    using L = FwdSmem<D, PAIR>;
    if constexpr (PAIR) {
        // persistent pairs, one CTA per SM (the shared-memory footprint allows no more): as
        // many as can be resident at once
        int pairs_cap = 0;
        const cudaError_t e =
            persistent_cluster_setup<attn_fwd_kernel<D, F16, PAIR>>((size_t)L::kAlloc, kFwdThreads, 2, &pairs_cap);
        if (e != cudaSuccess) return e;
        const int pairs = grid < pairs_cap ? grid : pairs_cap;
        return launch_kernel_cluster(attn_fwd_kernel<D, F16, PAIR>, dim3(2 * pairs), dim3(kFwdThreads),
                                     (size_t)L::kAlloc, s, true, 2, q, k, v, o, ores, a);
    } else {
        // persistent CTAs, one per SM
        int sms = 0;
        const cudaError_t e = persistent_setup<attn_fwd_kernel<D, F16, PAIR>>((size_t)L::kAlloc, &sms);
        if (e != cudaSuccess) return e;
        if (grid > sms) grid = sms;
        return launch_kernel(attn_fwd_kernel<D, F16, PAIR>, dim3(grid), dim3(kFwdThreads), (size_t)L::kAlloc, s, true,
                             q, k, v, o, ores, a);
    }
}

}  // namespace

cudaError_t launch_attn_fwd(int head_dim, const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                            const CUtensorMap& o, const CUtensorMap& o_res, const FwdArgs& a, int grid,
                            cudaStream_t s) {
    static_assert(fwd_item_rows<true>() == fwd_rows_per_item(128) && fwd_item_rows<false>() == fwd_rows_per_item(64),
                  "the scheduler's forward items and the kernels' must agree");
    if (a.f16) {
        if (head_dim == 128) return launch_fwd_impl<128, true, true>(q, k, v, o, o_res, a, grid, s);
        return launch_fwd_impl<64, true, false>(q, k, v, o, o_res, a, grid, s);
    }
    if (head_dim == 128) return launch_fwd_impl<128, false, true>(q, k, v, o, o_res, a, grid, s);
    return launch_fwd_impl<64, false, false>(q, k, v, o, o_res, a, grid, s);
}

}  // namespace usp
