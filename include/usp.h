/*
 * usp.h -- C ABI of libusp: the data-parallel hot path of Ulysses sequence
 * parallelism on one GB300 (sm_103a).
 *
 * Ulysses sequence parallelism splits a long sequence of T tokens over sp
 * ranks. Before attention each rank holds T/sp consecutive tokens with all H
 * heads; an all-to-all swaps the sharded dimension from sequence to heads, each
 * rank then computes ordinary attention over the full sequence for its H/sp
 * heads, and a second all-to-all swaps back (HF Transformers "Ulysses sequence
 * parallelism" guide, opening paragraph and layout figure; congresoia365
 * article "Nuevo método Ulysses...", section "Cómo Funciona Ulysses", steps
 * 1-5). Heads are independent, so the per-rank step is plain attention on a
 * subset of heads (same article, closing paragraph of that section).
 *
 * On one GPU the sp ranks are simulated as shards of one device buffer:
 *
 *   seq-sharded   [sp][T/sp][H][D]   (token-major; identical bytes to [T][H][D])
 *   head-sharded  [sp][H/sp][T][D]   (head-major;  identical bytes to [H][T][D])
 *
 * and the two all-to-alls become device-local permutations. No collective is
 * issued by this library.
 *
 * Conventions shared by every call:
 *   - The caller owns every buffer; the library never allocates device memory.
 *     Attention calls take a caller-provided workspace whose size is returned by
 *     usp_attn_workspace_size().
 *   - Pointers are device pointers, 16-byte aligned. `stream` is a cudaStream_t
 *     (NULL = legacy default stream). Calls are asynchronous on `stream`; the
 *     return value reports host-side validation and launch errors only. The
 *     first kernel of a call starts after all earlier work on `stream`; the
 *     call's later kernels are launched as programmatic dependents of the one
 *     before (they may start early and wait on the device for its results).
 *     Errors found on the device (malformed cu_seqlens, a wait that timed out)
 *     are written to the workspace status word; read it with
 *     usp_get_device_status().
 *   - No exception crosses the ABI. Calls are thread-safe as long as concurrent
 *     calls use distinct workspaces.
 *   - Every call launches on the device current on the calling thread. The
 *     kernels' shared-memory limits and the SM count are set up once per device
 *     (under a lock), so one process may drive several devices.
 */
#ifndef USP_H_
#define USP_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    USP_OK = 0,
    USP_ERR_INVALID_ARG = 1,  /* null/misaligned pointer, bad size, divisibility violated, overlap */
    USP_ERR_UNSUPPORTED = 2,  /* valid request this build does not implement (e.g. head_dim) */
    USP_ERR_CUDA = 3,         /* a CUDA runtime/driver call failed (launch, tensor map, attribute) */
    USP_ERR_WORKSPACE = 4,    /* workspace missing or smaller than usp_attn_workspace_size() */
    USP_ERR_TIMEOUT = 5,      /* device: a bounded wait inside a kernel expired; the kernel bailed out */
    USP_ERR_DEVICE_CHECK = 6  /* device: cu_seqlens malformed (cu[0] != 0, decreasing, cu[B] != T) */
} usp_status;

typedef enum { USP_BF16 = 0, USP_FP16 = 1, USP_FP32 = 2 } usp_dtype;

/*
 * usp_seq_to_head -- the first all-to-all of Ulysses (sequence -> heads), as a
 * device-local permutation over sp simulated ranks.
 *   Passage: HF Transformers "Ulysses sequence parallelism" guide, opening
 *   paragraph (the all-to-all moves the sharded dimension from sequence to
 *   attention heads) and its two-GPU layout figure; congresoia365 article,
 *   "Cómo Funciona Ulysses", step 3.
 *   out[r][hl][t][d] = in[t / S][t % S][r*Hl + hl][d],  S = T/sp, Hl = heads/sp.
 *   in   : [sp][S][heads][head_dim] elements of `dt` (read only)
 *   out  : [sp][Hl][T][head_dim]   elements of `dt` (written)
 *   The copy moves bits; `dt` only fixes the element size (2 or 4 bytes).
 * Errors: USP_ERR_INVALID_ARG if a pointer is NULL or not 16-byte aligned, the
 *   buffers overlap, sp < 1, total_tokens < 0, heads < 1, head_dim < 1,
 *   heads % sp != 0 (the head count must be divisible by sp_size: guide,
 *   "Configurar"), or total_tokens % sp != 0 (sequences are padded to a multiple
 *   of sp_size: same section). USP_ERR_UNSUPPORTED if a row (head_dim elements)
 *   is not a multiple of 16 bytes. total_tokens == 0 is a no-op (the buffers may
 *   then be NULL); the divisibility rules are still checked.
 */
usp_status usp_seq_to_head(const void* in, void* out, int sp, int64_t total_tokens, int heads,
                           int head_dim, usp_dtype dt, void* stream);

/*
 * usp_head_to_seq -- the second all-to-all (heads -> sequence), the inverse
 * permutation of usp_seq_to_head.
 *   Passage: guide, opening paragraph ("returns to the sequence-sharded
 *   layout") and the last row of its layout figure; congresoia365 article,
 *   step 5.
 *   out[t / S][t % S][r*Hl + hl][d] = in[r][hl][t][d].
 *   in : [sp][Hl][T][head_dim], out : [sp][S][heads][head_dim]. Same errors.
 */
usp_status usp_head_to_seq(const void* in, void* out, int sp, int64_t total_tokens, int heads,
                           int head_dim, usp_dtype dt, void* stream);

/*
 * usp_seq_to_head_kv / usp_head_to_seq_kv_grad -- the swaps for key/value heads,
 * including models with fewer key/value heads than ranks.
 *   Passage: HF Transformers guide, "Configurar" (heads must divide over sp_size);
 *   with GQA, query head h reads key/value head h / (hq / hkv). When hkv < sp
 *   (and sp % hkv == 0) each rank needs the one key/value head its query heads read,
 *   kv head r * hkv / sp, so every head is replicated sp / hkv times: this build's
 *   reading of the replication a GQA model needs for sp above its KV head count.
 *   hkv % sp == 0: identical to usp_seq_to_head / usp_head_to_seq.
 *   hkv < sp:  seq_to_head_kv writes out [sp][1][T][head_dim] with
 *              out[r][0][t] = in[t][r * hkv / sp];
 *              head_to_seq_kv_grad reads in [sp][1][T][head_dim] (per-rank gradients
 *              of the replicas) and writes out[t][g] = sum over the sp / hkv replicas
 *              of head g, accumulated in fp32 in rank order and rounded once
 *              (grad dt USP_BF16 or USP_FP32).
 * Errors: as usp_seq_to_head, and USP_ERR_INVALID_ARG when neither hkv % sp nor
 *   sp % hkv is 0; USP_ERR_UNSUPPORTED for an fp16 gradient sum.
 */
usp_status usp_seq_to_head_kv(const void* in, void* out, int sp, int64_t total_tokens, int hkv, int head_dim,
                              usp_dtype dt, void* stream);
usp_status usp_head_to_seq_kv_grad(const void* in, void* out, int sp, int64_t total_tokens, int hkv, int head_dim,
                                   usp_dtype dt, void* stream);

/*
 * usp_a2a_pack / usp_a2a_unpack -- the rank-local halves of Ulysses' all-to-all when the
 * ranks are real processes (one GPU each) and the exchange itself is a collective that
 * moves equal contiguous blocks (NCCL all-to-all; torch.distributed all_to_all_single).
 *   Passage: HF Transformers "Ulysses sequence parallelism" guide, opening paragraph and
 *   layout figure (each rank holds S = T/sp tokens with all heads before attention and
 *   all tokens of H/sp heads during it); congresoia365 article, "Cómo Funciona Ulysses",
 *   steps 3 and 5.
 *   usp_a2a_pack: in [S][heads][head_dim] (this rank's S = shard_tokens tokens) ->
 *     out [sp][S][nheads][head_dim], block r to be sent to rank r:
 *       out[r][s][j] = in[s][r*Hl + head0 + j], Hl = heads/sp, 0 <= head0,
 *       head0 + nheads <= Hl (a chunk of every rank's heads, so that the exchange of one
 *       chunk can overlap attention on another).
 *     After the collective the receive buffer [sp][S][nheads][D] is the token-major
 *     [T][nheads][D] layout the fused attention calls read (usp_ulysses_attn_fwd with
 *     sp = 1), and their token-major outputs go back as they are (block r' = the tokens
 *     of rank r').
 *   usp_a2a_unpack: in [sp][S][nheads][head_dim] received (block r from rank r) ->
 *     out [S][heads][head_dim]: out[s][r*Hl + head0 + j] = in[r][s][j]; heads outside the
 *     chunk are left untouched.
 *   Fewer key/value heads than ranks (heads < sp, sp % heads == 0; head0 = 0,
 *     nheads = 1): pack sends each rank the one head its query heads read,
 *     out[r][s][0] = in[s][r*heads/sp]; unpack receives the replicas' gradients and
 *     writes out[s][g] = the fp32 sum of in[r][s][0] over the sp/heads ranks r with
 *     r*heads/sp = g, in rank order, rounded once (dt USP_BF16 or USP_FP32).
 *   The copies move bits (dt fixes the element size) except for the replica sums.
 * Errors: USP_ERR_INVALID_ARG (NULL or misaligned pointer, overlapping buffers, sp < 1,
 *   shard_tokens < 0, heads neither dividing over sp nor dividing it, a head chunk
 *   outside the rank's heads); USP_ERR_UNSUPPORTED (a row not a multiple of 16 bytes,
 *   an fp16 replica sum). shard_tokens == 0 is a no-op.
 */
usp_status usp_a2a_pack(const void* in, void* out, int sp, int64_t shard_tokens, int heads, int head_dim,
                        int head0, int nheads, usp_dtype dt, void* stream);
usp_status usp_a2a_unpack(const void* in, void* out, int sp, int64_t shard_tokens, int heads, int head_dim,
                          int head0, int nheads, usp_dtype dt, void* stream);

/* ------------------------------------------------------------------------------
 * Ring-attention steps. In ring attention every rank keeps a chunk of the queries
 * while the key/value chunks travel around the ring; each step attends the local
 * queries to the visiting chunk and the partial results are combined through their
 * log-sum-exp (ColossalAI sequence parallelism tutorial, the ring-attention plugin
 * set-up and its closing comparison of Ulysses and ring attention). With equal chunks
 * of one sequence (packed samples split evenly, the same chunk-local cu_seqlens for
 * every chunk), the causal mask on global positions makes a step unmasked for an
 * earlier key chunk, causal for the query chunk's own keys and empty for a later one:
 * one attention call (causal 0 or 1) of this library, or none. The calls below do the
 * rest of a step; the Python class RingAttention chains them.
 * ------------------------------------------------------------------------------ */

/*
 * usp_lse_merge -- o_acc, lse_acc <- the softmax over the union of the keys seen so far
 * and a new disjoint key set, from each side's normalised output and log-sum-exp:
 *   lse = log(e^lse_acc + e^lse_part),
 *   o_acc = e^(lse_acc - lse) o_acc + e^(lse_part - lse) (o_part + o_part_res).
 *   A side with lse = -inf contributes nothing (both -inf: o 0, lse -inf).
 *   o_acc : fp32, o_part / o_part_res : dt (USP_BF16 or USP_FP16; o_part_res may be
 *   NULL), all [T][heads][head_dim] when token_major, else [heads][T][head_dim];
 *   lse_acc, lse_part : fp32 [heads][T] (natural log). init != 0: o_acc and lse_acc
 *   are set to the part (their contents are not read).
 * Errors: USP_ERR_INVALID_ARG (NULL or misaligned pointer, T < 0, heads < 1, head_dim
 *   not 64 or 128, dt not 16-bit). T == 0 is a no-op.
 */
usp_status usp_lse_merge(float* o_acc, float* lse_acc, const void* o_part, const void* o_part_res,
                         const float* lse_part, int64_t total_tokens, int heads, int head_dim, int token_major,
                         usp_dtype dt, int init, void* stream);

/*
 * usp_o_finalize -- o = round(o_acc) and o_res = round(o_acc - o) in dt (bf16 or fp16),
 * element by element (`elements` a multiple of 4; o_res may be NULL): the merged output
 * in the form the backward calls take (o and its rounding residual).
 */
usp_status usp_o_finalize(const float* o_acc, void* o, void* o_res, int64_t elements, usp_dtype dt, void* stream);

/*
 * usp_accumulate_f32 -- acc += part over `elements` fp32 values (a multiple of 4): sums
 * the gradient shares of the ring steps.
 */
usp_status usp_accumulate_f32(float* acc, const float* part, int64_t elements, void* stream);

/*
 * usp_attn_workspace_size -- bytes of workspace the attention calls need for
 * these sizes (bwd != 0: for usp_attn_bwd_varlen, which also needs per-row
 * Delta, an fp32 dQ accumulator and the fp16 copies of q, k, v and d_o). The workspace holds
 * a status word, the varlen work list and those buffers; it may be reused
 * across calls on the same stream and needs no initialisation: every call
 * writes each part of it before reading it.
 */
size_t usp_attn_workspace_size(int64_t total_tokens, int num_seqs, int hq, int hkv, int head_dim, int bwd);

/*
 * usp_attn_fwd_varlen -- local attention of one or more Ulysses ranks: causal,
 * sample-boundary-masked softmax attention over the full (packed) sequence
 * for the heads given.
 *   Passages: congresoia365 article, "Cómo Funciona Ulysses", step 4 (standard
 *   attention for the assigned heads over all positions) and "El Desafío..."
 *   (FlashAttention-style computation keeps memory O(n) without materialising
 *   the score matrix); HF guide, "Configurar" (packed samples must not attend
 *   across their boundaries; no dense 4-D mask).
 *   s_ij = scale * q_i . k_j; allowed(i,j) = same sample and (!causal or j <= i);
 *   lse_i = log sum_{allowed j} exp(s_ij);  o_i = sum_j exp(s_ij - lse_i) v_j.
 *   q   : bf16 [hq][T][head_dim]        k, v : bf16 [hkv][T][head_dim]
 *   o   : bf16 [hq][T][head_dim]        lse  : fp32 [hq][T] (natural log, includes scale)
 *   o_res : NULL, or bf16 [hq][T][head_dim]: the rounding residual of o, o_res =
 *         round(O - o) for the fp32 result O, so that o + o_res carries O to about 16
 *         significant bits. Passed on to the backward it makes Delta = dO . O exact to
 *         that precision instead of to bf16's 8 bits (a bf16 O alone puts an error of
 *         the order of the 2e-2 gradient tolerance into dS on short samples).
 *   cu_seqlens : device int32 [num_seqs + 1], cu[0] = 0, non-decreasing, cu[num_seqs] = T.
 *   Query head h reads key/value head h / (hq / hkv).
 *   softmax_scale <= 0 selects 1/sqrt(head_dim).
 *   The heads may be one rank's H/sp heads or all ranks' heads in one call.
 * Errors: USP_ERR_INVALID_ARG (NULL/misaligned pointer, T < 0, num_seqs < 1 when
 *   T > 0, hq or hkv < 1, hq % hkv != 0); USP_ERR_UNSUPPORTED (head_dim not 64
 *   or 128); USP_ERR_WORKSPACE (ws_bytes too small). Malformed cu_seqlens is
 *   detected on the device: the status word becomes USP_ERR_DEVICE_CHECK and
 *   no output is written. T == 0 is a no-op (the buffers may then be NULL).
 */
usp_status usp_attn_fwd_varlen(const void* q, const void* k, const void* v, void* o, void* o_res, float* lse,
                               const int32_t* cu_seqlens, int num_seqs, int64_t total_tokens, int hq,
                               int hkv, int head_dim, float softmax_scale, int causal, void* workspace,
                               size_t ws_bytes, void* stream);

/*
 * usp_attn_bwd_varlen -- gradient of usp_attn_fwd_varlen with respect to q, k
 * and v, from the saved logsumexp (the backward of the local attention step
 * each rank runs; the pages' training loops call it through backward()).
 *   dP_ij = dO_i . v_j; Delta_i = sum_j P_ij dP_ij (= dO_i . o_i);
 *   dS_ij = P_ij (dP_ij - Delta_i); dq_i = scale sum_j dS_ij k_j;
 *   dk_j = scale sum_i dS_ij q_i; dv_j = sum_i P_ij dO_i, where dk and dv of a
 *   key/value head sum over the hq/hkv query heads that read it.
 *   q, k, v, o, d_o : bf16 as in the forward; lse : fp32 [hq][T] from the forward;
 *   o_res : NULL or the forward's o_res (Delta is then taken from o + o_res).
 *   dq : [hq][T][head_dim], dk, dv : [hkv][T][head_dim] of grad_dt (USP_BF16 or USP_FP32).
 *   Precision: the call first copies q, k, v and d_o into the workspace as fp16, each
 *   scaled by a power of two per key/value group so that its largest magnitude lies in
 *   [8, 16); the products then round P and dS to fp16 (11 significant bits) and the
 *   results are scaled back exactly. Values must stay below 2^40 in magnitude.
 * Errors: as usp_attn_fwd_varlen; USP_ERR_UNSUPPORTED for grad_dt = USP_FP16.
 */
usp_status usp_attn_bwd_varlen(const void* q, const void* k, const void* v, const void* o,
                               const void* o_res, const float* lse, const void* d_o, void* dq, void* dk, void* dv,
                               usp_dtype grad_dt, const int32_t* cu_seqlens, int num_seqs,
                               int64_t total_tokens, int hq, int hkv, int head_dim, float softmax_scale,
                               int causal, void* workspace, size_t ws_bytes, void* stream);

/*
 * usp_ulysses_attn_fwd -- the forward attention step of Ulysses for all sp simulated
 * ranks with both layout swaps fused into the attention kernel: it reads the
 * seq-sharded q, k, v and writes the seq-sharded output, so the result equals
 * usp_seq_to_head on q, k and v, then usp_attn_fwd_varlen, then usp_head_to_seq on o,
 * without the four intermediate copies.
 *   Passages: as usp_seq_to_head, usp_attn_fwd_varlen and usp_head_to_seq. On one
 *   device the swap only changes which rows the kernel reads: head h of token t lives
 *   at row t*H + h of the seq-sharded buffer and at row h*T + t of the head-sharded
 *   one, whatever sp is.
 *   q   : dt [sp][T/sp][hq][D]        k, v : dt [sp][T/sp][hkv][D]
 *   o   : dt [sp][T/sp][hq][D]        lse  : fp32 [hq][T] (as usp_attn_fwd_varlen)
 *   o_res : NULL or dt [sp][T/sp][hq][D], the rounding residual of o (as usp_attn_fwd_varlen)
 *   dt  : USP_BF16 or USP_FP16, the type of q, k, v and o. Scores, softmax and the
 *         accumulators are fp32 either way; P is rounded to dt before the P.V MMA,
 *         whose operands must share a type. USP_FP32 returns USP_ERR_UNSUPPORTED.
 *   The workspace is that of usp_attn_fwd_varlen for the same sizes.
 * Errors: as usp_attn_fwd_varlen, and USP_ERR_INVALID_ARG when sp < 1, hq % sp or
 *   total_tokens % sp is non-zero (guide, "Configurar"), or when neither hkv % sp nor
 *   sp % hkv is zero. hkv < sp with sp % hkv == 0 is the replicated key/value case of
 *   usp_seq_to_head_kv: the kernels read each shared head in place.
 */
usp_status usp_ulysses_attn_fwd(const void* q, const void* k, const void* v, void* o, void* o_res, float* lse,
                                const int32_t* cu_seqlens, int num_seqs, int64_t total_tokens, int sp, int hq,
                                int hkv, int head_dim, float softmax_scale, int causal, usp_dtype dt,
                                void* workspace, size_t ws_bytes, void* stream);

/*
 * usp_ulysses_attn_bwd -- the backward attention step with the layout swaps fused:
 * the seq-sharded dO in, the seq-sharded dq, dk, dv out. Equals usp_seq_to_head on dO,
 * usp_attn_bwd_varlen (on the head-sharded q, k, v, o), then usp_head_to_seq on the
 * three gradients.
 *   q, o, d_o : dt [sp][T/sp][hq][D]; k, v : dt [sp][T/sp][hkv][D]; lse : fp32 [hq][T];
 *   o_res : NULL or the forward's o_res; dt USP_BF16 or USP_FP16 (the products run on the
 *   scaled fp16 copies of usp_attn_bwd_varlen either way).
 *   dq : [sp][T/sp][hq][D], dk, dv : [sp][T/sp][hkv][D] of grad_dt: dt or USP_FP32.
 *   The workspace is that of usp_attn_bwd_varlen for the same sizes.
 * Errors: as usp_attn_bwd_varlen, and the sp rules of usp_ulysses_attn_fwd.
 */
usp_status usp_ulysses_attn_bwd(const void* q, const void* k, const void* v, const void* o,
                                const void* o_res, const float* lse, const void* d_o, void* dq, void* dk, void* dv,
                                usp_dtype grad_dt, const int32_t* cu_seqlens, int num_seqs, int64_t total_tokens,
                                int sp, int hq, int hkv, int head_dim, float softmax_scale, int causal,
                                usp_dtype dt, void* workspace, size_t ws_bytes, void* stream);

/*
 * usp_get_device_status -- synchronises `stream`, then returns the status word
 * the last attention call on `workspace` left there (USP_OK,
 * USP_ERR_DEVICE_CHECK or USP_ERR_TIMEOUT), or USP_ERR_CUDA if the stream
 * reports an error. Does not clear the word; every attention call resets it.
 */
usp_status usp_get_device_status(const void* workspace, void* stream);

/*
 * usp_attn_fwd_varlen_noalloc -- usp_attn_fwd_varlen for callers that cannot
 * allocate device memory. This entry point is an addition of this library; the
 * pages have no counterpart to it.
 *   Who needs it: code inside a framework whose caching allocator owns all
 *   device memory and does not tolerate raw cudaMalloc/cudaFree next to it,
 *   real-time or embedded hosts that reserve a fixed memory budget up front and
 *   must not allocate per call, and plug-in code called through a hook that has
 *   no allocator handle and nowhere to keep a workspace between calls. None of
 *   them can provide the workspace the other attention calls take. Here the
 *   scratch data (status word, scheduler histogram, varlen work list) lives in
 *   a static 1 MiB array in the library's own device memory, which every GPU
 *   that loads the library holds until the process exits. The call allocates
 *   and frees nothing.
 *   Arguments, layouts and results are those of usp_attn_fwd_varlen, without
 *   the workspace. `status` (device int32, may be NULL) receives the
 *   device-side outcome once the call's kernels finish: USP_OK,
 *   USP_ERR_DEVICE_CHECK (malformed cu_seqlens; no output written) or
 *   USP_ERR_TIMEOUT.
 *   Set-up: the first call on each device looks up the array's device address
 *   (cudaGetSymbolAddress, with that device current) and sets the forward
 *   kernel's shared-memory limit there, which may load the library's device
 *   code; make that first call before any stream capture. Each device has its
 *   own array.
 *   Sharing: every call uses the same array, which keeps the previous call's
 *   contents (each call writes the parts it reads first). Calls whose
 *   kernels could overlap on the GPU (two streams, or two host threads without
 *   ordering) race on it; the caller must serialise them.
 * Errors: as usp_attn_fwd_varlen (the same host-side size checks), and
 *   USP_ERR_WORKSPACE when total_tokens > 2^30 or the work list for these sizes
 *   does not fit the 1 MiB array (roughly hq * (T/256 + num_seqs) above 60000
 *   items); no kernel is launched then.
 */
usp_status usp_attn_fwd_varlen_noalloc(const void* q, const void* k, const void* v, void* o, float* lse,
                                       const int32_t* cu_seqlens, int num_seqs, int64_t total_tokens, int hq,
                                       int hkv, int head_dim, float softmax_scale, int causal, int32_t* status,
                                       void* stream);

/* ------------------------------------------------------------------------------
 * Sample boundaries, label shift and loss over the SP ranks.
 *
 * Bookkeeping that the HF Transformers "Ulysses sequence parallelism" guide
 * (section on the Accelerate configuration file) lists around the attention:
 * position_ids generation, the label shift and the loss aggregation across SP
 * ranks. The jianying88 article on DeepSpeed Ulysses in Transformers (section
 * "3. 跨 rank 的加权 loss 聚合") defines the aggregation. Readings where the
 * pages leave a step open: position ids count up from 0 inside each packed
 * sample; a token's shifted label is the next token's label inside its sample
 * and -100 on the sample's last token; the weighted mean over zero good tokens
 * is 0. On one device the seq-sharded [sp][T/sp] buffers of all ranks are one
 * contiguous [T] buffer, so every call below takes all T tokens at once.
 * ------------------------------------------------------------------------------ */

/* Bytes of workspace usp_position_ids_to_cu_seqlens needs for total_tokens
 * (256 + 4 per 2048 tokens); 0 when total_tokens < 0. */
size_t usp_position_ids_workspace_size(int64_t total_tokens);

/*
 * usp_position_ids_to_cu_seqlens -- sample boundaries of a packed row from its
 * position ids, on the device, so that the attention can follow without a host
 * synchronisation.
 *   position_ids : int64[T] device (T = total_tokens < 2^31). A sample starts
 *                  wherever the id is 0; elsewhere the id must be the previous
 *                  token's id + 1.
 *   cu_seqlens   : int32[max_seqs + 1] device, written: the n sample starts,
 *                  then T in cu_seqlens[n..max_seqs]. Padding entries describe
 *                  empty samples, so the attention calls accept the array with
 *                  num_seqs = max_seqs.
 *   num_seqs     : int32 device (may be NULL): receives n.
 *   workspace    : device, 16-byte aligned, usp_position_ids_workspace_size
 *                  bytes; its first int32 is the status word read by
 *                  usp_get_device_status.
 *   All work is enqueued on `stream`; nothing is allocated.
 * Errors: USP_ERR_INVALID_ARG (NULL or misaligned pointer, T < 0 or >= 2^31,
 *   max_seqs < 1); USP_ERR_WORKSPACE. On the device: malformed ids set the status
 *   word to USP_ERR_DEVICE_CHECK and leave cu_seqlens and num_seqs unwritten; more
 *   than max_seqs samples set USP_ERR_DEVICE_CHECK, leave cu_seqlens unwritten and
 *   still write n to num_seqs. T = 0 writes cu_seqlens = 0 and n = 0.
 */
usp_status usp_position_ids_to_cu_seqlens(const int64_t* position_ids, int64_t total_tokens, int32_t* cu_seqlens,
                                          int max_seqs, int32_t* num_seqs, void* workspace, size_t workspace_bytes,
                                          void* stream);

/*
 * usp_cu_seqlens_to_position_ids -- position id of every token (its offset in its
 * own sample): position_ids[t] = t - cu_seqlens[b] for the sample b holding t.
 *   cu_seqlens   : int32[num_seqs + 1] device, non-decreasing, 0 first, T last
 *                  (empty samples allowed). A malformed array gives unspecified
 *                  ids, but every access stays in bounds.
 *   position_ids : int64[T] device, written.
 * Errors: USP_ERR_INVALID_ARG (NULL/misaligned pointer, num_seqs < 1 when T > 0,
 *   T < 0 or >= 2^31). T = 0 does nothing.
 */
usp_status usp_cu_seqlens_to_position_ids(const int32_t* cu_seqlens, int num_seqs, int64_t total_tokens,
                                          int64_t* position_ids, void* stream);

/*
 * usp_shift_labels -- labels shifted inside packed samples, and each SP rank's
 * count of good tokens.
 *   labels       : int64[T] device (-100 = ignored).
 *   cu_seqlens   : int32[num_seqs + 1] device, as for the attention calls.
 *   shift_labels : int64[T] device, written: shift[t] = labels[t+1] when t+1 is in
 *                  t's sample, else -100. Must not overlap `labels`.
 *   good_tokens  : int64[sp] device, written: good_tokens[r] = number of t in rank
 *                  r's shard [r*T/sp, (r+1)*T/sp) with shift[t] != -100.
 * Errors: USP_ERR_INVALID_ARG (NULL/misaligned pointer, overlap, sp < 1, T % sp,
 *   num_seqs < 1 when T > 0, T >= 2^31). A malformed cu_seqlens gives unspecified
 *   results with every access in bounds.
 */
usp_status usp_shift_labels(const int64_t* labels, const int32_t* cu_seqlens, int num_seqs, int64_t total_tokens,
                            int sp, int64_t* shift_labels, int64_t* good_tokens, void* stream);

/*
 * usp_sp_weighted_loss -- the loss of the whole SP group from each rank's loss and
 * good-token count: sum over ranks with good_tokens[r] > 0 of
 * rank_loss[r] * good_tokens[r], divided by the sum of good_tokens; 0 when no rank
 * has a good token. Ranks without good tokens are left out, so their loss (NaN for
 * a mean over nothing) does not reach the result. Accumulated in float64.
 *   rank_loss   : float32[sp] device;  good_tokens : int64[sp] device;
 *   loss        : float32 device, written.
 * Errors: USP_ERR_INVALID_ARG (NULL/misaligned pointer, sp < 1).
 */
usp_status usp_sp_weighted_loss(const float* rank_loss, const int64_t* good_tokens, int sp, float* loss,
                                void* stream);

/* Human-readable name of a status code (static string). */
const char* usp_status_string(usp_status status);

/*
 * usp_debug_wait_timeout -- launches one kernel that waits on an mbarrier that
 * nothing ever arrives on, with a wall-clock limit of `limit_ns`, and records
 * USP_ERR_TIMEOUT in the workspace status word when the limit expires. The
 * kernel then returns normally, so the CUDA context stays usable. Exists to
 * test the bounded-wait error path of the attention kernels without faulting
 * or hanging a GPU. limit_ns is clamped to [1e3, 5e9].
 */
usp_status usp_debug_wait_timeout(void* workspace, size_t ws_bytes, uint64_t limit_ns, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* USP_H_ */
