/*
 * usp.h — C ABI of the GB300 Ulysses sequence-parallel attention hot path.
 *
 * The library emulates P sequence-parallel ranks inside one GPU's memory.  The
 * calls follow the attention wrapper of huggingface/accelerate PR #4209
 * ("Add an FSDP2-native Ulysses sequence parallelism backend"):
 *
 *   1. usp_relayout_fwd   q, k, v: "gather sequence, scatter heads"
 *                         (_gather_seq_scatter_heads, the all-to-all comment)
 *   2. usp_cu_seqlens_from_position_ids
 *                         document boundaries rebuilt from the *gathered*
 *                         position_ids, never the collator's per-shard
 *                         cu_seq_lens_q/k (the stale-kwargs comment: 41.8% of
 *                         logits mismatched with the per-shard ones)
 *   3. usp_attn_fwd       varlen causal GQA attention over the gathered
 *                         sequence, optional sliding window, one sink logit per
 *                         head sliced to the rank's heads (the gpt-oss finding)
 *   4. usp_relayout_bwd   the output: "gather heads, scatter sequence"
 *                         (_gather_heads_scatter_seq)
 *   backward: usp_relayout_fwd(dO), usp_attn_bwd, usp_relayout_bwd(dQ, dK, dV):
 *   the exchanges swap scatter and gather (same comment).
 *
 * Conventions shared by every call
 *   - Every pointer is a DEVICE pointer owned by the caller.  The library never
 *     allocates or frees device memory; scratch space is passed in as a
 *     workspace whose size a *_workspace_bytes query returns.
 *   - Every call only enqueues work on `stream` and returns without
 *     synchronising.  Results are valid once the stream reaches that point.
 *   - The return value reports host-side argument checks and launch errors.
 *     Data errors found on the device (stale or malformed cu_seqlens, negative
 *     position ids) are written to *dev_status (device int32, may be NULL)
 *     as a usp_status code; a call never clears *dev_status, so zero it
 *     before the first call and read it after synchronising.
 *   - Pointers passed to the relayout and attention calls must be 16-byte
 *     aligned (USP_ERR_ALIGNMENT otherwise).
 *   - Layout names:  seq-layout  [P][B][S/P][H][D]  rank r holds positions
 *                                 [r*S/P, (r+1)*S/P) of every row, all heads;
 *                    head-layout [P][B][S][H/P][D]  rank r holds every position,
 *                                 heads [r*H/P, (r+1)*H/P).
 *     Sequence chunks are contiguous in rank order, heads go to ranks in
 *     contiguous blocks, so rank r's query heads r*hq..r*hq+hq-1 read its own
 *     key/value heads under GQA.
 *   - The library is thread-safe per stream and keeps no state beyond a
 *     per-device cache of the SM count.
 */
#ifndef USP_H_
#define USP_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same object as cudaStream_t / CUstream; NULL is the legacy default stream. */
typedef struct CUstream_st* usp_stream_t;

typedef enum {
  USP_OK = 0,
  USP_ERR_INVALID_ARG = 1,   /* null pointer, non-positive size, bad flag */
  USP_ERR_INDIVISIBLE = 2,   /* P does not divide S, Hq or Hkv, or Hkv does not divide Hq
                                (accelerate PR #4209: "sp_size not dividing the heads" is refused) */
  USP_ERR_UNSUPPORTED = 3,   /* head dim, element size or size outside what the kernels take */
  USP_ERR_ALIGNMENT = 4,     /* pointer or contiguous run not a multiple of 16 bytes */
  USP_ERR_BAD_SEQLENS = 5,   /* device: cu_seqlens[0] != 0, not increasing, or cu_seqlens[n] != B*S
                                (e.g. a shard's stale per-shard boundaries) */
  USP_ERR_BAD_POSITIONS = 6, /* device: a negative position id */
  USP_ERR_TIMEOUT = 7,       /* device: a bounded wait inside a kernel gave up */
  USP_ERR_CUDA = 8,          /* a CUDA runtime/driver call or launch failed */
  USP_ERR_WORKSPACE = 9      /* workspace pointer null/misaligned or smaller than required */
} usp_status;

/* Static, human-readable name of a status code.  Never NULL. */
const char* usp_status_string(int status);

/* Library version as major*10000 + minor*100 + patch. */
int usp_version(void);

/* ------------------------------------------------------------------------
 * Relayout (the all-to-all of each rank, emulated as one permutation of the
 * P ranks' buffers).  accelerate PR #4209, the comment on the four
 * _SeqAllToAll.apply call sites: queries/keys/values go from the local
 * sequence chunk with all heads to the whole sequence with H/P heads, and the
 * output comes back per rank as its sequence chunk with the heads of every rank.
 *
 *   usp_relayout_fwd:  x_head[r][b][r'*S/P + s'][j][d] = x_seq[r'][b][s'][r*H/P + j][d]
 *   usp_relayout_bwd:  x_seq[r'][b][s'][r*H/P + j][d]  = x_head[r][b][r'*S/P + s'][j][d]
 *
 * x_seq:  [P][B][S/P][H][D] elements of elem_bytes bytes (input of fwd, output of bwd)
 * x_head: [P][B][S][H/P][D]                          (output of fwd, input of bwd)
 *
 * Fewer heads than ranks (H < P, P a multiple of H; kv-head replication, a
 * follow-up listed in PR #4209): every head is replicated on P/H ranks, rank r
 * holding head r / (P/H), so x_head is [P][B][S][1][D] and
 *   usp_relayout_fwd:  x_head[r][b][r'*S/P + s'][0][d] = x_seq[r'][b][s'][r / (P/H)][d]
 *   usp_relayout_bwd:  x_seq[r'][b][s'][h][d] = sum over the P/H ranks r with r / (P/H) == h of
 *                      x_head[r][b][r'*S/P + s'][0][d]
 * (the exchange back of a gradient is the adjoint of the copy: the replicas'
 * gradients add up).  The sum is taken in fp32 in rank order and rounded once;
 * it is defined for bf16 only (elem_bytes 2, else USP_ERR_UNSUPPORTED).
 *
 * The two buffers must not overlap.  Each contiguous run, (H/P)*D*elem_bytes
 * bytes (D*elem_bytes when replicated), must be a multiple of 16
 * (USP_ERR_ALIGNMENT otherwise).
 * Errors: USP_ERR_INVALID_ARG (null pointer, size <= 0, elem_bytes not 1/2/4/8),
 *         USP_ERR_INDIVISIBLE (S % P, or H % P when H >= P, or P % H when H < P),
 *         USP_ERR_ALIGNMENT, USP_ERR_UNSUPPORTED, USP_ERR_CUDA.
 * Apart from the replica sum the result is a bit-exact copy of every element.
 * ---------------------------------------------------------------------- */
int usp_relayout_fwd(const void* x_seq, void* x_head, int B, int S, int H, int D, int P,
                     int elem_bytes, usp_stream_t stream);
int usp_relayout_bwd(const void* x_head, void* x_seq, int B, int S, int H, int D, int P,
                     int elem_bytes, usp_stream_t stream);

/* Same permutation for three tensors in one launch: q (Hq heads) and k, v
 * (Hkv heads, replicated when Hkv < P), all with head dim D.  Equivalent to
 * three usp_relayout_fwd calls; meant for the q/k/v exchange of one attention
 * layer.  Hq % P != 0 is USP_ERR_INDIVISIBLE (query heads are never replicated). */
int usp_relayout_fwd_qkv(const void* q_seq, const void* k_seq, const void* v_seq,
                         void* q_head, void* k_head, void* v_head,
                         int B, int S, int Hq, int Hkv, int D, int P, int elem_bytes,
                         usp_stream_t stream);

/* ------------------------------------------------------------------------
 * One real rank's side of the exchanges, for P processes (one per GPU) that
 * run the all-to-all themselves (NCCL all_to_all_single, or any transport
 * that sends chunk p of a buffer to rank p and lays the received chunks out
 * in source-rank order).  accelerate PR #4209, the comment on the four
 * _SeqAllToAll.apply call sites: each rank sends every other rank that rank's
 * heads of its own sequence chunk and receives its own heads of every chunk;
 * the way back swaps scatter and gather.
 *
 * Shapes (Sl = S/P positions per rank, hpr = H/P heads per rank, or 1 with
 * H < P where each head is replicated on P/H ranks, rank p holding head
 * p / (P/H)):
 *   x_local [B][Sl][H][D]     the rank's sequence chunk, all heads
 *   x_head  [B][P*Sl][hpr][D] the whole sequence, the rank's heads (what
 *                             usp_attn_fwd/_bwd take with P = 1 and Hq/Hkv set
 *                             to the rank's head counts)
 *   send, recv [P][B][Sl][hpr][D]  chunk p goes to / came from rank p
 *
 *   usp_a2a_pack_seq_to_head:   send[p][b][s][j][d] = x_local[b][s][p*hpr + j][d]
 *                               (H < P: x_local[b][s][p / (P/H)][d])
 *   usp_a2a_unpack_seq_to_head: x_head[b][p*Sl + s][j][d] = recv[p][b][s][j][d]
 *   usp_a2a_pack_head_to_seq:   send[p][b][s][j][d] = x_head[b][p*Sl + s][j][d]
 *   usp_a2a_unpack_head_to_seq: x_local[b][s][p*hpr + j][d] = recv[p][b][s][j][d]
 *                               (H < P: x_local[b][s][h][d] = sum over the P/H ranks p
 *                               with p / (P/H) == h of recv[p][b][s][0][d], in fp32 in
 *                               rank order, rounded once; bf16 only)
 * With B == 1 the unpack after the seq->head exchange and the pack before the
 * head->seq exchange are plain copies (recv already is x_head, x_head already
 * is send), and a caller may skip them.  H is always the global head count.
 * Apart from the replica sum every result is a bit-exact copy.  Buffers must
 * not overlap; pointers and each contiguous run of hpr*D*elem_bytes bytes must
 * be 16-byte aligned.
 * Errors: USP_ERR_INVALID_ARG, USP_ERR_INDIVISIBLE (H and P), USP_ERR_ALIGNMENT,
 * USP_ERR_UNSUPPORTED, USP_ERR_CUDA.
 * ---------------------------------------------------------------------- */
int usp_a2a_pack_seq_to_head(const void* x_local, void* send, int B, int S_local, int H, int D, int P,
                             int elem_bytes, usp_stream_t stream);
int usp_a2a_unpack_seq_to_head(const void* recv, void* x_head, int B, int S_local, int H, int D, int P,
                               int elem_bytes, usp_stream_t stream);
int usp_a2a_pack_head_to_seq(const void* x_head, void* send, int B, int S_local, int H, int D, int P,
                             int elem_bytes, usp_stream_t stream);
int usp_a2a_unpack_head_to_seq(const void* recv, void* x_local, int B, int S_local, int H, int D, int P,
                               int elem_bytes, usp_stream_t stream);

/* ------------------------------------------------------------------------
 * Document boundaries from the gathered position_ids.  accelerate PR #4209:
 * position_ids are all-gathered once per forward in the model's pre-hook and
 * every layer reads them; the per-shard cu_seq_lens_q/k and max_length_q/k a
 * padding-free collator computed are dropped and rebuilt from the gathered
 * positions.
 *
 * pos:         int32 [P][B][S/P], each rank's shard.  The gathered sequence is
 *              gathered[b][r*S/P + s'] = pos[r][b][s'] (for B == 1 the buffer
 *              already *is* the gathered [S], byte for byte).
 * cu_seqlens:  int32, capacity B*S + 1 (output).  A document starts at every
 *              row start b*S and wherever the gathered position is 0.
 *              cu_seqlens[0] = 0, cu_seqlens[n_docs] = B*S, strictly increasing.
 * n_docs:      int32 device scalar (output): number of documents.
 * max_len:     int32 device scalar (output): longest document.
 * ws:          device workspace of at least usp_cu_seqlens_workspace_bytes(B, S)
 *              bytes, 16-byte aligned; its contents on entry do not matter.
 * dev_status:  device int32 (nullable): USP_ERR_BAD_POSITIONS if any position is
 *              negative (the outputs are then unspecified).
 * Output is bit-exact (integers).  Errors: USP_ERR_INVALID_ARG, USP_ERR_INDIVISIBLE
 * (S % P), USP_ERR_UNSUPPORTED (B*S >= 2^31 - 1), USP_ERR_WORKSPACE, USP_ERR_CUDA.
 * ---------------------------------------------------------------------- */
size_t usp_cu_seqlens_workspace_bytes(int B, int S);
int usp_cu_seqlens_from_position_ids(const int32_t* pos, int B, int S, int P,
                                     int32_t* cu_seqlens, int32_t* n_docs, int32_t* max_len,
                                     void* ws, size_t ws_bytes, int32_t* dev_status,
                                     usp_stream_t stream);

/* Same result as usp_cu_seqlens_from_position_ids, for callers that cannot
 * allocate device memory or hand over a workspace (for example code whose
 * device memory is entirely reserved by another allocator, or a plugin
 * interface that passes only input and output pointers).  It allocates
 * nothing: the scan's scratch lives in a fixed 64 KiB device array inside the
 * library, which every GPU that loads the library holds until the process
 * exits.  The pages have no counterpart of this call.
 *   - B*S may be at most 2^24 tokens; larger sizes return USP_ERR_UNSUPPORTED.
 *   - Every call looks up the array's device address on the current device
 *     (the first lookup on a device may load the library's device code
 *     there); make the first call on a device before any stream capture.
 *   - Every call shares the one array: calls whose kernels may overlap on the
 *     GPU (other streams, other host threads) race and must be ordered by the
 *     caller.  Leftover contents from an earlier call never matter.
 * Other arguments, outputs and errors are those of
 * usp_cu_seqlens_from_position_ids. */
int usp_cu_seqlens_from_position_ids_noalloc(const int32_t* pos, int B, int S, int P, int32_t* cu_seqlens,
                                             int32_t* n_docs, int32_t* max_len, int32_t* dev_status,
                                             usp_stream_t stream);

/* ------------------------------------------------------------------------
 * Attention over the gathered sequence, all P emulated ranks in one launch.
 *
 * For rank r, local query head j (global head r*hq + j, hq = Hq/P), its key/
 * value head j / (Hq/Hkv), token t of document [a, b): visible keys u are
 * a <= u <= t (causal; without causal a <= u < b) and t - u <= window_left
 * when window_left >= 0.  With s = softmax_scale * q_t . k_u and the sink
 * logit z = sinks[r*hq + j] (not scaled; absent when sinks == NULL):
 *     LSE_t = ln( sum_u exp(s_tu) + exp(z) )
 *     O_t   = sum_u exp(s_tu - LSE_t) v_u
 * (softmax over the keys plus one value-less sink logit; accelerate PR #4209,
 * the gpt-oss finding: each head has a single sink logit, so after the exchange
 * a rank uses the slice of the sinks for the heads it holds).
 * ---------------------------------------------------------------------- */
typedef struct {
  int B, S, Hq, Hkv, D, P;   /* global sizes; D must be 64 or 128 */
  int causal;                /* 1: causal mask inside each document; 0: full document */
  int window_left;           /* -1: none; else t - u <= window_left ("window 128" = 127) */
  float softmax_scale;       /* 0: 1/sqrt(D) */
  const int32_t* cu_seqlens; /* device int32 [n_docs+1], from usp_cu_seqlens_from_position_ids */
  const int32_t* n_docs;     /* device int32 scalar */
  const float* sinks;        /* device fp32 [Hq] (global heads), or NULL */
  int io_layout;             /* USP_IO_HEAD (0): q, k, v, dO, o, dq, dk, dv in head-layout;
                                USP_IO_SEQ (1): the same tensors in seq-layout — the exchanges
                                are fused into the kernels' loads and stores; needs (S/P) % 128 == 0;
                                USP_IO_SEQ_KV_HEAD (2, usp_attn_fwd only): q and o in seq-layout,
                                k and v in head-layout (the forward re-reads every k/v tile many
                                times, which runs faster from head-layout rows than from rows
                                strided over all key/value heads; the backward entry points
                                return USP_ERR_UNSUPPORTED for it) */
  int ring;                  /* ring x Ulysses hybrid: ring degree R (0 or 1: no ring).  With R > 1,
                                P is the Ulysses degree and a call computes one ring step: rows of
                                super-chunk a (S/R positions each) see only the keys of super-chunk
                                (a - ring_step) mod R.  The tensors are the hybrid head-layout of
                                usp_hybrid_relayout_fwd (USP_IO_HEAD) or the P*R sequence shards
                                [P*R][B][S/(P*R)][H][D] (USP_IO_SEQ, needs (S/(P*R)) % 128 == 0).
                                Needs (S/R) % 256 == 0. */
  int ring_step;             /* 0 <= ring_step < R */
  int head_first, head_count; /* usp_attn_bwd_dkdv / usp_attn_bwd_dq with USP_IO_SEQ only: process the
                                key/value heads [head_first, head_first + head_count) and their query
                                heads (0, 0: all), so that the stored dS of a long sequence can be
                                produced and consumed a group of heads at a time; every other entry
                                point needs 0, 0 */
} usp_attn_params;

enum { USP_IO_HEAD = 0, USP_IO_SEQ = 1, USP_IO_SEQ_KV_HEAD = 2 };

/* q:   bf16 head-layout [P][B][S][Hq/P][D];  k, v: bf16 [P][B][S][Hkv/P][D]
 *      (with io_layout = USP_IO_SEQ: seq-layout [P][B][S/P][Hq][D] and [P][B][S/P][Hkv][D],
 *      i.e. the shards each rank holds before the exchange; o then comes back in
 *      seq-layout too, exactly what usp_relayout_bwd of the head-layout o gives)
 * o:   bf16 head-layout like q (output)
 * lse: fp32 [P][B][Hq/P][S] natural-log LSE (output; includes the sink)
 * dev_status: nullable device int32; USP_ERR_BAD_SEQLENS when cu_seqlens does
 *   not start at 0, is not strictly increasing, or does not end at B*S (the
 *   outputs are then left unwritten).
 * Errors: USP_ERR_INVALID_ARG (also an unknown io_layout), USP_ERR_INDIVISIBLE,
 * USP_ERR_UNSUPPORTED (D not 64/128, window_left < -1, B*S >= 2^30 or
 * B*S*Hq >= 2^31, Hq > 1024, USP_IO_SEQ with (S/P) % 128 != 0), USP_ERR_ALIGNMENT,
 * USP_ERR_CUDA. */
int usp_attn_fwd(const usp_attn_params* params, const void* q, const void* k, const void* v,
                 void* o, float* lse, int32_t* dev_status, usp_stream_t stream);

/* ------------------------------------------------------------------------
 * Ring x Ulysses hybrid (USP; feifeibear/long-context-attention issue #135,
 * the device-mesh script: ranks form a (ring, ulysses) mesh with the Ulysses
 * dimension innermost and contiguous ("basic") sequence chunks).
 *
 * P = ring * ulysses ranks; rank p = rho*ulysses + u holds positions
 * [p*S/P, (p+1)*S/P).  The Ulysses exchange runs inside each ring group
 * rho, after which rank (rho, w) holds super-chunk rho (positions
 * [rho*C, (rho+1)*C), C = S/ring) for heads [w*H/U, (w+1)*H/U), U = ulysses.
 * The hybrid head-layout [U][B][S][H/U][D] lays the ring ranks' super-chunks
 * end to end for each w:
 *   x_head[w][b][rho*C + u*S/P + s'][j][d] = x_seq[rho*U + u][b][s'][w*H/U + j][d]
 * (H < U: replicated heads as in usp_relayout_fwd; the bwd exchange sums them).
 * ring = 1 is usp_relayout_fwd/bwd with P = ulysses.  Errors as usp_relayout_fwd,
 * with S % (ring*ulysses) for USP_ERR_INDIVISIBLE.
 * ---------------------------------------------------------------------- */
int usp_hybrid_relayout_fwd(const void* x_seq, void* x_head, int B, int S, int H, int D, int ring, int ulysses,
                            int elem_bytes, usp_stream_t stream);
int usp_hybrid_relayout_bwd(const void* x_head, void* x_seq, int B, int S, int H, int D, int ring, int ulysses,
                            int elem_bytes, usp_stream_t stream);
int usp_hybrid_relayout_fwd_qkv(const void* q_seq, const void* k_seq, const void* v_seq,
                                void* q_head, void* k_head, void* v_head,
                                int B, int S, int Hq, int Hkv, int D, int ring, int ulysses, int elem_bytes,
                                usp_stream_t stream);

enum { USP_RING_FIRST = 1, USP_RING_LAST = 2 };

/* Forward of one ring step's result into the running output: with the step's
 * o_step (bf16, head layout like o) and lse_step (fp32 [P][B][hq][S], -inf for
 * rows that saw no key) from usp_attn_fwd with params->ring_step = s:
 *   L = ln(e^L_acc + e^L_step),  O = e^(L_acc - L) O_acc + e^(L_step - L) O_step
 * o_step, o_acc and o share the layout params->io_layout names (the hybrid
 * head layout, or the sequence shards with USP_IO_SEQ); lse_* are always
 * [P][B][hq][S].
 * flags USP_RING_FIRST: the running values start as the step's (o_acc/lse_acc
 * are not read).  USP_RING_LAST: the sink logit z = sinks[r*hq + j] (if
 * params->sinks) joins once, L' = ln(e^L + e^z), O' = e^(L - L') O, and the
 * result goes to o (bf16) and lse (fp32), o_acc/lse_acc are not written;
 * otherwise it goes to o_acc (fp32, shaped like o) and lse_acc.  params is the
 * step call's (ring and ring_step are not read; sinks are, at the last step).
 * Pointers 16-byte aligned.  Errors: as usp_attn_fwd. */
int usp_ring_fwd_merge(const usp_attn_params* params, const void* o_step, const float* lse_step,
                       float* o_acc, float* lse_acc, void* o, float* lse, int flags, usp_stream_t stream);

/* Backward of the ring: g_acc (fp32) += g_step (bf16), n elements (a multiple
 * of 8).  USP_RING_FIRST: g_acc starts at zero (not read).  USP_RING_LAST: the
 * sum is rounded once to bf16 into g_out and g_acc is not written.  Every
 * step's dQ (kept by its rank) and dK/dV (carried with their super-chunk) is
 * summed at the element's own address.  Pointers 16-byte aligned.
 * Errors: USP_ERR_INVALID_ARG, USP_ERR_ALIGNMENT, USP_ERR_UNSUPPORTED (n/8 >= 2^32), USP_ERR_CUDA. */
int usp_ring_grad_accumulate(const void* g_step, float* g_acc, void* g_out, size_t n, int flags,
                             usp_stream_t stream);

/* Workspace that enables the faster backward: the dK/dV pass also stores dS
 * (bf16 blocks of [128 keys][64 queries] for every (query head, row, key tile,
 * query slice) pair a causal mask can reach) and the dQ pass computes
 * dQ = scale * dS K from them instead of recomputing S and dP.  Returns the
 * whole workspace size (the statistics of usp_attn_bwd_workspace_bytes plus
 * the blocks), or 0 when the shape has no such path (causal == 0, or S not a
 * multiple of 128).  The blocks' count depends only on the shape (the longest
 * possible document), so it is known without reading cu_seqlens.  Any
 * backward call given ws_bytes >= this size takes the stored-dS path; the
 * dK/dV and dQ calls of one backward must get the same ws and ws_bytes, with
 * the dK/dV call first. */
size_t usp_attn_bwd_fast_workspace_bytes(const usp_attn_params* params);
/* (With params->head_count > 0 the blocks are those of that head group, and
 * the dK/dV and dQ calls of the group use that workspace; the statistics
 * part still covers every head, as the preprocess writes it for all.) */

/* Bytes of workspace usp_attn_bwd needs: the fp32 row statistic
 * D_t = sum_d dO_td O_td for every query row and head, 256-byte aligned. */
size_t usp_attn_bwd_workspace_bytes(const usp_attn_params* params);

/* Gradients of usp_attn_fwd for the loss sum(O * dO):
 *   P_tu = exp(s_tu - LSE_t), dS_tu = P_tu (dO_t . v_u - D_t)
 *   dQ_t = scale sum_u dS_tu k_u,   dK_u = scale sum_t dS_tu q_t,
 *   dV_u = sum_t P_tu dO_t,         dsink = -sum_t exp(z - LSE_t) D_t
 * (key/value gradients sum over the query heads of their GQA group).
 * q, k, v, o, lse: the forward's inputs and outputs; dO: bf16 like o.
 * dq, dk, dv: bf16 outputs shaped like q, k, v.  dsinks: fp32 [Hq] output or
 * NULL (ignored when params->sinks is NULL).  ws: at least
 * usp_attn_bwd_workspace_bytes(params) bytes, 256-byte aligned.
 * The result is deterministic: no floating-point atomics.
 * Errors: as usp_attn_fwd, plus USP_ERR_WORKSPACE. */
int usp_attn_bwd(const usp_attn_params* params, const void* q, const void* k, const void* v,
                 const void* o, const float* lse, const void* dO,
                 void* dq, void* dk, void* dv, float* dsinks,
                 void* ws, size_t ws_bytes, int32_t* dev_status, usp_stream_t stream);

/* The three phases usp_attn_bwd runs, in order, each one kernel launch (the
 * preprocess adds one small reduction when sinks are given).  They are exposed
 * so that a caller can time them or place the two gradient passes, which only
 * read what the preprocess wrote, on different streams.  `ws` is
 * usp_attn_bwd's workspace: the preprocess writes D_t there, the gradient
 * passes read it.  Arguments and errors are as in usp_attn_bwd.
 *   usp_attn_bwd_preprocess: D_t = sum_d dO_td O_td; dsinks (nullable).
 *   usp_attn_bwd_dkdv:       dK, dV (every query head of each GQA group).
 *   usp_attn_bwd_dq:         dQ. */
int usp_attn_bwd_preprocess(const usp_attn_params* params, const void* o, const float* lse, const void* dO,
                            float* dsinks, void* ws, size_t ws_bytes, int32_t* dev_status, usp_stream_t stream);
int usp_attn_bwd_dkdv(const usp_attn_params* params, const void* q, const void* k, const void* v,
                      const float* lse, const void* dO, void* dk, void* dv, const void* ws, size_t ws_bytes,
                      int32_t* dev_status, usp_stream_t stream);
int usp_attn_bwd_dq(const usp_attn_params* params, const void* q, const void* k, const void* v,
                    const float* lse, const void* dO, void* dq, const void* ws, size_t ws_bytes,
                    int32_t* dev_status, usp_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* USP_H_ */
