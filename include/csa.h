/*
 * csa.h — C ABI of one layer of DeepSeek-V4 Compressed Sparse Attention (CSA)
 * on a single GB300 (sm_103a).
 *
 * The layer (DeepSeek-V4-Flash shapes) has four parts, each a call here:
 *   csa_compress_append      gated-pooling compressor: projects tokens, pools
 *                            ratio-4 overlapping or ratio-128 windows, RMSNorm,
 *                            RoPE at the window start, appends rows to a pool.
 *   csa_index_topk           indexer: ReLU-weighted multi-head scores of the
 *                            query against the index-key pool, exact top-k.
 *   csa_attend_decode        MQA-shaped attention of H heads over one shared
 *                            latent (K = V): selected pool rows + sliding
 *                            window, sink logits, split-K partial softmax and
 *                            merge, inverse RoPE on the output.
 *   csa_attend_prefill_chunk the same for a chunk of T queries of one
 *                            sequence, each with its own causal top-k.
 *   (*_varlen: a packed batch of chunks of different lengths; *_verify: verify
 *   blocks of T tokens per sequence; csa_trim: rewind for speculative decoding.)
 *
 * Definitions follow the pages the method is described on:
 *   [MTPLX#216]  "DeepSeek-V4-Flash: native deepseek_v4 AR backend"
 *   [mlx-lm#1189] "feat: add DeepSeek-V4 (Pro/Flash) model support"
 *   [v41-mlx]    "deepseek-v41-mlx" README
 *
 * Conventions for every call
 *   - Every tensor argument is a DEVICE pointer owned by the caller, dense,
 *     row-major, 16-byte aligned.  The library never allocates or frees device
 *     memory and keeps no state between calls.  Scratch memory comes from the
 *     caller through (ws, ws_bytes); csa_workspace_size() gives the size.
 *   - Storage dtype (layer->dtype): CSA_BF16 or CSA_F32 for activations,
 *     weights, pools, windows and outputs ("model dtype").  APE, norm weights,
 *     sink logits and the RoPE table are always fp32.  Arithmetic is fp32.
 *   - All work is enqueued asynchronously on `stream` (a cudaStream_t; NULL is
 *     the legacy default stream).  No call synchronises or reads device memory
 *     on the host, so calls can be captured in a CUDA graph.
 *   - Kernels are launched with programmatic dependent launch: each lets its
 *     successor in the stream start early and waits for its predecessor before
 *     reading anything that predecessor chain writes.  Before that wait a
 *     kernel may read its call's step inputs (queries, new tokens, weights,
 *     positions) and the window ring, so these must be complete when the call
 *     is enqueued behind work that does not trigger early (any ordinary kernel
 *     or copy; csa_advance_positions for pos).
 *   - Errors found on the host are returned synchronously, before anything is
 *     enqueued (fail closed: nothing is modified).  Errors that depend on
 *     device-resident values (positions, row counts, indices) are OR-ed into
 *     the caller's device error word `err` (CSA_DEV_* bits) and the offending
 *     sequence / row is skipped; no call traps or asserts on the device.
 *   - RoPE: rope dims are the LAST R dims of a row, rotated as interleaved
 *     pairs (D-R+2i, D-R+2i+1) by theta_i = (float)p * inv_freq[i] (one fp32
 *     multiply).  inv_freq is a device fp32 table of R/2 entries, so the
 *     caller chooses plain or YaRN-scaled frequencies ([mlx-lm#1189], OmarB97's
 *     RoPE fixes: the rotary setting depends on the layer kind, and compress
 *     layers use base 160000).
 */
#ifndef CSA_H
#define CSA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  CSA_OK = 0,
  CSA_ERR_ARG = 1,         /* null / misaligned pointer, inconsistent or out-of-range sizes */
  CSA_ERR_UNSUPPORTED = 2, /* valid arguments with no kernel for them (see each call) */
  CSA_ERR_CUDA = 3,        /* a kernel launch failed (cudaGetLastError after enqueue) */
  CSA_ERR_WORKSPACE = 4    /* ws_bytes smaller than csa_workspace_size() */
} csa_status;

enum { CSA_F32 = 0, CSA_BF16 = 1 };

/* bits of the device error word */
enum {
  CSA_DEV_CAPACITY = 1, /* a compress call would emit a row at index >= cap: sequence skipped */
  CSA_DEV_STATE = 2,    /* n_rows[b] != floor(pos[b] / ratio) or pos[b] < 0: sequence skipped */
  CSA_DEV_RANGE = 4,    /* a selected row index outside [0, n_rows[b]): that row is skipped */
  CSA_DEV_ROLLBACK = 8  /* csa_trim beyond the rollback margin (or below 0): sequence left unchanged */
};

/* operation ids for csa_workspace_size */
enum {
  CSA_OP_COMPRESS = 0,
  CSA_OP_INDEX_TOPK = 1,
  CSA_OP_ATTEND_DECODE = 2,
  CSA_OP_ATTEND_PREFILL = 3,
  CSA_OP_COMPRESS_PAIR = 4, /* csa_compress_append_pair (ratio-4 layers) */
  CSA_OP_COMPRESS_VARLEN = 5,       /* csa_compress_append_varlen: B sequences, T = N packed tokens */
  CSA_OP_ATTEND_PREFILL_VARLEN = 6  /* csa_attend_prefill_varlen: B sequences, T = N packed tokens */
};

/* One CSA layer.
 *   H query heads over one latent of D dims (K = V), rope on the last R dims;
 *   W-token sliding window; compress `ratio` (4: overlapping windows of 8
 *   tokens through two lanes, with the indexer; any other ratio r: one lane,
 *   non-overlapping windows of r tokens, no indexer); indexer Hi heads of Di
 *   dims keeping `topk` rows; hidden size X.
 *   scale: attention logit scale (the pages' kernels use D^-1/2; 0 selects it).
 *   rms_eps: RMSNorm epsilon of the compressed rows.
 *   rollback: tokens csa_trim may rewind (0: none).  The window ring then holds
 *     W + rollback slots (token t in slot t mod (W + rollback)) and each frontier
 *     ring csa_frontier_slots(ratio) + rollback slots (its journal of projected
 *     rows); a query still attends only its last W tokens.  Every call of a layer
 *     takes buffers of those sizes.
 *   index_fp8: 0 (index keys in the model dtype) or 1 (fp8 index rows of
 *     CSA_FP8_ROW_BYTES: the index pool, written by the compress calls and read
 *     by every index call (csa_index_topk, _verify, csa_attend_prefill_chunk,
 *     _varlen), is then a [B, cap, 144] byte tensor (a prefill chunk's ikeys
 *     [cap, 144]); ratio 4, bf16, Hi = 64, Di = 128 (D != 128), R <= 64 only,
 *     else CSA_ERR_UNSUPPORTED; csa_index_topk_overlapped returns
 *     CSA_ERR_UNSUPPORTED with it). */
typedef struct {
  int dtype;
  int H, D, R, W, ratio, Hi, Di, topk, X;
  float scale;
  float rms_eps;
  int rollback;
  int index_fp8;
} csa_layer;

/* Bytes of one index-key row when layer->index_fp8 = 1: the row (already in
 * the model dtype, as the bf16 format would store it) rotated by the
 * unnormalised 128-point Walsh-Hadamard transform (fp32 butterflies of span
 * 1, 2, .., 64), as 128 E4M3 codes of rotated / scale (nearest even,
 * saturating), then the fp32 scale = amax / 448 at byte 128, then padding.
 * The index queries are rotated and quantised per head the same way and a
 * score is the bf16 definition on the decoded values, divided by 128
 * ([mlx-lm#1189], the indexer thread: a Hadamard rotation and a low-precision
 * activation simulation in the indexer, the rotation cancelling in the dot
 * product; the format itself is this library's choice). */
#define CSA_FP8_ROW_BYTES 144

/* One compressor (the attention pool's, d = D, or the index pool's, d = Di).
 * L = 2 lanes when ratio == 4, else 1.
 *   wkv, wgate [L*d, X] model dtype (out-features x in-features);
 *   ape  [ratio, L*d] fp32: absolute position embedding added to the gates;
 *   norm_w [d] fp32: RMSNorm weight.
 * Lane 0 (first d outputs) pools the previous window, lane 1 the current one.
 * For the Flash ratio-4 attention pool that makes ape [4, 1024] and wkv, wgate
 * [1024, 4096] ([mlx-lm#1189], Thump604's fixes, on the overlap compressor's
 * weight shapes). */
typedef struct {
  const void* wkv;
  const void* wgate;
  const float* ape;
  const float* norm_w;
  int d;
} csa_compressor;

/* Frontier ring length in tokens without a rollback journal: 2*ratio when
 * ratio == 4, else ratio (a layer with rollback r adds r slots). */
int csa_frontier_slots(int ratio);

/* Bytes of scratch memory `op` needs for batch B (T: tokens per sequence for
 * CSA_OP_COMPRESS, chunk length for CSA_OP_ATTEND_PREFILL, else ignored) and
 * pool capacity `cap` rows.  Returns CSA_ERR_ARG on bad dimensions. */
csa_status csa_workspace_size(const csa_layer* layer, int op, int B, int T, int cap, size_t* bytes);

/* csa_compress_append — append T tokens per sequence to one compressed pool.
 *
 * Definition ([MTPLX#216] "What V4 adds": learned gated pooling over
 * overlapping ratio-4 or non-overlapping ratio-128 windows, maintained
 * incrementally by prefill and decode alike; [mlx-lm#1189] OmarB97's RoPE
 * fixes: a pool row is rotated when emitted; stepnoy "Fix" 3: the chunk tail is carried
 * and the absolute position accumulates; [MTPLX#216] "Decode path": the row is
 * pooled in fp32 and cast back before the norm):
 *   for token p = pos[b] + i:  kv_p = Wkv x_p,  g_p = Wgate x_p  (model dtype)
 *   when p = (j+1)*ratio - 1 completes window j:
 *     entries: ratio 4 -> tokens of window j-1 via lane 0 (absent for j = 0)
 *              and tokens of window j via lane 1; otherwise window j's tokens;
 *     per channel c: u_c = sum_e softmax_e(g_e,c + ape[t_e mod ratio][c]) kv_e,c
 *     row j = RoPE(RMSNorm(u), j*ratio), rounded to the model dtype at each step,
 *     written to pool[b][j]; n_rows[b] = j + 1.
 * Arguments
 *   x        [B, T, X]             model dtype, tokens at pos[b] .. pos[b]+T-1
 *   pos      [B] int32 (device)    position of x[b][0]; the library never writes it
 *   frontier [B, F, 2*L*d]         model dtype, F = csa_frontier_slots(ratio) + layer->rollback:
 *                                  ring of the projected (kv | gate) rows of the last F tokens,
 *                                  slot t mod F; read for tokens before pos[b], rewritten for the
 *                                  last tokens
 *   pool     [B, cap, d]           model dtype, rows [0, n_rows[b]) valid
 *   n_rows   [B] int32 (device)    in/out; must equal floor(pos[b] / ratio) on entry
 *   inv_freq [R/2] fp32
 *   err      int32 (device)        error word (CSA_DEV_STATE, CSA_DEV_CAPACITY); a sequence
 *                                  that would fail is left entirely unchanged
 * Call it once for the attention pool and, on ratio-4 layers, once for the
 * index pool, with the same pos and the same n_rows values. */
csa_status csa_compress_append(const csa_layer* layer, const csa_compressor* comp, const void* x, int B, int T,
                               const int32_t* pos, void* frontier, void* pool, int cap, int32_t* n_rows,
                               const float* inv_freq, void* ws, size_t ws_bytes, int32_t* err, void* stream);

/* csa_compress_append_pair — both compressed pools of a ratio-4 layer (the
 * attention pool, comp_a with d = D, and the index pool, comp_i with d = Di) for
 * the same T tokens per sequence: the arguments, errors and definition of
 * csa_compress_append for the attention pool and then for the index pool, with
 * each pool's own frontier, pool, cap and n_rows, and one shared x, pos,
 * inv_freq and error word.  Results are those two calls' (identical for T > 1;
 * for one token the projections' fp32 sums may be split differently along the
 * hidden axis, within the projection's own rounding).  The pages compress both pools from the same hidden
 * states at the same positions ([MTPLX#216] "What V4 adds": the indexer keeps
 * its own compressed keys beside the attention pool).  Workspace:
 * CSA_OP_COMPRESS_PAIR.  With one token per sequence (decode) the two
 * projections run as one kernel and the two pooling steps as one, so that
 * neither call waits behind the other; longer chunks run the two calls in turn.
 * CSA_ERR_UNSUPPORTED on layers without an indexer (ratio != 4). */
csa_status csa_compress_append_pair(const csa_layer* layer, const csa_compressor* comp_a,
                                    const csa_compressor* comp_i, const void* x, int B, int T, const int32_t* pos,
                                    void* frontier_a, void* pool_a, int cap_a, int32_t* n_rows_a, void* frontier_i,
                                    void* pool_i, int cap_i, int32_t* n_rows_i, const float* inv_freq, void* ws,
                                    size_t ws_bytes, int32_t* err, void* stream);

/* csa_index_topk — the indexer for one decode query per sequence.
 *
 * Definition ([mlx-lm#1189] stepnoy's patch point 3 and aidiffuser's indexer:
 * raw head weights with the scale folded in, no sigmoid, ReLU on the logits,
 * sum over heads; the index pool accumulates in the cache so its row space is
 * the attention pool's; OmarB97: row j is visible to position p iff
 * (j+1)*ratio <= p+1):
 *   n_vis = min(n_rows[b], floor((pos[b]+1)/ratio))
 *   q_h   = RoPE(iq[b][h], pos[b])  (model dtype)
 *   s_j   = sum_h iw[b][h] * Di^-1/2 * Hi^-1/2 * max(q_h . ikeys[b][j], 0),  j < n_vis
 *   if n_vis <= topk: sel = 0 .. n_vis-1; else the topk largest s_j, ties to
 *   the lower j.  sel is written in ascending row order, padded with -1.
 * Arguments
 *   iq [B, Hi, Di], iw [B, Hi]   model dtype
 *   ikeys [B, cap, Di]           model dtype index-key pool
 *   n_rows, pos [B] int32 (device)
 *   sel [B, topk] int32, n_sel [B] int32 (device outputs)
 * Requires ratio == 4 (the layers that carry an indexer) and topk <= 4096. */
csa_status csa_index_topk(const csa_layer* layer, const void* iq, const void* iw, int B, const void* ikeys, int cap,
                          const int32_t* n_rows, const int32_t* pos, const float* inv_freq, int32_t* sel,
                          int32_t* n_sel, void* ws, size_t ws_bytes, int32_t* err, void* stream);

/* csa_index_topk_overlapped — csa_index_topk split around the index pool's
 * compress call for the same token, so that the scan of the cached index keys
 * (the bulk of the call) runs while that compress call runs on another stream.
 * The pages define the same selection as csa_index_topk and have no such split:
 * it is a scheduling form of that call, with identical outputs up to the
 * floating-point order of the two rows scored in its second stage.
 *   stage 1 (enqueued on `stream` at once): s_j for rows j < floor(pos[b]/ratio),
 *     the rows complete before the token; reads neither n_rows nor any index-key
 *     row the concurrent compress call may write;
 *   then `stream` waits for `pool_ready` (a cudaEvent_t recorded after
 *     csa_compress_append for the index pool and this token; NULL: no wait);
 *   stage 2: s_j for row floor(pos[b]/ratio) and row n_rows[b]-1 (the rows that
 *     call may have written), then the selection exactly as csa_index_topk.
 * Arguments, workspace (CSA_OP_INDEX_TOPK) and errors as csa_index_topk; the
 * caller orders the compress call after any earlier use of the index pool, and
 * must not start another call that writes ikeys or n_rows for these sequences
 * before this one completes.  Shapes the tensor-core scan does not cover, or
 * cap > 16384, run the whole call after the event.
 * One stream, no event: enqueued right after csa_compress_append(_pair) for the
 * same token on the same stream, with pool_ready NULL, stage 1 runs beside that
 * call's kernels: it does not wait for the kernels before it (it reads only the
 * rows complete before the token and the step's inputs, and writes only its
 * workspace) and waits for them at its end, and the compress call's projection
 * kernel lets its successors start only once all earlier work in the stream
 * is complete.  Enqueued behind anything else, stage 1's inputs must be complete
 * and its workspace free when it is enqueued behind work that does not trigger
 * early. */
csa_status csa_index_topk_overlapped(const csa_layer* layer, const void* iq, const void* iw, int B, const void* ikeys,
                                     int cap, const int32_t* n_rows, const int32_t* pos, const float* inv_freq,
                                     int32_t* sel, int32_t* n_sel, void* ws, size_t ws_bytes, int32_t* err,
                                     void* stream, void* pool_ready);

/* csa_attend_decode — one decode query per sequence.
 *
 * Definition ([MTPLX#216] "What V4 adds": 64 query heads over one 512-dim
 * latent with per-head sink logits and a 128-token sliding window; [v41-mlx]:
 * the inverse rope on the attention output, sinks in the softmax denominator
 * only; [mlx-lm#1189] stepnoy: decode gathers its own top-k rows so the softmax
 * is not diluted over the whole pool):
 *   window[b][p mod W] = RoPE(kv_new[b], p)            p = pos[b]
 *   keys  = pool[b][sel[b][0 .. n_sel[b])]  (sel == NULL: rows 0 .. n_vis-1)
 *           ++ window tokens t in [max(0, p-W+1), p]
 *   l_ht  = scale * RoPE(q[b][h], p) . key_t
 *   o_h   = sum_t e^{l_ht} key_t / (e^{sink[h]} + sum_t e^{l_ht})
 *   out[b][h] = RoPE^-1(o_h, p)   (model dtype before and after the rotation)
 * computed as split-K partial softmaxes (m, l, acc) merged in a second pass.
 * Arguments
 *   q [B, H, D], kv_new [B, D]   model dtype
 *   sink [H] fp32
 *   window [B, Wr, D]            model dtype ring, Wr = W + layer->rollback, slot t mod Wr
 *                                (written at slot p mod Wr)
 *   pool [B, cap, D]             model dtype
 *   n_rows, n_sel, pos [B] int32 (device); sel [B, topk] int32 or NULL
 *   out [B, H, D]                model dtype
 * A selected index outside [0, n_rows[b]) raises CSA_DEV_RANGE and is skipped. */
csa_status csa_attend_decode(const csa_layer* layer, const void* q, const void* kv_new, const float* sink, int B,
                             void* window, const void* pool, int cap, const int32_t* n_rows, const int32_t* sel,
                             const int32_t* n_sel, const int32_t* pos, const float* inv_freq, void* out, void* ws,
                             size_t ws_bytes, int32_t* err, void* stream);

/* csa_attend_prefill_chunk — T queries of one sequence at positions pos0 .. pos0+T-1.
 *
 * The compressors must already have consumed the chunk (n_rows counts the rows
 * emitted up to its end).  Each query p attends the pool rows visible to it,
 * reduced by its OWN top-k when the layer has an indexer and more than topk
 * rows are visible ([mlx-lm#1189] stepnoy's patch point 3: per-query top-k
 * AND-ed with the visibility mask; aidiffuser: build the membership from the
 * index list rather than a dense compare), plus its window tokens: ring
 * entries for tokens before pos0, the chunk's own kv_new roped at their
 * positions otherwise.  After the chunk the window ring holds its last
 * W + rollback tokens.  Same formulas as csa_attend_decode / csa_index_topk per query.
 * Arguments
 *   q [T, H, D], kv_new [T, D], iq [T, Hi, Di], iw [T, Hi]   model dtype (iq, iw,
 *                                  ikeys may be NULL when ratio != 4)
 *   sink [H] fp32; pos0 host int; window [W + rollback, D]; pool [cap, D]; ikeys [cap, Di]
 *   n_rows int32 (device, one value)
 *   out [T, H, D]; sel_out [T, topk] int32 or NULL (the selected rows, -1 padded)
 * Requires 1 <= T <= 16384 and ratio == 4 or no indexer use. */
csa_status csa_attend_prefill_chunk(const csa_layer* layer, const void* q, const void* kv_new, const void* iq,
                                    const void* iw, const float* sink, int T, int32_t pos0, void* window,
                                    const void* pool, const void* ikeys, int cap, const int32_t* n_rows,
                                    const float* inv_freq, void* out, int32_t* sel_out, void* ws, size_t ws_bytes,
                                    int32_t* err, void* stream);

/* csa_compress_append_varlen, csa_attend_prefill_varlen — a packed batch of
 * prefill chunks of different lengths (ragged batched prefill): sequence b's
 * chunk is rows cu_seqlens[b] .. cu_seqlens[b+1]-1 of every packed tensor, at
 * positions pos[b] .. pos[b] + T_b - 1 (T_b = cu_seqlens[b+1] - cu_seqlens[b]).
 *
 * Definition: for every sequence, exactly csa_compress_append on its chunk (each
 * pool), then csa_attend_prefill_chunk on it with pos0 = pos[b] ([MTPLX#216]
 * "Verification": decode == prefill across chunked prefill and batching).  The
 * sequences share the launches: one projection over the N packed tokens, and
 * per-query scoring, top-k and attention over all of them.
 * Arguments
 *   x [N, X]; q [N, H, D]; kv_new [N, D]; iq [N, Hi, Di]; iw [N, Hi]   model dtype,
 *     packed (iq, iw, ikeys may be NULL when ratio != 4)
 *   cu_seqlens int32 [B + 1] (device): 0 = cu[0] <= cu[1] <= ... <= cu[B] = N
 *     (an empty chunk is allowed); T_max (host) >= every T_b sizes the grids
 *   pos int32 [B] (device): each chunk's first position; not advanced here
 *   frontier, pool, n_rows, window, ikeys: per sequence as for csa_compress_append
 *     and csa_attend_decode ([B, ...] with pool capacity cap)
 *   out [N, H, D]; sel_out [N, topk] int32 or NULL
 * Workspace: csa_workspace_size(.., CSA_OP_COMPRESS_VARLEN, B, N, cap, ..) and
 *   (.., CSA_OP_ATTEND_PREFILL_VARLEN, B, N, cap, ..).
 * Errors: as the single-chunk calls; N <= 2^20 for the compress call and
 *   N <= 16384 for the attention call (CSA_ERR_ARG beyond).  A row-table entry
 *   with cu[b] < 0, cu[b+1] < cu[b] or cu[b+1] > N is flagged CSA_DEV_STATE by
 *   the compress call, which leaves that sequence unchanged; every packed row
 *   index the attention call derives from the table is clamped into [0, N).
 *   The attention call needs the tensor-core shapes (bf16, H = 64, D = 512,
 *   R = 64; Hi = 64, Di = 128 with an indexer): CSA_ERR_UNSUPPORTED otherwise. */
csa_status csa_compress_append_varlen(const csa_layer* layer, const csa_compressor* comp, const void* x, int B,
                                      const int32_t* cu_seqlens, int N, int T_max, const int32_t* pos,
                                      void* frontier, void* pool, int cap, int32_t* n_rows, const float* inv_freq,
                                      void* ws, size_t ws_bytes, int32_t* err, void* stream);
csa_status csa_attend_prefill_varlen(const csa_layer* layer, const void* q, const void* kv_new, const void* iq,
                                     const void* iw, const float* sink, int B, const int32_t* cu_seqlens, int N,
                                     int T_max, const int32_t* pos, void* window, const void* pool,
                                     const void* ikeys, int cap, const int32_t* n_rows, const float* inv_freq,
                                     void* out, int32_t* sel_out, void* ws, size_t ws_bytes, int32_t* err,
                                     void* stream);

/* csa_index_topk_verify, csa_attend_verify — a verify block: T consecutive tokens
 * per sequence (a speculative step's last accepted token and its T-1 drafts),
 * each query with its own causal top-k and attention, B sequences at once.
 *
 * Definition ([MTPLX#216], "Benchmark notes" and the MTP post: verification runs
 * a K+1-wide query block per sequence, the KV projected inside a K+1-wide GEMM;
 * the per-query semantics are those of a prefill chunk, [mlx-lm#1189] stepnoy's
 * patch point 3): call csa_compress_append (or _pair) with the block's T tokens
 * first; then, for query i of sequence b at p = pos[b] + i, the selection and the
 * output are csa_index_topk's and csa_attend_decode's at position p, with the
 * rows visible at p (those emitted by tokens <= p) and the window tokens
 * [p-W+1, p], the block's own earlier tokens included.  csa_attend_verify first
 * writes all T tokens, roped, to their ring slots (pos[b] + i) mod (W + rollback),
 * so the layer needs rollback >= T - 1 (else CSA_ERR_ARG): the block's later
 * tokens must not overwrite window rows its earlier queries attend.  Neither call
 * advances pos; after verification the caller advances it by T (csa_advance_positions)
 * and rewinds the rejected drafts with csa_trim.
 * Arguments as csa_index_topk / csa_attend_decode with one more axis of T queries
 * per sequence: iq [B, T, Hi, Di], iw [B, T, Hi], q [B, T, H, D], kv_new [B, T, D],
 * sel [B, T, topk], n_sel [B, T], out [B, T, H, D]; pos [B] is the position of each
 * block's first token; 1 <= T <= 64.  Workspaces: csa_workspace_size(..,
 * CSA_OP_INDEX_TOPK, B * T, 1, cap, ..) and (.., CSA_OP_ATTEND_DECODE, B * T, ..).
 * Tensor-core shapes (bf16, 64 x 512 latent, 64 x 128 indexer) with an indexer
 * (ratio 4); other layers get CSA_ERR_UNSUPPORTED. */
csa_status csa_index_topk_verify(const csa_layer* layer, const void* iq, const void* iw, int B, int T,
                                 const void* ikeys, int cap, const int32_t* n_rows, const int32_t* pos,
                                 const float* inv_freq, int32_t* sel, int32_t* n_sel, void* ws, size_t ws_bytes,
                                 int32_t* err, void* stream);
csa_status csa_attend_verify(const csa_layer* layer, const void* q, const void* kv_new, const float* sink, int B, int T,
                             void* window, const void* pool, int cap, const int32_t* n_rows, const int32_t* sel,
                             const int32_t* n_sel, const int32_t* pos, const float* inv_freq, void* out, void* ws,
                             size_t ws_bytes, int32_t* err, void* stream);

/* csa_trim — rewind sequences by n_back[b] tokens, exactly (speculative decoding:
 * the rejected draft tokens are taken back).
 *
 * Definition ([MTPLX#216], the MTP / speculative-lane post: the cache trim rewinds
 * every lane exactly; emitted compressed rows are truncated, since a row depends
 * only on its one completed window; the compressor frontiers are rebuilt from a
 * bounded journal of their own projected rows; the sliding window keeps
 * rollback_capacity extra rows, since an evicted row cannot be recovered; asked
 * to go further, trim refuses instead of clamping).  Here the journal and the
 * extra window rows are the layer's rollback slots (csa_layer.rollback), so a
 * trim moves no data: with p = pos[b] and p' = p - n_back[b],
 *   hw[b]       = max(hw[b], p)          (the highest position the sequence reached)
 *   refuse      if n_back[b] < 0, p' < 0, p' < hw[b] - rollback, or n_rows[b] != p / ratio
 *   pos[b]      = p'
 *   n_rows[b]   = p' / ratio  (for n_rows_a and, when given, n_rows_i)
 * After it, decoding tokens from p' gives bit for bit what the sequence would
 * have given had the rewound tokens never been decoded: the frontier ring still
 * holds the projections of the ratio-window tokens before p', the window ring
 * the W tokens before p', and pool rows past the new n_rows are rewritten when
 * their windows complete again.
 * Arguments (device, int32 [B]): n_back; pos, n_rows_a (attention pool) and
 * n_rows_i (index pool; NULL for layers without an indexer) in/out; hw in/out,
 * caller-owned, set to the sequence's position when it starts (0 for a new one).
 * A refused sequence is left entirely unchanged and CSA_DEV_ROLLBACK (or
 * CSA_DEV_STATE) is OR-ed into err.  One small kernel on `stream`. */
csa_status csa_trim(const csa_layer* layer, int B, const int32_t* n_back, int32_t* pos, int32_t* n_rows_a,
                    int32_t* n_rows_i, int32_t* hw, int32_t* err, void* stream);

/* csa_index_topk_static — csa_index_topk without a caller-supplied workspace.
 *
 * No counterpart in the paper: this is a calling convention, not a step of the
 * method.  Some callers cannot allocate device memory at the point where they
 * run the indexer: code running inside a region whose allocator is frozen (a
 * serving engine that reserves all device memory up front and hands out no
 * scratch, or a runtime that forbids cudaMalloc and its implicit device-wide
 * synchronisation on a latency-critical decode path), or a plain C caller with
 * no allocator of its own.  This entry point takes its scratch memory from a
 * file-scope device array of csa_static_scratch_bytes() bytes (4 MiB) inside
 * the library; it allocates and frees nothing.
 *   - Arguments, results and errors are those of csa_index_topk, without ws.
 *   - Returns CSA_ERR_WORKSPACE when the call needs more scratch than the array
 *     holds (csa_workspace_size(..., CSA_OP_INDEX_TOPK, B, 1, cap) bytes; about
 *     B * (Hi*Di*4 + cap*4) — e.g. 32 sequences with 8400-row pools fit).
 *   - The first call on each device looks up the array's device address (with
 *     that device current) and keeps it together with the id of the device's
 *     CUDA context; make that first call before any stream capture.  A call in
 *     a context other than the one the address was found in (the device was
 *     reset and its context created again) looks it up again, since the array
 *     may then sit elsewhere: that call too should come before any capture.
 *   - Every call on a device shares the one array: calls whose kernels overlap
 *     on the GPU (different streams without ordering) race on it.  Calls in one
 *     stream are ordered and safe.  Nothing in the array needs to start at zero;
 *     it keeps the last call's contents.
 *   - Every GPU that loads the library holds the array until the process exits. */
size_t csa_static_scratch_bytes(void);
csa_status csa_index_topk_static(const csa_layer* layer, const void* iq, const void* iw, int B, const void* ikeys,
                                 int cap, const int32_t* n_rows, const int32_t* pos, const float* inv_freq,
                                 int32_t* sel, int32_t* n_sel, int32_t* err, void* stream);

/* Advance the positions of B sequences by `by` tokens: pos[b] += by, in one kernel
 * on `stream` (a device array of B int32, caller-owned).  A decode loop calls it
 * after the step's last library call (csa_attend_decode), since every call of a
 * step reads pos; it is not part of the method ("Decode path": the position of
 * the next token), only the loop's bookkeeping, launched like the library's
 * other kernels so that it may start while the step's last kernel finishes.
 * Unlike them it lets the next kernel start only once it has written pos, so
 * the next step's calls may read pos before their programmatic wait.
 * Errors: CSA_ERR_ARG for a null pos, B < 0; CSA_ERR_CUDA if the launch fails.
 * B == 0 enqueues nothing. */
csa_status csa_advance_positions(int32_t* pos, int B, int by, void* stream);

/* csa_index_rows_fp8 — index-key rows in the model dtype to fp8 index rows.
 *
 * src: n rows of Di = 128 bf16 values (an index pool written with index_fp8 = 0,
 * or rows from elsewhere; device, 16-byte aligned, caller-owned, read only);
 * dst: n rows of CSA_FP8_ROW_BYTES bytes (device, 16-byte aligned, caller-owned,
 * written).  Each row becomes exactly the row csa_compress_append would store
 * for it in a layer with index_fp8 = 1 (rotation, scale, E4M3 codes, zero
 * padding; see CSA_FP8_ROW_BYTES), so a cache built in the model dtype can be
 * carried over to the fp8 format.  Not a step of the method: a format
 * conversion.  The layer must have index_fp8 = 1 (else CSA_ERR_UNSUPPORTED).
 * Errors: CSA_ERR_ARG for n < 0 or n > 2^34, a null or misaligned pointer;
 * CSA_ERR_CUDA if the launch fails.  n == 0 enqueues nothing.  One kernel on
 * `stream`; src and dst must not overlap. */
csa_status csa_index_rows_fp8(const csa_layer* layer, const void* src, long long n, void* dst, void* stream);

/* Number of kernels this library has enqueued in this process (all calls,
 * all devices).  Diagnostic only: lets a caller count the launches of a region. */
unsigned long long csa_kernel_launches(void);

/* Human-readable name of a status code. */
const char* csa_status_string(csa_status s);

#ifdef __cplusplus
}
#endif
#endif /* CSA_H */
