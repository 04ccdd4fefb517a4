// Internal interface between the C-ABI entry points (api.cu) and the kernel
// translation units.  Host-side only declarations; no torch types anywhere.
#pragma once
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/csa.h"

namespace csa {

// Validated layer dimensions.
struct Dims {
  int dtype, H, D, R, W, ratio, Hi, Di, topk, X;
  float scale, eps;
  int lanes;     // 2 when ratio == 4 (overlapping windows), else 1
  int rollback;  // tokens csa_trim may rewind
  int Wr;        // window ring slots: W + rollback (a query attends its last W tokens)
  int F;         // frontier ring slots: 2 ratio (ratio 4) or ratio, + rollback (the journal)
  int ikey_fp8;  // index keys as fp8 rows (CSA_FP8_ROW_BYTES each: 128 E4M3 codes of the rotated row, fp32 scale)
  bool has_indexer() const { return ratio == 4; }
};

// Carves 256-byte aligned sub-buffers out of the caller's workspace; with a
// null base it only measures.
struct Carver {
  char* base;
  size_t off = 0;
  explicit Carver(void* b) : base(static_cast<char*>(b)) {}
  template <typename E> E* take(size_t n) {
    off = (off + 255) & ~size_t(255);
    E* p = base ? reinterpret_cast<E*>(base + off) : nullptr;
    off += n * sizeof(E);
    return p;
  }
};

inline size_t esize(int dtype) { return dtype == CSA_BF16 ? 2 : 4; }

// Number of kernels this library has enqueued in this process (diagnostics).
void count_launches(int n);

// Launch with programmatic stream serialization (see pdl_trigger / pdl_wait).
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                              Args... args) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  count_launches(1);
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// The same with thread-block clusters of cluster_x consecutive blocks (grid.x a multiple of cluster_x).
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl_cluster(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                                      int cluster_x, Args... args) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = cluster_x;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  count_launches(1);
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

#define CSA_LAUNCH(...)                           \
  do {                                            \
    cudaError_t csa_e_ = launch_pdl(__VA_ARGS__); \
    if (csa_e_ != cudaSuccess) return csa_e_;     \
  } while (0)

// ---- compress.cu
struct CompressWs {
  int32_t* flags;  // [B] 1 = sequence valid for this call
  void* proj;      // [B*T, 2*L*d] model dtype: kv | gate of every new token
  float* part;     // tensor-core projection: split-K partials (or null)
  int* tickets;    // tensor-core projection: per-tile arrival counters (or null)
};
CompressWs carve_compress(Carver& c, const Dims& L, int d, int B, int T);
// The attention pool (ca, workspace wa) and the index pool (ci, wi) of one call's tokens.
cudaError_t launch_compress_pair(const Dims& L, const csa_compressor& ca, const csa_compressor& ci, const void* x,
                                 int B, int T, const int32_t* pos, void* fa, void* pa, int cap_a, int32_t* na,
                                 void* fi, void* pi, int cap_i, int32_t* ni, const float* inv_freq,
                                 const CompressWs& wa, const CompressWs& wi, int32_t* err, cudaStream_t s);
cudaError_t launch_compress(const Dims& L, const csa_compressor& comp, const void* x, int B, int T,
                            const int32_t* pos, void* frontier, void* pool, int cap, int32_t* n_rows,
                            const float* inv_freq, const CompressWs& ws, int32_t* err, cudaStream_t s);
// A packed variable-length batch: x [N, X], sequence b's chunk = rows cu[b] .. cu[b+1]-1 at positions pos[b] ..;
// ws carved for B sequences and N tokens (carve_compress(c, L, d, B, ceil(N / B)) is not enough: use
// carve_compress_varlen).  A sequence whose row-table entries are inconsistent is flagged CSA_DEV_STATE and left.
cudaError_t launch_compress_varlen(const Dims& L, const csa_compressor& comp, const void* x, int B,
                                   const int32_t* cu, int N, int T_max, const int32_t* pos, void* frontier,
                                   void* pool, int cap, int32_t* n_rows, const float* inv_freq,
                                   const CompressWs& ws, int32_t* err, cudaStream_t s);
CompressWs carve_compress_varlen(Carver& c, const Dims& L, int d, int B, int N);

// ---- indexer.cu
struct IndexWs {
  float* qr;      // [Q, Hi, Di] roped index queries (model-dtype values held as fp32)
  float* scores;  // [Q, cap]
};
IndexWs carve_index(Carver& c, const Dims& L, int Q, int cap);
// The indexer in two stages around `ready` (an event recorded after the index pool's compress call for the same
// token, possibly on another stream; null: no wait): the scan of the rows complete before the token, then,
// after the event, the rows that call may have written and the selection.  Decode, tensor-core shapes only;
// otherwise the whole call waits for the event and runs as launch_index_topk.
cudaError_t launch_index_topk_overlapped(const Dims& L, const void* iq, const void* iw, int Q, const void* ikeys,
                                         int cap, const int32_t* n_rows, const int32_t* pos, const float* inv_freq,
                                         int32_t* sel, int32_t* n_sel, const IndexWs& ws, int32_t* err,
                                         cudaStream_t s, cudaEvent_t ready);
// Scores and top-k for Q queries.  Query q belongs to sequence bseq(q) at position p(q): without pos, 0 and
// pos0 + q (one chunk); with pos, q / t and pos[q / t] + q % t, t = max(1, pos0) (decode, verify blocks); with
// cu (a packed variable-length batch of pos0 sequences, row table cu [pos0 + 1]), the b with cu[b] <= q <
// cu[b+1] and pos[b] + q - cu[b].  Its visible rows are min(n_rows[bseq], (p+1)/ratio).  sel [Q, topk], n_sel [Q].
cudaError_t launch_index_topk(const Dims& L, const void* iq, const void* iw, int Q, const void* ikeys, int cap,
                              const int32_t* n_rows, const int32_t* pos, int pos0, const float* inv_freq,
                              int32_t* sel, int32_t* n_sel, const IndexWs& ws, int32_t* err, cudaStream_t s,
                              const int32_t* cu = nullptr);

// ---- tc_project.cu (tensor-core compressor projections; bf16)
bool tc_project_supported(const Dims& L, int d);
void carve_tc_project(Carver& c, const Dims& L, int d, int ntok, float** part, int** tickets);
// K splits the projection of ntok tokens uses (1: proj is written directly).
int tc_project_splits(const Dims& L, int d, int ntok);
// Padded token count (rows of each split's partial block).
int tc_project_cols(const Dims& L, int d, int ntok);
// fixup = false (splits > 1): the fp32 partials [splits, ntok (padded), 2*L*d] are left for the consumer.
cudaError_t launch_tc_project(const Dims& L, int d, const void* x, int ntok, const void* wkv, const void* wgate,
                              void* proj, float* part, int* tickets, bool fixup, int32_t* err, cudaStream_t s);
// The index pool's and the attention pool's single-token projections as one grid (partials only; the pooling
// kernel sums them).  plan_project_pair picks the split counts (false: use two launches).
bool plan_project_pair(const Dims& L, int d0, int d1, int ntok, int* s0, int* s1);
cudaError_t launch_tc_project_pair(const Dims& L, int d0, const void* wkv0, const void* wg0, float* part0, int d1,
                                   const void* wkv1, const void* wg1, float* part1, const void* x, int ntok, int s0,
                                   int s1, int32_t* err, cudaStream_t s);

// ---- tc_indexer.cu (tensor-core scores; bf16, Hi = 64, Di = 128)
bool tc_index_supported(const Dims& L);
size_t tc_index_ws(const Dims& L, int Q);
// scores[q][j] for every q whose visible rows exceed topk; keys of query q are
// ikeys[pos ? q : 0]; ws needs tc_index_ws() bytes.
// overlap (decode only): score only rows < floor(pos/ratio) without reading n_rows, and leave the roped
// queries (bf16 [Q,64,128]) and scaled head weights (fp32 [Q,64]) at the start of ws for the selection stage.
cudaError_t launch_tc_index_scores(const Dims& L, const void* iq, const void* iw, int Q, const void* ikeys, int Bk,
                                   int cap, const int32_t* n_rows, const int32_t* pos, int pos0,
                                   const float* inv_freq, void* ws, float* scores, int32_t* err, cudaStream_t s,
                                   bool overlap = false, const int32_t* cu = nullptr, bool fp8 = false);

// ---- tc_attend.cu (tensor-core attention; bf16, H = 64, D = 512, R = 64)
bool tc_attend_supported(const Dims& L);
// Q queries (decode: pos[q], ring[q], pool[q]; prefill: pos == null, positions pos0 + q, batch 1, chunk rows
// kvr), S key splits per query: S > 1 writes (m, l, acc) partials, S == 1 the final output.
// Decode passes kv_new: the CTA that owns the new token's row ropes it and writes its ring slot.
cudaError_t launch_tc_attend(const Dims& L, const void* q, const void* pool, void* ring, const void* kvr,
                             const void* kv_new, const int32_t* sel, const int32_t* n_sel, const int32_t* n_rows,
                             const int32_t* pos, int pos0, int cap, const float* sink, const float* inv_freq, int Q,
                             int S, float* part_ml, float* part_acc, void* out, int32_t* err, cudaStream_t s);
// Merge of decode split partials for H % 8 == 0, D == 512 (one warp per head, 16 dims per lane).
// qps: consecutive queries per sequence (query q at pos[q / qps] + q % qps).
cudaError_t launch_tc_merge(const Dims& L, const float* part_ml, const float* part_acc, int S, int Q,
                            const float* sink, const int32_t* pos, const float* inv_freq, void* out, cudaStream_t s,
                            int qps = 1);

// ---- attend.cu: pos[b] += by for b < B
cudaError_t launch_advance_positions(int32_t* pos, int B, int by, cudaStream_t s);
// n rows of 128 bf16 values (src) -> n fp8 index rows of kFp8RowBytes (dst)
cudaError_t launch_index_rows_fp8(const void* src, long long n, void* dst, cudaStream_t s);
// ---- attend.cu: csa_trim (rewind B sequences by n_back tokens within the rollback margin)
cudaError_t launch_trim(const Dims& L, int B, const int32_t* n_back, int32_t* pos, int32_t* n_rows_a,
                        int32_t* n_rows_i, int32_t* hw, int32_t* err, cudaStream_t s);

// ---- tc_attend_prefill.cu (tensor-core chunked-prefill attention; bf16, H = 64, D = 512, R = 64)
// T queries of one sequence at positions pos0 + q; the chunk's roped rows kvr [T, D], the ring before the
// chunk, pool [cap, D]; persistent CTAs (one per SM) finalise the output.  Requires tc_attend_supported(L).
// With device positions (verify blocks): query q of sequence q / qps at pos[q / qps] + q % qps over pool
// [B, cap, D] and ring [B, Wr, D], every window token (the block's included) read from the ring; kvr unused.
// With a row table cu (a packed variable-length batch of qps chunks, T = N rows): query q of sequence b at
// pos[b] + q - cu[b]; tokens before pos[b] from the ring, the chunk's own from kvr [N, D] (roped).
cudaError_t launch_tc_attend_prefill(const Dims& L, const void* q, const void* pool, const void* ring,
                                     const void* kvr, const int32_t* sel, const int32_t* n_sel,
                                     const int32_t* n_rows, int pos0, int cap, const float* sink,
                                     const float* inv_freq, int T, void* out, int32_t* err, cudaStream_t s,
                                     const int32_t* pos = nullptr, int qps = 1, const int32_t* cu = nullptr);

// ---- tc_attend_decode.cu (tensor-core decode attention; bf16, H = 64, D = 512, R = 64)
bool tc_attend_decode_supported(const Dims& L);
// Key splits per query for Q queries over a window of W rows and at most n_max selected rows: each split's window
// share plus selection share fits one 160-row tile, more splits while every CTA still fits one wave; 0 when
// max_splits cannot hold enough splits.
int tc_attend_decode_splits(int Q, int W, int n_max, int max_splits);
// One CTA per (query, split).  S > 1 writes (m, l, acc) partials (merge follows), S == 1 the final output.
// Decode (qps 1): the new token kv_new[b] is roped in-kernel and written to ring slot pos[b] % Wr.  Verify blocks
// (qps tokens per sequence, kv_in_ring): query q belongs to sequence q / qps at pos[q / qps] + q % qps and every
// block token is already in the ring.
cudaError_t launch_tc_attend_decode(const Dims& L, const void* q, const void* pool, void* ring, const void* kv_new,
                                    const int32_t* sel, const int32_t* n_sel, const int32_t* n_rows,
                                    const int32_t* pos, int cap, const float* sink, const float* inv_freq, int Q,
                                    int S, float* part_ml, float* part_acc, void* out, int32_t* err, cudaStream_t s,
                                    int qps = 1, bool kv_in_ring = false, bool cluster = false);
// Whether S splits can merge inside a cluster (S in {2, 4} and the device places such clusters): the decode
// kernel then writes the output itself and no merge kernel runs.
bool tc_attend_decode_cluster(int S);

// ---- attend.cu
struct AttendWs {
  void* qr;        // [Q, H, D] roped queries, model dtype
  void* kvr;       // [T, D] roped chunk kv (prefill only)
  float* part_ml;  // [Q, S, H, 2] split partial (max, sum)
  float* part_acc; // [Q, S, H, D] split partial accumulators
  int S;           // splits per query
};
int attend_splits(const Dims& L, bool prefill, bool all_rows, int cap);
AttendWs carve_attend(Carver& c, const Dims& L, int Q, int S, int T);
// Decode: Q = B sequences, positions pos[b], window rings window[b].
cudaError_t launch_attend_decode(const Dims& L, const void* q, const void* kv_new, const float* sink, int B,
                                 void* window, const void* pool, int cap, const int32_t* n_rows, const int32_t* sel,
                                 const int32_t* n_sel, const int32_t* pos, const float* inv_freq, void* out,
                                 const AttendWs& ws, int32_t* err, cudaStream_t s);
// Prefill: T queries of one sequence at pos0 + t.  sel/n_sel from the indexer (or null: all visible rows).
cudaError_t launch_attend_prefill(const Dims& L, const void* q, const void* kv_new, const float* sink, int T,
                                  int pos0, void* window, const void* pool, int cap, const int32_t* n_rows,
                                  const int32_t* sel, const int32_t* n_sel, const float* inv_freq, void* out,
                                  const AttendWs& ws, int32_t* err, cudaStream_t s);

// A packed variable-length batch of B prefill chunks (row table cu [B + 1], N rows, the longest T_max): the rows
// are roped at their positions into ws.kvr, every query attends, then each sequence's last min(T_b, Wr) rows
// enter its ring.  Tensor-core shapes only.
cudaError_t launch_attend_prefill_varlen(const Dims& L, const void* q, const void* kv_new, const float* sink, int B,
                                         const int32_t* cu, int N, int T_max, void* window, const void* pool, int cap,
                                         const int32_t* n_rows, const int32_t* sel, const int32_t* n_sel,
                                         const int32_t* pos, const float* inv_freq, void* out, const AttendWs& ws,
                                         int32_t* err, cudaStream_t s);

// Verify blocks: T tokens per sequence appended to the window ring (roped), then each attended by its own query.
cudaError_t launch_attend_verify(const Dims& L, const void* q, const void* kv_new, const float* sink, int B, int T,
                                 void* window, const void* pool, int cap, const int32_t* n_rows, const int32_t* sel,
                                 const int32_t* n_sel, const int32_t* pos, const float* inv_freq, void* out,
                                 const AttendWs& ws, int32_t* err, cudaStream_t s);

}  // namespace csa
