// C-ABI entry points: argument validation (fail closed, before any launch),
// workspace carving, dispatch to the kernel translation units.
#include <math.h>

#include "kernels.h"

#include <atomic>

using namespace csa;

static std::atomic<unsigned long long> g_launches{0};
void csa::count_launches(int n) { g_launches.fetch_add((unsigned long long)n, std::memory_order_relaxed); }

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }
bool dev_tensor(const void* p) { return p != nullptr && aligned16(p); }
bool dev_i32(const void* p) { return p != nullptr && aligned4(p); }

csa_status make_dims(const csa_layer* l, Dims* d) {
  if (!l) return CSA_ERR_ARG;
  if (l->dtype != CSA_F32 && l->dtype != CSA_BF16) return CSA_ERR_ARG;
  if (l->H < 1 || l->D < 8 || l->D % 8 || l->D > 1024) return CSA_ERR_ARG;
  if (l->R < 2 || l->R > l->D || l->R % 8 || (l->D - l->R) % 8) return CSA_ERR_ARG;
  if (l->W < 1 || l->ratio < 1 || l->X < 8 || l->X % 8) return CSA_ERR_ARG;
  if (l->ratio == 4) {
    if (l->Hi < 1 || l->Di < 8 || l->Di % 8 || l->R > l->Di || (l->Di - l->R) % 2) return CSA_ERR_ARG;
    if (l->topk < 1 || l->topk > 4096) return CSA_ERR_ARG;
  }
  if (!(l->rms_eps >= 0.f) || !(l->scale >= 0.f)) return CSA_ERR_ARG;
  if (l->rollback < 0 || l->rollback > (1 << 20)) return CSA_ERR_ARG;
  if (l->index_fp8 != 0 && l->index_fp8 != 1) return CSA_ERR_ARG;
  // (the index pool is told apart from the attention pool by its row length)
  if (l->index_fp8 && (l->ratio != 4 || l->dtype != CSA_BF16 || l->Hi != 64 || l->Di != 128 || l->D == l->Di ||
                       l->R > 64 || l->R % 8))
    return CSA_ERR_UNSUPPORTED;
  d->dtype = l->dtype;
  d->H = l->H; d->D = l->D; d->R = l->R; d->W = l->W; d->ratio = l->ratio;
  d->Hi = l->Hi; d->Di = l->Di; d->topk = l->topk; d->X = l->X;
  d->scale = l->scale > 0.f ? l->scale : (float)(1.0 / sqrt((double)l->D));
  d->eps = l->rms_eps;
  d->lanes = (l->ratio == 4) ? 2 : 1;
  d->rollback = l->rollback;
  d->Wr = l->W + l->rollback;
  d->F = csa_frontier_slots(l->ratio) + l->rollback;
  d->ikey_fp8 = l->index_fp8;
  return CSA_OK;
}

csa_status cuda_status(cudaError_t e) { return e == cudaSuccess ? CSA_OK : CSA_ERR_CUDA; }

size_t ws_compress(const Dims& L, int d, int B, int T) {
  Carver c(nullptr);
  carve_compress(c, L, d, B, T);
  return c.off;
}
size_t ws_compress_pair(const Dims& L, int B, int T) {
  Carver c(nullptr);
  carve_compress(c, L, L.D, B, T);
  carve_compress(c, L, L.Di, B, T);
  return c.off;
}
size_t ws_index(const Dims& L, int B, int cap) {
  Carver c(nullptr);
  carve_index(c, L, B, cap);
  return c.off;
}
size_t ws_decode(const Dims& L, int B, int cap) {
  Carver c(nullptr);
  carve_attend(c, L, B, attend_splits(L, false, !L.has_indexer(), cap), 0);
  return c.off;
}
void carve_prefill(Carver& c, const Dims& L, int T, int cap, IndexWs* iw, int32_t** sel, int32_t** n_sel,
                   AttendWs* aw) {
  if (L.has_indexer()) {
    *iw = carve_index(c, L, T, cap);
    *sel = c.take<int32_t>((size_t)T * L.topk);
    *n_sel = c.take<int32_t>(T);
  }
  *aw = carve_attend(c, L, T, attend_splits(L, true, false, cap), T);
}
size_t ws_compress_varlen(const Dims& L, int B, int N) {
  size_t best = 0;
  for (int d : {L.D, L.Di}) {
    if (d == L.Di && !L.has_indexer()) continue;
    Carver c(nullptr);
    carve_compress_varlen(c, L, d, B, N);
    best = c.off > best ? c.off : best;
  }
  return best;
}
size_t ws_prefill(const Dims& L, int T, int cap) {
  Carver c(nullptr);
  IndexWs iw{};
  int32_t *s = nullptr, *n = nullptr;
  AttendWs aw{};
  carve_prefill(c, L, T, cap, &iw, &s, &n, &aw);
  return c.off;
}

}  // namespace

extern "C" {

unsigned long long csa_kernel_launches(void) { return g_launches.load(std::memory_order_relaxed); }

int csa_frontier_slots(int ratio) { return ratio == 4 ? 2 * ratio : ratio; }

const char* csa_status_string(csa_status s) {
  switch (s) {
    case CSA_OK: return "CSA_OK";
    case CSA_ERR_ARG: return "CSA_ERR_ARG: invalid argument";
    case CSA_ERR_UNSUPPORTED: return "CSA_ERR_UNSUPPORTED: no kernel for these arguments";
    case CSA_ERR_CUDA: return "CSA_ERR_CUDA: kernel launch failed";
    case CSA_ERR_WORKSPACE: return "CSA_ERR_WORKSPACE: workspace too small";
  }
  return "unknown csa_status";
}

csa_status csa_workspace_size(const csa_layer* layer, int op, int B, int T, int cap, size_t* bytes) {
  Dims L;
  csa_status st = make_dims(layer, &L);
  if (st != CSA_OK) return st;
  if (!bytes || B < 1 || cap < 1) return CSA_ERR_ARG;
  switch (op) {
    case CSA_OP_COMPRESS:
      if (T < 1) return CSA_ERR_ARG;
      *bytes = ws_compress(L, L.D, B, T);
      if (L.has_indexer()) {
        const size_t bi = ws_compress(L, L.Di, B, T);
        if (bi > *bytes) *bytes = bi;
      }
      return CSA_OK;
    case CSA_OP_COMPRESS_PAIR:
      if (T < 1 || !L.has_indexer()) return CSA_ERR_ARG;
      *bytes = ws_compress_pair(L, B, T);
      return CSA_OK;
    case CSA_OP_INDEX_TOPK:
      *bytes = ws_index(L, B, cap);
      return CSA_OK;
    case CSA_OP_ATTEND_DECODE:
      *bytes = ws_decode(L, B, cap);
      return CSA_OK;
    case CSA_OP_ATTEND_PREFILL:
      if (T < 1 || T > 16384) return CSA_ERR_ARG;
      *bytes = ws_prefill(L, T, cap);
      return CSA_OK;
    case CSA_OP_COMPRESS_VARLEN:  // T: the batch's total tokens N
      if (T < 1 || T > (1 << 20)) return CSA_ERR_ARG;
      *bytes = ws_compress_varlen(L, B, T);
      return CSA_OK;
    case CSA_OP_ATTEND_PREFILL_VARLEN:  // T: the batch's total tokens N
      if (T < 1 || T > 16384) return CSA_ERR_ARG;
      *bytes = ws_prefill(L, T, cap);
      return CSA_OK;
  }
  return CSA_ERR_ARG;
}

// Argument checks shared by the one-pool and two-pool compress calls.
static bool compress_args_ok(const Dims& L, const csa_compressor* comp, int B, int T, int cap, const void* frontier,
                             const void* pool, const int32_t* n_rows) {
  if (!comp || B < 1 || T < 1 || cap < 1) return false;
  if (comp->d < L.R || comp->d % 8 || (comp->d != L.D && comp->d != L.Di)) return false;
  if (!dev_tensor(comp->wkv) || !dev_tensor(comp->wgate) || !dev_tensor(comp->ape) || !dev_tensor(comp->norm_w))
    return false;
  return dev_tensor(frontier) && dev_tensor(pool) && dev_i32(n_rows);
}

csa_status csa_compress_append(const csa_layer* layer, const csa_compressor* comp, const void* x, int B, int T,
                               const int32_t* pos, void* frontier, void* pool, int cap, int32_t* n_rows,
                               const float* inv_freq, void* ws, size_t ws_bytes, int32_t* err, void* stream) {
  Dims L;
  csa_status st = make_dims(layer, &L);
  if (st != CSA_OK) return st;
  if (!compress_args_ok(L, comp, B, T, cap, frontier, pool, n_rows)) return CSA_ERR_ARG;
  if (!dev_tensor(x) || !dev_tensor(inv_freq) || !dev_i32(pos) || !dev_i32(err)) return CSA_ERR_ARG;
  const size_t need = ws_compress(L, comp->d, B, T);
  if (ws_bytes < need || (need && !dev_tensor(ws))) return CSA_ERR_WORKSPACE;
  Carver c(ws);
  CompressWs w = carve_compress(c, L, comp->d, B, T);
  return cuda_status(launch_compress(L, *comp, x, B, T, pos, frontier, pool, cap, n_rows, inv_freq, w, err,
                                     static_cast<cudaStream_t>(stream)));
}

csa_status csa_compress_append_pair(const csa_layer* layer, const csa_compressor* comp_a,
                                    const csa_compressor* comp_i, const void* x, int B, int T, const int32_t* pos,
                                    void* frontier_a, void* pool_a, int cap_a, int32_t* n_rows_a, void* frontier_i,
                                    void* pool_i, int cap_i, int32_t* n_rows_i, const float* inv_freq, void* ws,
                                    size_t ws_bytes, int32_t* err, void* stream) {
  Dims L;
  csa_status st = make_dims(layer, &L);
  if (st != CSA_OK) return st;
  if (!L.has_indexer()) return CSA_ERR_UNSUPPORTED;
  if (!compress_args_ok(L, comp_a, B, T, cap_a, frontier_a, pool_a, n_rows_a) ||
      !compress_args_ok(L, comp_i, B, T, cap_i, frontier_i, pool_i, n_rows_i))
    return CSA_ERR_ARG;
  if (comp_a->d != L.D || comp_i->d != L.Di) return CSA_ERR_ARG;
  if (!dev_tensor(x) || !dev_tensor(inv_freq) || !dev_i32(pos) || !dev_i32(err)) return CSA_ERR_ARG;
  const size_t need = ws_compress_pair(L, B, T);
  if (ws_bytes < need || !dev_tensor(ws)) return CSA_ERR_WORKSPACE;
  Carver c(ws);
  const CompressWs wa = carve_compress(c, L, L.D, B, T);
  const CompressWs wi = carve_compress(c, L, L.Di, B, T);
  return cuda_status(launch_compress_pair(L, *comp_a, *comp_i, x, B, T, pos, frontier_a, pool_a, cap_a, n_rows_a,
                                          frontier_i, pool_i, cap_i, n_rows_i, inv_freq, wa, wi, err,
                                          static_cast<cudaStream_t>(stream)));
}

csa_status csa_index_topk(const csa_layer* layer, const void* iq, const void* iw, int B, const void* ikeys, int cap,
                          const int32_t* n_rows, const int32_t* pos, const float* inv_freq, int32_t* sel,
                          int32_t* n_sel, void* ws, size_t ws_bytes, int32_t* err, void* stream) {
  Dims L;
  csa_status st = make_dims(layer, &L);
  if (st != CSA_OK) return st;
  if (!L.has_indexer()) return CSA_ERR_UNSUPPORTED;
  if (B < 1 || cap < 1) return CSA_ERR_ARG;
  if (!dev_tensor(iq) || !dev_i32(iw) || !dev_tensor(ikeys) || !dev_tensor(inv_freq)) return CSA_ERR_ARG;
  if (!dev_i32(n_rows) || !dev_i32(pos) || !dev_i32(sel) || !dev_i32(n_sel) || !dev_i32(err)) return CSA_ERR_ARG;
  const size_t need = ws_index(L, B, cap);
  if (ws_bytes < need || !dev_tensor(ws)) return CSA_ERR_WORKSPACE;
  Carver c(ws);
  IndexWs w = carve_index(c, L, B, cap);
  return cuda_status(launch_index_topk(L, iq, iw, B, ikeys, cap, n_rows, pos, 0, inv_freq, sel, n_sel, w, err,
                                       static_cast<cudaStream_t>(stream)));
}

csa_status csa_index_topk_overlapped(const csa_layer* layer, const void* iq, const void* iw, int B, const void* ikeys,
                                     int cap, const int32_t* n_rows, const int32_t* pos, const float* inv_freq,
                                     int32_t* sel, int32_t* n_sel, void* ws, size_t ws_bytes, int32_t* err,
                                     void* stream, void* pool_ready) {
  Dims L;
  csa_status st = make_dims(layer, &L);
  if (st != CSA_OK) return st;
  if (!L.has_indexer() || L.ikey_fp8) return CSA_ERR_UNSUPPORTED;
  if (B < 1 || cap < 1) return CSA_ERR_ARG;
  if (!dev_tensor(iq) || !dev_i32(iw) || !dev_tensor(ikeys) || !dev_tensor(inv_freq)) return CSA_ERR_ARG;
  if (!dev_i32(n_rows) || !dev_i32(pos) || !dev_i32(sel) || !dev_i32(n_sel) || !dev_i32(err)) return CSA_ERR_ARG;
  const size_t need = ws_index(L, B, cap);
  if (ws_bytes < need || !dev_tensor(ws)) return CSA_ERR_WORKSPACE;
  Carver c(ws);
  IndexWs w = carve_index(c, L, B, cap);
  return cuda_status(launch_index_topk_overlapped(L, iq, iw, B, ikeys, cap, n_rows, pos, inv_freq, sel, n_sel, w,
                                                  err, static_cast<cudaStream_t>(stream),
                                                  static_cast<cudaEvent_t>(pool_ready)));
}

csa_status csa_attend_decode(const csa_layer* layer, const void* q, const void* kv_new, const float* sink, int B,
                             void* window, const void* pool, int cap, const int32_t* n_rows, const int32_t* sel,
                             const int32_t* n_sel, const int32_t* pos, const float* inv_freq, void* out, void* ws,
                             size_t ws_bytes, int32_t* err, void* stream) {
  Dims L;
  csa_status st = make_dims(layer, &L);
  if (st != CSA_OK) return st;
  if (B < 1 || cap < 1) return CSA_ERR_ARG;
  if (!dev_tensor(q) || !dev_tensor(kv_new) || !dev_i32(sink) || !dev_tensor(window) || !dev_tensor(pool) ||
      !dev_tensor(inv_freq) || !dev_tensor(out))
    return CSA_ERR_ARG;
  if (!dev_i32(n_rows) || !dev_i32(pos) || !dev_i32(err)) return CSA_ERR_ARG;
  if (sel && (!dev_i32(sel) || !dev_i32(n_sel))) return CSA_ERR_ARG;
  if (sel && !L.has_indexer()) return CSA_ERR_ARG;
  const size_t need = ws_decode(L, B, cap);
  if (ws_bytes < need || !dev_tensor(ws)) return CSA_ERR_WORKSPACE;
  Carver c(ws);
  AttendWs w = carve_attend(c, L, B, attend_splits(L, false, !L.has_indexer(), cap), 0);
  return cuda_status(launch_attend_decode(L, q, kv_new, sink, B, window, pool, cap, n_rows, sel, n_sel, pos,
                                          inv_freq, out, w, err, static_cast<cudaStream_t>(stream)));
}

csa_status csa_attend_prefill_chunk(const csa_layer* layer, const void* q, const void* kv_new, const void* iq,
                                    const void* iw, const float* sink, int T, int32_t pos0, void* window,
                                    const void* pool, const void* ikeys, int cap, const int32_t* n_rows,
                                    const float* inv_freq, void* out, int32_t* sel_out, void* ws, size_t ws_bytes,
                                    int32_t* err, void* stream) {
  Dims L;
  csa_status st = make_dims(layer, &L);
  if (st != CSA_OK) return st;
  if (T < 1 || T > 16384 || pos0 < 0 || cap < 1) return CSA_ERR_ARG;
  if (!dev_tensor(q) || !dev_tensor(kv_new) || !dev_i32(sink) || !dev_tensor(window) || !dev_tensor(pool) ||
      !dev_tensor(inv_freq) || !dev_tensor(out))
    return CSA_ERR_ARG;
  if (!dev_i32(n_rows) || !dev_i32(err)) return CSA_ERR_ARG;
  if (L.has_indexer() && (!dev_tensor(iq) || !dev_i32(iw) || !dev_tensor(ikeys))) return CSA_ERR_ARG;
  if (sel_out && !dev_i32(sel_out)) return CSA_ERR_ARG;
  const size_t need = ws_prefill(L, T, cap);
  if (ws_bytes < need || !dev_tensor(ws)) return CSA_ERR_WORKSPACE;
  Carver c(ws);
  IndexWs iws{};
  int32_t *sel = nullptr, *n_sel = nullptr;
  AttendWs aw{};
  carve_prefill(c, L, T, cap, &iws, &sel, &n_sel, &aw);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (L.has_indexer()) {
    if (sel_out) sel = sel_out;
    cudaError_t e = launch_index_topk(L, iq, iw, T, ikeys, cap, n_rows, nullptr, pos0, inv_freq, sel, n_sel, iws,
                                      err, s);
    if (e != cudaSuccess) return CSA_ERR_CUDA;
  } else if (sel_out && L.topk > 0) {
    cudaMemsetAsync(sel_out, 0xff, (size_t)T * L.topk * sizeof(int32_t), s);
  }
  return cuda_status(launch_attend_prefill(L, q, kv_new, sink, T, pos0, window, pool, cap, n_rows,
                                           L.has_indexer() ? sel : nullptr, n_sel, inv_freq, out, aw, err, s));
}

// Host-side checks of a packed variable-length batch's sizes (the row table itself is on the device).
static bool varlen_args_ok(int B, const int32_t* cu_seqlens, int N, int T_max) {
  // (B + 1 <= 4096 N: the index scan's group table fits the query area of its workspace)
  return B >= 1 && B <= (1 << 16) && N >= 1 && T_max >= 1 && T_max <= N && (long long)B + 1 <= 4096LL * N &&
         dev_i32(cu_seqlens);
}

csa_status csa_compress_append_varlen(const csa_layer* layer, const csa_compressor* comp, const void* x, int B,
                                      const int32_t* cu_seqlens, int N, int T_max, const int32_t* pos,
                                      void* frontier, void* pool, int cap, int32_t* n_rows, const float* inv_freq,
                                      void* ws, size_t ws_bytes, int32_t* err, void* stream) {
  Dims L;
  csa_status st = make_dims(layer, &L);
  if (st != CSA_OK) return st;
  if (!varlen_args_ok(B, cu_seqlens, N, T_max) || N > (1 << 20)) return CSA_ERR_ARG;
  if (!compress_args_ok(L, comp, B, 1, cap, frontier, pool, n_rows)) return CSA_ERR_ARG;
  if (!dev_tensor(x) || !dev_i32(pos) || !dev_tensor(inv_freq) || !dev_i32(err)) return CSA_ERR_ARG;
  Carver c0(nullptr);
  carve_compress_varlen(c0, L, comp->d, B, N);
  if (ws_bytes < c0.off || !dev_tensor(ws)) return CSA_ERR_WORKSPACE;
  Carver c(ws);
  const CompressWs w = carve_compress_varlen(c, L, comp->d, B, N);
  return cuda_status(launch_compress_varlen(L, *comp, x, B, cu_seqlens, N, T_max, pos, frontier, pool, cap, n_rows,
                                            inv_freq, w, err, static_cast<cudaStream_t>(stream)));
}

csa_status csa_attend_prefill_varlen(const csa_layer* layer, const void* q, const void* kv_new, const void* iq,
                                     const void* iw, const float* sink, int B, const int32_t* cu_seqlens, int N,
                                     int T_max, const int32_t* pos, void* window, const void* pool,
                                     const void* ikeys, int cap, const int32_t* n_rows, const float* inv_freq,
                                     void* out, int32_t* sel_out, void* ws, size_t ws_bytes, int32_t* err,
                                     void* stream) {
  Dims L;
  csa_status st = make_dims(layer, &L);
  if (st != CSA_OK) return st;
  if (!varlen_args_ok(B, cu_seqlens, N, T_max) || N > 16384 || cap < 1) return CSA_ERR_ARG;
  if (!tc_attend_supported(L) || (L.has_indexer() && !tc_index_supported(L))) return CSA_ERR_UNSUPPORTED;
  if (!dev_tensor(q) || !dev_tensor(kv_new) || !dev_i32(sink) || !dev_tensor(window) || !dev_tensor(pool) ||
      !dev_tensor(inv_freq) || !dev_tensor(out))
    return CSA_ERR_ARG;
  if (!dev_i32(pos) || !dev_i32(n_rows) || !dev_i32(err)) return CSA_ERR_ARG;
  if (L.has_indexer() && (!dev_tensor(iq) || !dev_i32(iw) || !dev_tensor(ikeys))) return CSA_ERR_ARG;
  if (sel_out && !dev_i32(sel_out)) return CSA_ERR_ARG;
  const size_t need = ws_prefill(L, N, cap);
  if (ws_bytes < need || !dev_tensor(ws)) return CSA_ERR_WORKSPACE;
  Carver c(ws);
  IndexWs iws{};
  int32_t *sel = nullptr, *n_sel = nullptr;
  AttendWs aw{};
  carve_prefill(c, L, N, cap, &iws, &sel, &n_sel, &aw);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (L.has_indexer()) {
    if (sel_out) sel = sel_out;
    cudaError_t e = launch_index_topk(L, iq, iw, N, ikeys, cap, n_rows, pos, B, inv_freq, sel, n_sel, iws, err, s,
                                      cu_seqlens);
    if (e != cudaSuccess) return CSA_ERR_CUDA;
  } else if (sel_out && L.topk > 0) {
    cudaMemsetAsync(sel_out, 0xff, (size_t)N * L.topk * sizeof(int32_t), s);
  }
  return cuda_status(launch_attend_prefill_varlen(L, q, kv_new, sink, B, cu_seqlens, N, T_max, window, pool, cap,
                                                  n_rows, L.has_indexer() ? sel : nullptr, n_sel, pos, inv_freq,
                                                  out, aw, err, s));
}

csa_status csa_index_topk_verify(const csa_layer* layer, const void* iq, const void* iw, int B, int T,
                                 const void* ikeys, int cap, const int32_t* n_rows, const int32_t* pos,
                                 const float* inv_freq, int32_t* sel, int32_t* n_sel, void* ws, size_t ws_bytes,
                                 int32_t* err, void* stream) {
  Dims L;
  csa_status st = make_dims(layer, &L);
  if (st != CSA_OK) return st;
  if (!L.has_indexer()) return CSA_ERR_UNSUPPORTED;
  if (B < 1 || T < 1 || T > 64 || cap < 1 || (long long)B * T > (1 << 20)) return CSA_ERR_ARG;
  if (!dev_tensor(iq) || !dev_i32(iw) || !dev_tensor(ikeys) || !dev_tensor(inv_freq)) return CSA_ERR_ARG;
  if (!dev_i32(n_rows) || !dev_i32(pos) || !dev_i32(sel) || !dev_i32(n_sel) || !dev_i32(err)) return CSA_ERR_ARG;
  const size_t need = ws_index(L, B * T, cap);
  if (ws_bytes < need || !dev_tensor(ws)) return CSA_ERR_WORKSPACE;
  Carver c(ws);
  IndexWs w = carve_index(c, L, B * T, cap);
  // with device positions the index kernels take the queries per sequence in place of pos0
  return cuda_status(launch_index_topk(L, iq, iw, B * T, ikeys, cap, n_rows, pos, T, inv_freq, sel, n_sel, w, err,
                                       static_cast<cudaStream_t>(stream)));
}

csa_status csa_attend_verify(const csa_layer* layer, const void* q, const void* kv_new, const float* sink, int B, int T,
                             void* window, const void* pool, int cap, const int32_t* n_rows, const int32_t* sel,
                             const int32_t* n_sel, const int32_t* pos, const float* inv_freq, void* out, void* ws,
                             size_t ws_bytes, int32_t* err, void* stream) {
  Dims L;
  csa_status st = make_dims(layer, &L);
  if (st != CSA_OK) return st;
  if (!L.has_indexer() || !tc_attend_decode_supported(L)) return CSA_ERR_UNSUPPORTED;
  if (B < 1 || T < 1 || T > 64 || cap < 1 || (long long)B * T > (1 << 20)) return CSA_ERR_ARG;
  if (T - 1 > L.rollback) return CSA_ERR_ARG;  // the block's later tokens would overwrite window rows still attended
  if (!dev_tensor(q) || !dev_tensor(kv_new) || !dev_i32(sink) || !dev_tensor(window) || !dev_tensor(pool) ||
      !dev_tensor(inv_freq) || !dev_tensor(out))
    return CSA_ERR_ARG;
  if (!dev_i32(n_rows) || !dev_i32(pos) || !dev_i32(err) || !dev_i32(sel) || !dev_i32(n_sel)) return CSA_ERR_ARG;
  const size_t need = ws_decode(L, B * T, cap);
  if (ws_bytes < need || !dev_tensor(ws)) return CSA_ERR_WORKSPACE;
  Carver c(ws);
  AttendWs w = carve_attend(c, L, B * T, attend_splits(L, false, false, cap), 0);
  return cuda_status(launch_attend_verify(L, q, kv_new, sink, B, T, window, pool, cap, n_rows, sel, n_sel, pos,
                                          inv_freq, out, w, err, static_cast<cudaStream_t>(stream)));
}

csa_status csa_trim(const csa_layer* layer, int B, const int32_t* n_back, int32_t* pos, int32_t* n_rows_a,
                    int32_t* n_rows_i, int32_t* hw, int32_t* err, void* stream) {
  Dims L;
  csa_status st = make_dims(layer, &L);
  if (st != CSA_OK) return st;
  if (B < 0) return CSA_ERR_ARG;
  if (B == 0) return CSA_OK;
  if (!dev_i32(n_back) || !dev_i32(pos) || !dev_i32(n_rows_a) || !dev_i32(hw) || !dev_i32(err)) return CSA_ERR_ARG;
  if (n_rows_i && !dev_i32(n_rows_i)) return CSA_ERR_ARG;
  if (L.has_indexer() && !n_rows_i) return CSA_ERR_ARG;
  return cuda_status(launch_trim(L, B, n_back, pos, n_rows_a, n_rows_i, hw, err, static_cast<cudaStream_t>(stream)));
}

csa_status csa_advance_positions(int32_t* pos, int B, int by, void* stream) {
  if (B < 0 || (B > 0 && !pos)) return CSA_ERR_ARG;
  if (B == 0) return CSA_OK;
  return cuda_status(launch_advance_positions(pos, B, by, static_cast<cudaStream_t>(stream)));
}

csa_status csa_index_rows_fp8(const csa_layer* layer, const void* src, long long n, void* dst, void* stream) {
  Dims L;
  csa_status st = make_dims(layer, &L);
  if (st != CSA_OK) return st;
  if (!L.ikey_fp8) return CSA_ERR_UNSUPPORTED;
  if (n < 0 || n > (1LL << 34)) return CSA_ERR_ARG;
  if (n == 0) return CSA_OK;
  if (!dev_tensor(src) || !dev_tensor(dst)) return CSA_ERR_ARG;
  return cuda_status(launch_index_rows_fp8(src, n, dst, static_cast<cudaStream_t>(stream)));
}

}  // extern "C"
