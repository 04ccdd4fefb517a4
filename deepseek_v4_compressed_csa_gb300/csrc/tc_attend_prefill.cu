// Chunked-prefill attention on the 5th-generation tensor cores for the Flash
// shapes (64 query heads over one 512-dim latent, K = V, bf16, RoPE on the last
// 64 dims).  A persistent CTA per SM walks its share of the chunk's queries; each
// query attends to its own selected pool rows plus its window tokens, taken in
// tiles of 128 rows.
//
// Definitions: "DeepSeek-V4-Flash: native deepseek_v4 AR backend" (MTPLX #216),
// "What V4 adds" (MQA-shaped MLA with per-head sink logits, 128-token window)
// and "Decode path" (bf16 in/out, fp32 softmax state, the probability block
// cast to bf16 before the PV product); "deepseek-v41-mlx" README (inverse rope
// on the output, sinks in the denominator only); "feat: add DeepSeek-V4
// (Pro/Flash) model support" (mlx-lm #1189), stepnoy: prefill applies a
// per-query top-k AND-ed with the visibility mask.
//
// A prefill CTA handles tens of queries of several tiles each, so the kernel is
// a pipeline of three warp roles rather than one latency-bound chunk:
//   loaders (warps 9-10)   gather a tile's rows with cp.async into one 128-row,
//            128-byte-swizzled tile, as four pairs of 64-dim boxes (128 latent
//            dims each).  A pair is refilled with the next tile's rows as soon
//            as the PV product of the current tile has read it, so the next
//            tile streams in under the current PV.  They also copy each query
//            block (64 KB) once the previous query's last score product has
//            retired, and rope it in place.
//   MMA (warp 8)   S^T = K Q^T (M = 128 rows, N = 64 heads, K = 512) pair by pair
//            as the rows land, then O^T += V^T P^T per 128-dim tile of the
//            latent: tiles 0-2 with [P_hi | P_lo] side by side (N = 128, one
//            read of V for both parts, two accumulators), tile 3 with P_hi and
//            P_lo in turn into one accumulator (N = 64), which leaves the last 64
//            TMEM columns to S^T.  P_hi = bf16(P), P_lo = bf16(P - P_hi): the
//            product keeps ~16 bits of P.
//   softmax (warps 0-7)   thread = (row, 32 heads).  The reference max of a head
//            is the column max of the query's first tile, raised only when a
//            later tile exceeds it by 2^8 (O^T and the running sums are then
//            rescaled).  Row sums stay per thread and are reduced once per
//            query; after the query's last PV the same warps finalise the
//            output (sink, normalisation, bf16, inverse RoPE, bf16).
#include "common.cuh"
#include "kernels.h"
#include "tc.cuh"

namespace csa {

namespace {

constexpr int kPR = 128;                 // rows per tile
constexpr int kAD = 512;                 // latent dims
constexpr int kAH = 64;                  // heads
constexpr int kBox = kPR * 128;          // 64 dims x 128 rows (16 KB)
constexpr int kRowsBytes = 8 * kBox;     // 128 KB
constexpr int kQBox = kAH * 128;         // 64 dims x 64 heads (8 KB)
constexpr int kQBytes = 8 * kQBox;       // 64 KB
constexpr int kPPart = kPR * 128;        // P^T part: 128 rows x 64 heads, MN-major (16 KB)
constexpr int kSoftWarps = 8;            // warps 0-7: (lane quarter, head half)
constexpr int kSoft = 32 * kSoftWarps;
constexpr int kHalf = kSoft / 2;         // threads of one head half
constexpr int kMmaWarp = kSoftWarps;     // warp 8: TMEM owner and MMA issuer
constexpr int kLoadWarp0 = kMmaWarp + 1; // warps 9-10
constexpr int kLoaders = 64;
constexpr int kThreads = kSoft + 32 + kLoaders;
constexpr int kTmemCols = 512;
constexpr uint32_t kColO3 = 384;         // O^T tile 3 (hi + lo in one accumulator)
constexpr uint32_t kColS = 448;          // S^T
constexpr float kRescaleAt = 8.f;        // log2 headroom before O is rescaled
constexpr int kBarLoad = 3;              // named barrier of the loader warps (1, 2: softmax halves)

// shared memory (byte offsets from the 1024-aligned base)
constexpr int kOffQ = kRowsBytes;
constexpr int kOffP = kOffQ + kQBytes;
constexpr int kOffRowc = kOffP + 2 * kPPart;   // [128] row codes of the tile in flight
constexpr int kOffRed = kOffRowc + kPR * 4;    // [4 lane quarters][64 heads] column maxima / sums
constexpr int kOffMref = kOffRed + 4 * 64 * 4;   // [64] reference max per head (log2 units)
constexpr int kOffBars = kOffMref + 64 * 4;
constexpr int kNumBars = 16;
constexpr int kOffTmem = kOffBars + kNumBars * 8;
constexpr int kSmem = kOffTmem + 16 + 1024;    // + alignment slack
static_assert(kSmem <= 232448, "shared memory per block");

// row codes: >= 0 pool row; kRowNone: empty (zero-filled, masked); <= kRowTok0: window token kRowTok0 - code
constexpr int kRowNone = -1;
constexpr int kRowTok0 = -2;

struct PfArgs {
  const __nv_bfloat16* q;      // [T, 64, 512] queries before RoPE
  const __nv_bfloat16* pool;   // [cap, 512] compressed rows (pool of the one sequence); verify: [B, cap, 512]
  const __nv_bfloat16* ring;   // [Wr, 512] window ring before the chunk (token t in slot t % Wr); verify: [B, Wr, 512]
  const __nv_bfloat16* kvr;    // [T, 512] roped rows of the chunk's tokens (unused for verify blocks)
  const int32_t* sel;          // [T, topk] or null (every visible row)
  const int32_t* n_sel;
  const int32_t* n_rows;       // [1]; verify: [B]
  const int32_t* pos;          // null: one chunk at pos0 + q; verify blocks: [B], query q at pos[q / qps] + q % qps
  int qps;                     // verify: queries per sequence (every window token of the block already in the ring)
  const int32_t* cu;           // packed variable-length batch of nseq chunks: row table [nseq + 1], query q of
  int nseq;                    // sequence b (cu[b] <= q < cu[b+1]) at pos[b] + q - cu[b]; kvr holds every chunk's rows
  const float* sink;
  const float* inv_freq;
  int T, pos0, cap, topk, W, ratio;
  int Wr;                      // ring slots (W + rollback); a query attends its last W tokens
  int chunk_tiles;             // T >= 128: 128-row boxes of the chunk's rows are available
  float scale2;                // softmax scale * log2(e)
  __nv_bfloat16* out;          // [T, 64, 512]
  int32_t* err;
};

struct Query {
  int b, p, nsel, nwin, nrows, ntiles;
};

__device__ __forceinline__ Query query_info(const PfArgs& a, int qi) {
  Query r;
  if (a.cu) {
    r.b = varlen_seq(a.cu, a.nseq, qi);
    r.p = a.pos[r.b] + qi - __ldg(a.cu + r.b);
  } else {
    r.b = a.pos ? qi / a.qps : 0;
    r.p = a.pos ? a.pos[r.b] + qi % a.qps : a.pos0 + qi;
  }
  r.nrows = min(a.n_rows[r.b], a.cap);
  r.nsel = a.sel ? min(max(a.n_sel[qi], 0), a.topk) : max(0, min(r.nrows, (r.p + 1) / a.ratio));
  r.nwin = r.p >= 0 ? min(a.W, r.p + 1) : 0;
  r.ntiles = max(1, (r.nsel + r.nwin + kPR - 1) / kPR);  // a query without rows still finalises a zero output
  return r;
}

// Code of row r_abs of query qi; j = sel[qi][r_abs] when a selection is given and r_abs < nsel.  A pool row's
// code is its row in the pool tensor map (b * cap + j); a window token's is kRowTok0 - token for a chunk, and
// kRowTok0 - (b * Wr + token mod Wr), its ring row, for verify blocks; in a variable-length batch, kRowTok0 -
// its ring row (tokens before the sequence's chunk) or kRowTok0 - (kChunkFlag + its packed chunk row).
constexpr int kChunkFlag = 1 << 29;
__device__ __forceinline__ int row_code(const PfArgs& a, const Query& qu, int r_abs, int j) {
  if (r_abs < qu.nsel) {
    if (!a.sel) j = r_abs;
    if (j >= 0 && j < qu.nrows) return qu.b * a.cap + j;
    atomicOr(a.err, CSA_DEV_RANGE);
    return kRowNone;
  }
  if (r_abs < qu.nsel + qu.nwin) {
    const int tok = qu.p - qu.nwin + 1 + (r_abs - qu.nsel);
    if (a.cu) {
      const int p0 = a.pos[qu.b];
      if (tok < p0) return kRowTok0 - (qu.b * a.Wr + tok % a.Wr);
      const int row = min(max(__ldg(a.cu + qu.b) + (tok - p0), 0), a.T - 1);  // inside the packed rows
      return kRowTok0 - (kChunkFlag + row);
    }
    return kRowTok0 - (a.pos ? qu.b * a.Wr + tok % a.Wr : tok);
  }
  return kRowNone;
}

// Tensor map of a row: the pool, the chunk's roped rows, the ring before the chunk; kSrcNone: empty row.
constexpr int kSrcPool = 0, kSrcChunk = 1, kSrcRing = 2, kSrcNone = 3;

__device__ __forceinline__ int row_src(const PfArgs& a, int code, int& row) {
  if (code >= 0) {
    row = code;
    return kSrcPool;
  }
  if (code <= kRowTok0) {
    const int tok = kRowTok0 - code;
    if (a.cu) {  // variable-length batch: the ring row or the flagged packed chunk row
      row = tok >= kChunkFlag ? tok - kChunkFlag : tok;
      return tok >= kChunkFlag ? kSrcChunk : kSrcRing;
    }
    if (a.pos) {
      row = tok;  // verify blocks: already the ring row
      return kSrcRing;
    }
    if (tok >= a.pos0) {
      row = tok - a.pos0;
      return kSrcChunk;
    }
    row = tok % a.Wr;
    return kSrcRing;
  }
  row = 0;
  return kSrcNone;
}

__device__ __forceinline__ const CUtensorMap* src_map(int src, const CUtensorMap* pool, const CUtensorMap* chunk,
                                                      const CUtensorMap* ring) {
  return src == kSrcPool ? pool : (src == kSrcChunk ? chunk : ring);
}

// Reduce 32 columns over the 32 lanes of a warp; lane L returns column L.
template <bool kMax>
__device__ __forceinline__ float reduce_scatter32(float (&v)[32]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int st = 0; st < 5; ++st) {
    const int half = 16 >> st;
    const bool upper = (lane & half) != 0;
#pragma unroll
    for (int i = 0; i < half; ++i) {
      const float send = upper ? v[i] : v[i + half];
      const float keep = upper ? v[i + half] : v[i];
      const float recv = __shfl_xor_sync(0xffffffffu, send, half);
      v[i] = kMax ? fmaxf(keep, recv) : keep + recv;
    }
  }
  return v[0];
}

// 2^x by the hardware approximation (relative error ~2^-22; results below 2^-126 flush to zero)
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// 32 scores of this thread's row from S^T (log2 units); masked rows read -inf
__device__ __forceinline__ void load_scores(uint32_t ta, bool valid, float scale2, float (&s)[32]) {
  uint32_t u[32];
  tc::tmem_ld32(ta, u);
  tc::tmem_wait_ld();
#pragma unroll
  for (int h = 0; h < 32; ++h) s[h] = valid ? __uint_as_float(u[h]) * scale2 : -INFINITY;
}

// RoPE of 8 consecutive dims (4 pairs) with their cos / sin
__device__ __forceinline__ void rope4(uint4& raw, const float (&rc)[4], const float (&rs)[4]) {
  __nv_bfloat162* hv = reinterpret_cast<__nv_bfloat162*>(&raw);
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float2 x = __bfloat1622float2(hv[k]);
    hv[k] = __floats2bfloat162_rn(fmaf(x.x, rc[k], -x.y * rs[k]), fmaf(x.x, rs[k], x.y * rc[k]));
  }
}

__global__ void __launch_bounds__(kThreads, 1)
    k_tc_attend_prefill(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_pool,
                        const __grid_constant__ CUtensorMap tm_kvr, const __grid_constant__ CUtensorMap tm_ring,
                        const __grid_constant__ CUtensorMap tm_kvr_tile, PfArgs a) {
  pdl_trigger();
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* rows = smem;
  uint8_t* qbuf = smem + kOffQ;
  uint8_t* pbuf = smem + kOffP;
  int* rowc = reinterpret_cast<int*>(smem + kOffRowc);
  float* red = reinterpret_cast<float*>(smem + kOffRed);
  float* mref = reinterpret_cast<float*>(smem + kOffMref);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBars);
  uint64_t* q_full = bars + 0;     // query block copied and roped (loaders)
  uint64_t* q_empty = bars + 1;    // the query's last score product retired (MMA)
  uint64_t* rows_full = bars + 2;  // [4] box pair m of the tile landed (loaders)
  uint64_t* box_free = bars + 6;   // [4] PV of tile m retired: box pair m may take the next tile (MMA)
  uint64_t* s_full = bars + 10;    // S^T of the tile in TMEM (MMA)
  uint64_t* p_full = bars + 11;    // P^T parts written, S^T read (softmax)
  uint64_t* pv_done = bars + 12;   // PV of the tile retired (MMA)
  uint64_t* o_free = bars + 13;    // the query's output read out of TMEM (softmax)
  uint64_t* drain = bars + 14;
  uint64_t* q_loaded = bars + 15;  // query block landed (TMA)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffTmem);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    tc::mbar_init(q_full, kLoaders);
    tc::mbar_init(q_empty, 1);
    for (int m = 0; m < 4; ++m) {
      tc::mbar_init(rows_full + m, kLoaders);  // one arrival (with its bytes) per loader thread
      tc::mbar_init(box_free + m, 1);
    }
    tc::mbar_init(s_full, 1);
    tc::mbar_init(p_full, kSoft);
    tc::mbar_init(pv_done, 1);
    tc::mbar_init(o_free, kSoft);
    tc::mbar_init(drain, 1);
    tc::mbar_init(q_loaded, 1);
    tc::fence_mbar_init();
  }
  pdl_wait();  // predecessor complete: its outputs are visible and its tensor memory is free
  if (warp == kMmaWarp) {
    tc::tmem_alloc(tmem_slot, kTmemCols);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  bool failed = false;

  if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t id_qk = tc::idesc_bf16(128, 64);
      constexpr uint32_t id_pv2 = tc::idesc_bf16(128, 128, true, true);
      constexpr uint32_t id_pv1 = tc::idesc_bf16(128, 64, true, true);
      const uint32_t r_base = tc::smem_u32(rows), q_base = tc::smem_u32(qbuf), p_base = tc::smem_u32(pbuf);
      uint32_t nq = 0, nt = 0;
      for (int qi = blockIdx.x; qi < a.T && !failed; qi += gridDim.x, ++nq) {
        const int ntiles = query_info(a, qi).ntiles;
        if (!tc::mbar_wait(q_full, nq & 1)) { failed = true; break; }
        tc::fence_after_sync();
        for (int t = 0; t < ntiles; ++t, ++nt) {
          const uint32_t par = nt & 1;
          // S^T = K Q^T, pair by pair as the rows land
          for (int m = 0; m < 4 && !failed; ++m) {
            if (!tc::mbar_wait(rows_full + m, par)) { failed = true; break; }
            tc::fence_after_sync();
#pragma unroll
            for (int k = 8 * m; k < 8 * m + 8; ++k) {
              const uint64_t ad = tc::sdesc_kmajor_sw128(r_base + (k >> 2) * kBox + (k & 3) * 32);
              const uint64_t bd = tc::sdesc_kmajor_sw128(q_base + (k >> 2) * kQBox + (k & 3) * 32);
              tc::mma_bf16(tmem + kColS, ad, bd, id_qk, k > 0);
            }
          }
          if (failed) break;
          tc::mma_commit(s_full);
          if (t == ntiles - 1) tc::mma_commit(q_empty);
          if (!tc::mbar_wait(p_full, par)) { failed = true; break; }
          tc::fence_after_sync();
          if (t == 0 && nq > 0) {
            // the previous query's output must be out of TMEM before this query's first product overwrites it
            if (!tc::mbar_wait(o_free, (nq - 1) & 1)) { failed = true; break; }
            tc::fence_after_sync();
          }
          // O^T += V^T P^T: 128-dim tiles 0-2 with both parts side by side, tile 3 with the parts in turn
#pragma unroll
          for (int m = 0; m < 4; ++m) {
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
              const uint64_t ad = tc::sdesc_mnmajor_sw128(r_base + 2 * m * kBox + kk * 2048, kBox, 1024);
              const uint64_t bd = tc::sdesc_mnmajor_sw128(p_base + kk * 2048, kPPart, 1024);
              const bool acc = (t > 0) || (kk > 0);
              if (m < 3) {
                tc::mma_bf16(tmem + 128 * m, ad, bd, id_pv2, acc);
              } else {
                const uint64_t bd_lo = tc::sdesc_mnmajor_sw128(p_base + kPPart + kk * 2048, kPPart, 1024);
                tc::mma_bf16(tmem + kColO3, ad, bd, id_pv1, acc);
                tc::mma_bf16(tmem + kColO3, ad, bd_lo, id_pv1, true);
              }
            }
            tc::mma_commit(box_free + m);
          }
          tc::mma_commit(pv_done);
        }
      }
    }
    __syncwarp();
    failed = __shfl_sync(0xffffffffu, (int)failed, 0) != 0;
  } else if (warp >= kLoadWarp0) {
    // ------------------------------------------------------------ loaders (warps 9-10, 64 threads)
    const int lt = tid - kLoadWarp0 * 32;
    if (lt == 0) {
      tc::tma_prefetch(&tm_q);
      tc::tma_prefetch(&tm_pool);
      tc::tma_prefetch(&tm_kvr);
      tc::tma_prefetch(&tm_ring);
      tc::tma_prefetch(&tm_kvr_tile);
    }
    uint32_t nq = 0, nt = 0;
    for (int qi = blockIdx.x; qi < a.T && !failed; qi += gridDim.x, ++nq) {
      const Query qu = query_info(a, qi);
      // codes of this thread's rows (lt, lt + 64) of a tile
      auto codes = [&](int t, int& x0, int& x1) {
        const int ra = t * kPR + lt, rb = ra + 64;
        const int ja = (a.sel && ra < qu.nsel) ? a.sel[(size_t)qi * a.topk + ra] : 0;
        const int jb = (a.sel && rb < qu.nsel) ? a.sel[(size_t)qi * a.topk + rb] : 0;
        x0 = row_code(a, qu, ra, ja);
        x1 = row_code(a, qu, rb, jb);
      };
      int c0, c1;
      codes(0, c0, c1);
      // ---- the query block (8 boxes of 64 heads x 64 dims), once the previous query's last score product
      // has retired; then RoPE on its last box
      if (nq > 0 && tc::named_bar_any(kBarLoad, kLoaders, !tc::mbar_wait(q_empty, (nq - 1) & 1))) {
        failed = true;
        break;
      }
      if (lt == 0) {
        tc::mbar_arrive_expect_tx(q_loaded, kQBytes);
        for (int c = 0; c < 8; ++c) tc::tma_load_2d(qbuf + c * kQBox, &tm_q, q_loaded, 64 * c, qi * kAH);
      }
      // this thread ropes chunk 56 + (lt & 7) (dims 448 + 8 (lt & 7) ..) of heads lt / 8 + 8 i: four frequencies
      const int rch = 56 + (lt & 7);
      float rcs[4], rsn[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) rope_cs(qu.p, a.inv_freq, (rch - 56) * 4 + k, &rcs[k], &rsn[k]);
      if (tc::named_bar_any(kBarLoad, kLoaders, !tc::mbar_wait(q_loaded, nq & 1))) {
        failed = true;
        break;
      }
#pragma unroll
      for (int h = lt >> 3; h < kAH; h += kLoaders / 8) {
        uint4* slot = reinterpret_cast<uint4*>(qbuf + 7 * kQBox + h * 128 + (((rch & 7) ^ (h & 7)) << 4));
        uint4 raw = *slot;
        rope4(raw, rcs, rsn);
        *slot = raw;
      }
      tc::fence_proxy_async_smem();
      tc::mbar_arrive(q_full);
      // ---- the query's tiles: thread lt loads rows 4 (lt / 2) .. + 3 of box 2m + lt % 2 of pair m
      const int g4 = 4 * (lt >> 1);
      for (int t = 0; t < qu.ntiles; ++t, ++nt) {
        const uint32_t par = (nt - 1) & 1;  // phase of the previous tile's releases
        if (nt > 0 && tc::named_bar_any(kBarLoad, kLoaders, !tc::mbar_wait(box_free, par))) {
          failed = true;
          break;
        }
        // the previous tile's softmax has read its codes (its P was complete before the first PV product)
        rowc[lt] = c0;
        rowc[lt + 64] = c1;
        tc::named_bar(kBarLoad, kLoaders);
        int src[4], row[4];
        bool same = true;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          src[i] = row_src(a, rowc[g4 + i], row[i]);
          same &= src[i] == src[0];
        }
        same &= src[0] != kSrcNone;
        // a tile of 128 consecutive chunk rows (a window in the chunk): one 128-row box load per 64 dims
        int row_first, row_last;
        const bool chunk_tile = a.chunk_tiles && row_src(a, rowc[0], row_first) == kSrcChunk &&
                                row_src(a, rowc[kPR - 1], row_last) == kSrcChunk;
        for (int m = 0; m < 4; ++m) {
          if (m > 0 && nt > 0 && tc::named_bar_any(kBarLoad, kLoaders, !tc::mbar_wait(box_free + m, par))) {
            failed = true;
            break;
          }
          const int box = 2 * m + (lt & 1);
          uint8_t* dst = rows + box * kBox + g4 * 128;
          if (chunk_tile) {
            if (lt < 2) {
              tc::mbar_arrive_expect_tx(rows_full + m, kBox);
              tc::tma_load_2d(rows + box * kBox, &tm_kvr_tile, rows_full + m, 64 * box, row_first);
            } else {
              tc::mbar_arrive(rows_full + m);
            }
          } else if (same) {
            tc::mbar_arrive_expect_tx(rows_full + m, 4 * 128);
            tc::tma_gather4(dst, src_map(src[0], &tm_pool, &tm_kvr, &tm_ring), rows_full + m, 64 * box, row[0], row[1],
                            row[2], row[3]);
          } else {
            // rows from different sources, or empty rows: one-row loads, zeros written here
            uint32_t bytes = 0;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              if (src[i] == kSrcNone) {
#pragma unroll
                for (int c = 0; c < 8; ++c) reinterpret_cast<uint4*>(dst + i * 128)[c] = make_uint4(0, 0, 0, 0);
              } else {
                bytes += 128;
              }
            }
            tc::fence_proxy_async_smem();
            tc::mbar_arrive_expect_tx(rows_full + m, bytes);
#pragma unroll
            for (int i = 0; i < 4; ++i)
              if (src[i] != kSrcNone)
                tc::tma_load_2d(dst + i * 128, src_map(src[i], &tm_pool, &tm_kvr, &tm_ring), rows_full + m, 64 * box,
                                row[i]);
          }
        }
        if (failed) break;
        if (t + 1 < qu.ntiles) codes(t + 1, c0, c1);
      }
    }
  } else {
    // ------------------------------------------------------------ softmax and epilogue (warps 0-7)
    // thread = row 32 * quad + lane of the tile (TMEM lane quarter = warp % 4), heads hb .. hb + 31
    const int quad = warp & 3, half = warp >> 2, hb = 32 * half;
    const int row = 32 * quad + lane;
    const int bar_half = 1 + half;
    const uint32_t lane_base = (uint32_t)(32 * quad) << 16;
    const float* mh = mref + hb;  // this half's reference maxima (the same for all its threads)
    float l[32];
    uint32_t nq = 0, nt = 0;
    for (int qi = blockIdx.x; qi < a.T && !failed; qi += gridDim.x, ++nq) {
      const Query qu = query_info(a, qi);
      for (int t = 0; t < qu.ntiles; ++t, ++nt) {
        if (tc::named_bar_any(bar_half, kHalf, !tc::mbar_wait(s_full, nt & 1))) {
          failed = true;
          break;
        }
        tc::fence_after_sync();
        const bool valid = rowc[row] != kRowNone;
        float s[32];
        load_scores(tmem + kColS + hb + lane_base, valid, a.scale2, s);
        bool ovf = false;
        if (t > 0) {
#pragma unroll
          for (int h = 0; h < 32; ++h) ovf |= s[h] > mh[h] + kRescaleAt;
        }
        if (t == 0 || tc::named_bar_any(bar_half, kHalf, ovf)) {
          // column maxima of the tile over the half's 128 rows (the reduction consumes s; S^T is read again)
          red[quad * 64 + hb + lane] = reduce_scatter32<true>(s);
          tc::named_bar(bar_half, kHalf);
          // new reference of head h: the tile max on the query's first tile, else raised when 2^8 above
          auto raise = [&](int h, float& fac) {
            const float mt = fmaxf(fmaxf(red[hb + h], red[64 + hb + h]), fmaxf(red[128 + hb + h], red[192 + hb + h]));
            const float old = mh[h];
            fac = 1.f;
            if (t == 0) return mt;
            if (mt > old + kRescaleAt) {
              fac = exp2f(old - mt);
              return mt;
            }
            return old;
          };
          bool resc = false;  // the same answer in every thread of the half: all read the same maxima
#pragma unroll
          for (int h = 0; h < 32; ++h) {
            raise(h, s[h]);  // s[h] = rescale factor of head h
            resc |= s[h] != 1.f;
          }
          tc::named_bar(bar_half, kHalf);  // every thread has read the old references
          if (quad == 0) {
            float fac;
            const float nw = raise(lane, fac);
            mref[hb + lane] = nw;
          }
          tc::named_bar(bar_half, kHalf);
          if (resc) {
            // raise the reference max: the running sums and O^T (every earlier PV has retired) *= factor
#pragma unroll
            for (int h = 0; h < 32; ++h) l[h] *= s[h];
#pragma unroll 1
            for (int c = 0; c < 7; ++c) {
              const uint32_t col = c < 6 ? 128 * (c >> 1) + 64 * (c & 1) : kColO3;
              const uint32_t ta = tmem + col + hb + lane_base;
              uint32_t u[32];
              tc::tmem_ld32(ta, u);
              tc::tmem_wait_ld();
#pragma unroll
              for (int h = 0; h < 32; ++h) u[h] = __float_as_uint(__uint_as_float(u[h]) * s[h]);
              tc::tmem_st32(ta, u);
            }
            tc::tmem_wait_st();
          }
          load_scores(tmem + kColS + hb + lane_base, valid, a.scale2, s);
        }
        // ---- probabilities: fp32 for the sums, bf16 hi + lo parts of P^T (MN-major) for the PV product
        float (&pe)[32] = s;
#pragma unroll
        for (int h = 0; h < 32; ++h) {
          const float ref = mh[h] == -INFINITY ? 0.f : mh[h];
          pe[h] = s[h] == -INFINITY ? 0.f : ex2_approx(s[h] - ref);
          l[h] = (t == 0) ? pe[h] : l[h] + pe[h];
        }
        uint8_t* dst = pbuf + (row >> 3) * 1024 + (row & 7) * 128;
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
          uint4 hi, lo;
          __nv_bfloat162* hv = reinterpret_cast<__nv_bfloat162*>(&hi);
          __nv_bfloat162* lv = reinterpret_cast<__nv_bfloat162*>(&lo);
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            hv[k] = __floats2bfloat162_rn(pe[8 * jj + 2 * k], pe[8 * jj + 2 * k + 1]);
            const float2 back = __bfloat1622float2(hv[k]);
            lv[k] = __floats2bfloat162_rn(pe[8 * jj + 2 * k] - back.x, pe[8 * jj + 2 * k + 1] - back.y);
          }
          const int off = ((4 * half + jj) ^ (row & 7)) << 4;
          *reinterpret_cast<uint4*>(dst + off) = hi;
          *reinterpret_cast<uint4*>(dst + kPPart + off) = lo;
        }
        tc::fence_proxy_async_smem();
        tc::fence_before_sync();
        tc::mbar_arrive(p_full);
      }
      if (failed) break;
      // ---- the query's output: per-head sums, then O^T tile by tile (thread = latent dim)
      tc::named_bar(bar_half, kHalf);  // the half is done with the column maxima
      red[quad * 64 + hb + lane] = reduce_scatter32<false>(l);
      tc::named_bar(bar_half, kHalf);
      float f[32];
#pragma unroll
      for (int h = 0; h < 32; ++h) {
        const float lsum = (red[hb + h] + red[64 + hb + h]) + (red[128 + hb + h] + red[192 + hb + h]);
        const float z2 = __ldg(a.sink + hb + h) * 1.4426950408889634f;
        const float mr = mh[h];
        const float M2 = fmaxf(z2, mr);
        const float ff = mr == -INFINITY ? 0.f : exp2f(mr - M2);
        const float Z = exp2f(z2 - M2) + lsum * ff;
        f[h] = ff / Z;
      }
      tc::named_bar(bar_half, kHalf);  // sums read: the next query's maxima may take the buffer
      if (tc::named_bar_any(bar_half, kHalf, !tc::mbar_wait(pv_done, (nt - 1) & 1))) {
        failed = true;
        break;
      }
      tc::fence_after_sync();
      // inverse RoPE of this thread's dim of tile 3 (dims 448-511 are lane quarters 2 and 3)
      float rc = 1.f, rs = 0.f;
      if (quad >= 2) rope_cs(qu.p, a.inv_freq, (32 * quad + lane - 64) >> 1, &rc, &rs);
      __nv_bfloat16* obase = a.out + (size_t)qi * kAH * kAD;
#pragma unroll 1
      for (int m = 0; m < 4; ++m) {
        const int d = 128 * m + 32 * quad + lane;
        float o[32];
        {
          uint32_t u[32];
          tc::tmem_ld32(tmem + (m < 3 ? 128 * m : kColO3) + hb + lane_base, u);
          tc::tmem_wait_ld();
#pragma unroll
          for (int h = 0; h < 32; ++h) o[h] = __uint_as_float(u[h]);
          if (m < 3) {
            tc::tmem_ld32(tmem + 128 * m + 64 + hb + lane_base, u);
            tc::tmem_wait_ld();
#pragma unroll
            for (int h = 0; h < 32; ++h) o[h] += __uint_as_float(u[h]);
          }
        }
        const bool rot = (m == 3) && quad >= 2;
#pragma unroll
        for (int h = 0; h < 32; ++h) {
          float v = rnd<__nv_bfloat16>(o[h] * f[h]);
          const float partner = __shfl_xor_sync(0xffffffffu, v, 1);
          if (rot) v = (d & 1) ? fmaf(-partner, rs, v * rc) : fmaf(v, rc, partner * rs);
          obase[(size_t)(hb + h) * kAD + d] = __float2bfloat16_rn(v);
        }
      }
      tc::fence_before_sync();
      tc::mbar_arrive(o_free);
    }
  }
  if (failed) atomicOr(a.err, tc::kErrTimeout);
  tc::fence_before_sync();
  __syncthreads();
  // retire every MMA before tensor memory is released
  if (warp == kMmaWarp && lane == 0) {
    tc::mma_commit(drain);
    if (!tc::mbar_wait(drain, 0)) atomicOr(a.err, tc::kErrTimeout);
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == kMmaWarp) tc::tmem_dealloc(tmem, kTmemCols);
}

int g_sms_pf = 0;

}  // namespace

cudaError_t launch_tc_attend_prefill(const Dims& L, const void* q, const void* pool, const void* ring,
                                     const void* kvr, const int32_t* sel, const int32_t* n_sel,
                                     const int32_t* n_rows, int pos0, int cap, const float* sink,
                                     const float* inv_freq, int T, void* out, int32_t* err, cudaStream_t s,
                                     const int32_t* pos, int qps, const int32_t* cu) {
  if (T <= 0) return cudaSuccess;
  if (cap <= 0) return cudaErrorInvalidValue;
  if (!g_sms_pf) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&g_sms_pf, cudaDevAttrMultiProcessorCount, dev);
  }
  PfArgs a{};
  a.q = static_cast<const __nv_bfloat16*>(q);
  a.pool = static_cast<const __nv_bfloat16*>(pool);
  a.ring = static_cast<const __nv_bfloat16*>(ring);
  a.kvr = static_cast<const __nv_bfloat16*>(kvr);
  a.sel = sel; a.n_sel = n_sel; a.n_rows = n_rows; a.sink = sink; a.inv_freq = inv_freq;
  a.T = T; a.pos0 = pos0; a.cap = cap; a.topk = L.topk; a.W = L.W; a.Wr = L.Wr; a.ratio = L.ratio;
  a.pos = pos; a.qps = max(1, qps);
  a.cu = cu; a.nseq = cu ? qps : 0;  // a row table: qps carries the number of sequences
  if (cu && (!pos || qps < 1 || !kvr)) return cudaErrorInvalidValue;
  const int nseq = cu ? qps : (pos ? (T + a.qps - 1) / a.qps : 1);
  if (pos && !kvr) kvr = q;  // verify blocks read no chunk rows: the chunk maps only need a valid address
  a.scale2 = L.scale * 1.4426950408889634f;
  a.out = static_cast<__nv_bfloat16*>(out);
  a.err = err;
  // one-row boxes for the row gathers (tile::gather4 and single rows), 64-row boxes for the query blocks
  // and 128-row boxes of the chunk's rows (whole window tiles)
  CUtensorMap tq, tp, tk, tr, tkt;
  a.chunk_tiles = (!pos || cu) && T >= kPR;
  if (!make_tmap_2d_bf16(&tq, q, (uint64_t)T * kAH, kAD, kAD * 2, 64) ||
      !make_tmap_2d_bf16(&tp, pool, (uint64_t)nseq * cap, kAD, kAD * 2, 1) ||
      !make_tmap_2d_bf16(&tk, kvr, (uint64_t)T, kAD, kAD * 2, 1) ||
      !make_tmap_2d_bf16(&tr, ring, (uint64_t)nseq * L.Wr, kAD, kAD * 2, 1) ||
      !make_tmap_2d_bf16(&tkt, kvr, (uint64_t)T, kAD, kAD * 2, a.chunk_tiles ? kPR : 1))
    return cudaErrorInvalidValue;
  cudaFuncSetAttribute(k_tc_attend_prefill, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
  CSA_LAUNCH(k_tc_attend_prefill, dim3(min(T, g_sms_pf)), dim3(kThreads), kSmem, s, tq, tp, tk, tr, tkt, a);
  return cudaGetLastError();
}

}  // namespace csa
