// Indexer scores on the 5th-generation tensor cores (bf16, Hi = 64 heads of
// Di = 128 dims; the Flash indexer).
//
// score_j(q) = sum_h w_qh * ReLU(RoPE(iq_qh, p_q) . key_j),  w_qh = iw_qh Di^-1/2 Hi^-1/2
// ("feat: add DeepSeek-V4 (Pro/Flash) model support", mlx-lm #1189: stepnoy's
// patch point 3 and aidiffuser's indexer).
//
// The contraction is computed transposed, S^T = K Q^T: M = 128 key rows per
// tile (TMEM lane = key row), N = 64 heads x G queries, K = Di = 128.  Each
// epilogue thread then owns one key row and reduces the head axis on its own
// (ReLU, weight, sum) without any cross-thread traffic.  Decode uses G = 1 (one
// query per sequence, each sequence with its own keys); a prefill chunk uses
// G = 4 queries of one sequence per MMA (N = 256), so a key tile is read once
// per 4 queries.
//
// One persistent CTA per SM, 8 warps: warp 0 issues TMA loads of a ring of 32 KB
// key tiles, warp 1 owns tensor memory and issues the MMAs from one thread,
// warps 2-5 drain the TMEM accumulators and write fp32 scores, warps 6-7 build
// each query block in shared memory (RoPE at the query's position, bf16, the
// 128-byte-swizzled K-major layout) and its scaled head weights, so no separate
// preparation pass runs before the scan.  Decode keeps two query blocks and
// four accumulators in flight.  With G = 4 a block (256 head rows, 64 KB) comes
// in one TMA copy, already in that layout, and its last R dims are roped in
// place: a CTA of a verify block's scan enters a new group every ~14 tiles, and
// copying the block through registers took eight dependent load rounds each
// time, with the one query slot (and so the tensor pipe) waiting.

#include "common.cuh"
#include "fp8_row.cuh"
#include "kernels.h"
#include "tc.cuh"

namespace csa {

namespace {

constexpr int kTileRows = 128;
constexpr int kPrepThreads = 64;                 // the last two warps

// kFp8: index keys and queries as E4M3 codes (a row of 128 bytes in shared memory, one 128-byte swizzle box)
template <int G, bool kFp8 = false>
struct IdxCfg {
  static constexpr int N = 64 * G;               // MMA N: 64 heads x G queries
  static constexpr int kRowBytes = kFp8 ? 128 : 256;           // a key row or a query head row in shared memory
  static constexpr int kTileBytes = kTileRows * kRowBytes;     // a key tile: 32 KB (bf16), 16 KB (e4m3)
  static constexpr int kQBytes = N * kRowBytes;  // one query block (bf16: 2 boxes of N rows x 128 B)
  static constexpr int kQSlots = G == 1 ? 2 : 1;
  // decode: five 32 KB key tiles in flight (measured best of 4-6); fp8: the same bytes in eight 16 KB tiles
  static constexpr int kStages = G == 1 ? (kFp8 ? 8 : 5) : (kFp8 ? 8 : 4);
  static constexpr int kAcc = G == 1 ? 4 : 2;    // TMEM accumulators of N columns
  static constexpr int kOffK = kQSlots * kQBytes;
  static constexpr int kOffW = kOffK + kStages * kTileBytes;   // [kQSlots][N] head weights
  static constexpr int kOffRope = kOffW + kQSlots * N * 4;     // [G][32] cos, [G][32] sin
  // fp8: the key rows' scales (bytes 128-143 of each row, 16 B a row) by a second TMA copy per tile into a ring
  // of kStages + kAcc slots: the producer refills a slot only once the epilogue is done with it (it has waited for
  // the MMA kStages tiles back, which waited for the epilogue kAcc tiles before that)
  static constexpr int kScaleSlots = kFp8 ? kStages + kAcc : 0;
  static constexpr int kScaleBytes = kTileRows * 16;
  static constexpr int kOffS = kOffRope + G * 64 * 4;
  static constexpr int kOffBars = kOffS + kScaleSlots * kScaleBytes;
  static constexpr int kNumBars = 2 * kStages + 4 * kQSlots + 2 * kAcc + 1 + kScaleSlots;
  static constexpr int kSmem = kOffBars + kNumBars * 8 + 16 + 1024;
  // warps: 0 TMA, 1 MMA, 2 .. 2 + kEpiWarps - 1 epilogue, then two query-block warps.  A prefill tile has four
  // queries' columns to reduce: eight epilogue warps, two per TMEM lane quarter, take two queries each.
  static constexpr int kEpiWarps = G == 1 ? 4 : 8;
  static constexpr int kQPerWarp = G / (kEpiWarps / 4);
  static constexpr int kPrepWarp0 = 2 + kEpiWarps;
  static constexpr int kThreads = 32 * kPrepWarp0 + kPrepThreads;
};

struct IdxArgs {
  const __nv_bfloat16* iq;  // [Q, 64, 128] index queries before RoPE
  const __nv_bfloat16* iw;  // [Q, 64] head weights
  const float* inv_freq;
  float wscale;             // Di^-1/2 Hi^-1/2
  int R;
  const int32_t* n_rows;
  const int32_t* pos;  // decode / verify positions [Q / qps] or null (prefill: pos0 + q)
  int qps;             // consecutive queries per sequence (a verify block of qps tokens; 1 for decode)
  const int32_t* cu;   // packed variable-length batch: row table [nseq + 1] (queries of sequence b: cu[b] ..), or null
  int nseq;
  const int32_t* gcu;  // G = 4 with a row table: group table [nseq + 1] (sequence b's ceil(T_b / 4) groups start at
                       // gcu[b]; a group never straddles two sequences), or null
  int pos0, ratio, topk, cap, Q, G, n_items, tiles_per_group;
  int group_penalty;  // partition weight of a group's query block, in tiles
  float* scores;     // [Q, cap]
  int32_t* err;
  // overlapped decode scan (kernel instance kOverlap): the roped queries and scaled head weights, left for the
  // selection stage
  __nv_bfloat16* qr_out;  // [Q, 64, 128]
  float* w_out;           // [Q, 64]
  // fp8 index keys (instance kFp8): the quantised queries, q8 [Q, 64, 128] codes and qs [Q, 64] scales; G = 4 takes
  // the head weights with the scale and the 1/128 folded in, w8 [Q, 64] (iw qs / 128)
  const uint8_t* q8;
  const float* qs;
  const float* w8;
};

__device__ __forceinline__ int idx_seq(const IdxArgs& a, int q) {
  if (a.cu) return varlen_seq(a.cu, a.nseq, q);
  return a.pos ? q / a.qps : 0;
}
__device__ __forceinline__ int idx_qpos(const IdxArgs& a, int q) {
  if (a.cu) {
    const int b = varlen_seq(a.cu, a.nseq, q);
    return a.pos[b] + q - __ldg(a.cu + b);
  }
  return a.pos ? a.pos[q / a.qps] + q % a.qps : a.pos0 + q;
}
// Group g's first query and query count (<= 0: no such group).  Without a group table: queries g G .. g G + G - 1
// (those below Q); with one: group k of sequence b (gcu[b] <= g < gcu[b+1]) holds queries cu[b] + 4k .. of its
// sequence only.
template <int G>
__device__ __forceinline__ int grp_first(const IdxArgs& a, int g, int& cnt) {
  if (G == 4 && a.gcu) {
    int lo = 0, hi = a.nseq - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (__ldg(a.gcu + mid) <= g) lo = mid; else hi = mid - 1;
    }
    const int q0 = __ldg(a.cu + lo) + 4 * (g - __ldg(a.gcu + lo));
    cnt = g < __ldg(a.gcu + a.nseq) ? min(4, __ldg(a.cu + lo + 1) - q0) : 0;
    cnt = q0 < 0 ? 0 : min(cnt, a.Q - q0);  // an inconsistent row table never reaches past the packed queries
    return q0;
  }
  cnt = min(G, a.Q - g * G);
  return g * G;
}
// query qq of group g, or -1
template <int G>
__device__ __forceinline__ int grp_query(const IdxArgs& a, int g, int qq) {
  int cnt;
  const int q0 = grp_first<G>(a, g, cnt);
  return qq < cnt ? q0 + qq : -1;
}
__device__ __forceinline__ int idx_nvis(const IdxArgs& a, int q) {
  const int b = idx_seq(a, q);
  return min(min(a.n_rows[b], a.cap), (idx_qpos(a, q) + 1) / a.ratio);
}
// Rows this scan scores for query q.  The overlapped decode scan, which runs while the index pool's compress
// call for the same token may still write, takes the rows complete before the query's token and does not read
// n_rows; the selection stage scores the rows that call may write.
template <bool kOverlap>
__device__ __forceinline__ int scan_rows(const IdxArgs& a, int q) {
  return kOverlap ? min(a.cap, idx_qpos(a, q) / a.ratio) : idx_nvis(a, q);
}
// tiles that group g must score (its last query sees the most rows); 0 if the group's queries keep every
// visible row anyway
template <int G, bool kOverlap>
__device__ __forceinline__ int group_tiles(const IdxArgs& a, int g) {
  int cnt;
  const int q0 = grp_first<G>(a, g, cnt);
  if (cnt <= 0) return 0;
  const int qlast = q0 + cnt - 1;
  if (kOverlap) {  // bound on the visible rows once the concurrent compress call has run
    if (min(a.cap, (idx_qpos(a, qlast) + 1) / a.ratio) <= a.topk) return 0;
    return (scan_rows<kOverlap>(a, qlast) + kTileRows - 1) / kTileRows;
  }
  const int nv = idx_nvis(a, qlast);
  return nv > a.topk ? (nv + kTileRows - 1) / kTileRows : 0;
}

// The CTA's work items are the (group, tile) pairs i_begin .. i_end-1 (item = group * tiles_per_group + tile); a
// group's tiles past its visible rows are skipped.  Every role walks the same sequence with this iterator: one
// division when it starts and one tile count per group, so that the MMA thread's per-tile bookkeeping stays a few
// instructions (a division per tile had cost it ~1k clocks a tile, leaving the tensor pipe idle between tiles).
template <int G, bool kOverlap>
struct Items {
  int g, t, t1, g_last, i_end, tpg;
  // first item at or after i_begin; false if none
  __device__ __forceinline__ bool start(const IdxArgs& a, int i_begin, int i_end_) {
    tpg = a.tiles_per_group;
    i_end = i_end_;
    g_last = i_begin < i_end ? (i_end - 1) / tpg : -1;
    g = i_begin < i_end ? i_begin / tpg : 0;
    t = i_begin - g * tpg;
    if (g > g_last) return false;
    bounds(a);
    return settle(a);
  }
  __device__ __forceinline__ bool advance(const IdxArgs& a) {
    ++t;
    return settle(a);
  }
  // first item of the next group that has one
  __device__ __forceinline__ bool next_group(const IdxArgs& a) {
    t = t1;
    return settle(a);
  }
  // the current item is the last of its group in this CTA's range
  __device__ __forceinline__ bool last_of_group() const { return t == t1 - 1; }

 private:
  __device__ __forceinline__ void bounds(const IdxArgs& a) {
    const int hi = (g == g_last) ? i_end - g * tpg : tpg;
    t1 = min(group_tiles<G, kOverlap>(a, g), hi);
  }
  __device__ __forceinline__ bool settle(const IdxArgs& a) {
    while (t >= t1) {
      if (++g > g_last) return false;
      t = 0;
      bounds(a);
    }
    return true;
  }
};

// Decode (G = 1) keeps to 128 registers a thread: the compress calls' small kernels running beside the scan
// on other streams (a pooling CTA: 256 threads x 64 registers) must still fit on the SMs it holds, or the
// scan's remaining CTAs wait for them to finish.
template <int G, bool kOverlap, bool kFp8 = false>
__global__ void __launch_bounds__(IdxCfg<G, kFp8>::kThreads, G == 1 ? 2 : 1)
    k_tc_index_scores(const __grid_constant__ CUtensorMap tm_keys, const __grid_constant__ CUtensorMap tm_q,
                      const __grid_constant__ CUtensorMap tm_ks, IdxArgs a) {
  using C = IdxCfg<G, kFp8>;
  constexpr int N = C::N;
  pdl_trigger();
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* qbuf = smem;                  // [kQSlots][2 boxes][N rows][128 B]
  uint8_t* kbuf = smem + C::kOffK;       // [kStages][2 boxes][128 rows][128 B]
  float* wbuf = reinterpret_cast<float*>(smem + C::kOffW);
  float* rcos = reinterpret_cast<float*>(smem + C::kOffRope);
  float* rsin = rcos + G * 32;
  uint8_t* sbuf = smem + C::kOffS;  // fp8: [kScaleSlots][128 rows][16 B], the row's scale first
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBars);
  uint64_t* full = bars;                        // [kStages] key tile landed
  uint64_t* empty = full + C::kStages;          // [kStages] key tile consumed
  uint64_t* q_full = empty + C::kStages;        // [kQSlots] query block and weights written
  uint64_t* q_empty = q_full + C::kQSlots;      // [kQSlots] last MMA of the group retired
  uint64_t* w_empty = q_empty + C::kQSlots;     // [kQSlots] epilogue done with the group's weights
  uint64_t* acc_full = w_empty + C::kQSlots;    // [kAcc]
  uint64_t* acc_empty = acc_full + C::kAcc;     // [kAcc]
  uint64_t* drain = acc_empty + C::kAcc;
  uint64_t* q_loaded = drain + 1;               // [kQSlots] G = 4: the query block's TMA copy landed
  uint64_t* s_full = q_loaded + C::kQSlots;     // [kScaleSlots] fp8: a tile's key scales landed
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(s_full + C::kScaleSlots);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      tc::mbar_init(&full[s], 1);
      tc::mbar_init(&empty[s], 1);
    }
    for (int s = 0; s < C::kQSlots; ++s) {
      tc::mbar_init(&q_full[s], kPrepThreads);
      tc::mbar_init(&q_empty[s], 1);
      tc::mbar_init(&w_empty[s], C::kEpiWarps);
    }
    for (int i = 0; i < C::kAcc; ++i) {
      tc::mbar_init(&acc_full[i], 1);
      tc::mbar_init(&acc_empty[i], 32 * C::kEpiWarps);
    }
    tc::mbar_init(drain, 1);
    for (int i = 0; i < C::kScaleSlots; ++i) tc::mbar_init(&s_full[i], 1);
    tc::fence_mbar_init();
  }
  // Query-block warps: everything the first query block needs (positions, frequencies, head weights and the first
  // batch of query chunks) is requested before the preceding kernel has completed: these are step inputs and
  // constants that no kernel writes.  16 chunks of 8 dims per head row; each thread takes 16 (G = 1) or 64 (G = 4)
  // chunks, in batches whose loads are all issued before any is used.
  // fp8: 8 chunks of 16 codes per head row, copied from the quantised queries (no RoPE here: the queries were
  // roped and quantised by the kernel before)
  constexpr int kChunksPerRow = kFp8 ? 8 : 16;
  constexpr int kBatch = G == 1 ? (kFp8 ? 8 : 16) : 8;  // prefill: fewer registers (twelve warps share the file)
  constexpr int kChunks = G * 64 * kChunksPerRow;
  const int pt = threadIdx.x - 32 * C::kPrepWarp0;
  struct Pre {
    uint4 raw[kBatch];
    float wv[G];
    float qsv;  // fp8: the scale of head pt
    float th_freq;
    int p;
  };
  // G = 4: the block of group g by TMA (rows 64 q0 .. + 255 of [Q*64, 128], q0 its first query; rows past the last
  // query read zeros, rows of another sequence's queries in a group of fewer than four are masked by the epilogue)
  auto issue_q = [&](int g) {
    if (pt == 0) {
      int cnt;
      const int q0 = grp_first<G>(a, g, cnt);
      tc::mbar_arrive_expect_tx(&q_loaded[0], C::kQBytes);
      tc::tma_load_2d(qbuf, &tm_q, &q_loaded[0], 0, q0 * 64);
      if constexpr (!kFp8)  // fp8: one 128-byte box of codes per head row
        tc::tma_load_2d(qbuf + C::kQBytes / 2, &tm_q, &q_loaded[0], 64, q0 * 64);
    }
  };
  // G = 1 (not overlapped): query g's block, already roped (bf16, k_rope_iq16) or quantised (fp8, k_quant_iq) by
  // the kernel before, copied by TMA into slot `slot`
  auto issue_q1 = [&](int g, int slot) {
    tc::mbar_arrive_expect_tx(&q_loaded[slot], C::kQBytes);
    tc::tma_load_2d(qbuf + slot * C::kQBytes, &tm_q, &q_loaded[slot], 0, g * 64);
    if constexpr (!kFp8)  // fp8: one 128-byte box of codes per head row
      tc::tma_load_2d(qbuf + slot * C::kQBytes + C::kQBytes / 2, &tm_q, &q_loaded[slot], 64, g * 64);
  };
  // fp8 (G = 1): group g's codes and head pt's scale, the preceding kernel's output (so after the wait); loads
  // that stay where they are written (the second group's must not be moved behind the key stream)
  auto load_codes = [&](int g, Pre& pre, bool codes = true) {
#pragma unroll
    for (int b = 0; b < kBatch && codes; ++b) {
      const int e = pt + b * kPrepThreads, h = (e >> 3) & 63, c = e & 7;
      pre.raw[b] = tc::ld_nc_v4_now(a.q8 + ((size_t)g * 64 + h) * 128 + c * 16);
    }
    pre.qsv = __uint_as_float(tc::ld_nc_u32_now(a.qs + (size_t)g * 64 + pt));
  };
  // (rows = false: everything but the query rows)
  auto load_first = [&](int g, Pre& pre, bool rows = true) {
    if constexpr (!kFp8 && G != 4) {
#pragma unroll
      for (int b = 0; b < kBatch && rows; ++b) {
        const int e = pt + b * kPrepThreads;
        const int q = g * G + (e >> 10), h = (e >> 4) & 63, c = e & 15;
        pre.raw[b] = (e < kChunks && q < a.Q)
                         ? __ldg(reinterpret_cast<const uint4*>(a.iq + ((size_t)q * 64 + h) * 128 + c * 8))
                         : make_uint4(0, 0, 0, 0);
      }
    }
#pragma unroll
    for (int i = 0; i < G; ++i) {
      const int e = pt + i * kPrepThreads, q = grp_query<G>(a, g, e / 64);
      if constexpr (kFp8 && G == 4)  // the folded weights, the preceding kernel's output (load_first runs after the wait)
        pre.wv[i] = q >= 0 ? a.w8[(size_t)q * 64 + (e & 63)] : 0.f;
      else
        pre.wv[i] = q >= 0 ? __bfloat162float(a.iw[(size_t)q * 64 + (e & 63)]) : 0.f;
    }
    // RoPE table entry e = pt (G = 1: threads 0-31) or pt, pt + 64 (G = 4: two per thread, see below)
    pre.th_freq = (pt & 31) < a.R / 2 ? __ldg(a.inv_freq + (pt & 31)) : 0.f;
    const int q0 = pt < G * 32 ? grp_query<G>(a, g, pt / 32) : -1;
    pre.p = q0 >= 0 ? idx_qpos(a, q0) : 0;
  };
  // Static partition of the items, weighted: each group costs its tiles plus group_penalty tile-equivalents (the
  // query block a CTA must build when its range enters the group), placed before the group's first tile.  A CTA
  // whose range crosses into a second group therefore gets fewer tiles; measured in the decode step, such CTAs
  // otherwise finished ~3 us (about three tiles) after the others and held up the successor.
  int i_begin, i_end;
  {
    const int unit = a.tiles_per_group + a.group_penalty;
    const long long total = (long long)(a.n_items / a.tiles_per_group) * unit;
    auto item_at = [&](long long x) {  // first item at or after cost position x
      const int g = (int)(x / unit), r = (int)(x - (long long)g * unit);
      return g * a.tiles_per_group + max(0, r - a.group_penalty);
    };
    const long long x0 = total * blockIdx.x / gridDim.x, x1 = total * (blockIdx.x + 1) / gridDim.x;
    i_begin = min(a.n_items, item_at(x0));
    i_end = blockIdx.x + 1 == gridDim.x ? a.n_items : min(a.n_items, item_at(x1));
  }
  Pre pre_a, pre_b;  // pre_b: the range's second group (fp8, or bf16 with roped copies)
  bool g1_loaded = false, q_copies = false;
  // bf16 decode (G = 1, not overlapped): the queries come roped from the kernel before, and the blocks of the range's
  // first two groups are copied by TMA right after the wait, before the key stream starts; the query warps then
  // only write the head weights (measured: behind the stream a load round trip takes ~10 us and 16 KB of
  // shared-memory stores ~8 us, so a block built there started a CTA's scan ~8 us after its wait)
  constexpr bool kRopedCopy = G == 1 && !kOverlap;  // (fp8: the codes of k_quant_iq, the same way)
  const int g0 = min(i_begin, a.n_items - 1) / a.tiles_per_group;
  const int g1 = (g0 + 1) * a.tiles_per_group < i_end ? g0 + 1 : -1;
  // The first query block is requested before the wait (step inputs), except with a group table, fp8 queries or
  // roped copies (G = 1), which the kernel before writes.  G = 4: the range's first group is copied now; whether it has tiles is known only after
  // the wait (a prefill chunk's first groups may have none), so the loop below drains this copy if it starts at a
  // later group.
  if (warp >= C::kPrepWarp0 && i_begin < i_end) {
    if ((G == 4 || kRopedCopy) && pt == 0) {
      // this thread issues the block copies: it initialises their barriers itself, ahead of the CTA-wide sync
      for (int sl = 0; sl < C::kQSlots; ++sl) tc::mbar_init(&q_loaded[sl], 1);
      tc::fence_mbar_init();
      tc::tma_prefetch(&tm_q);
    }
    if (G != 4 || !(a.gcu || kFp8)) {
      if (G == 4) issue_q(g0);
      load_first(g0, pre_a, !kRopedCopy);
      // fp8 and roped copies: the second group's weights and position too
      if ((kFp8 || kRopedCopy) && g1 >= 0) load_first(g1, pre_b, false);
    }
  }
  // The overlapped decode scan does not wait for its predecessors here: it reads only index-key rows complete
  // before the token and the step's inputs, and writes only its own scratch, so it runs beside the compress
  // call's kernels; it waits for them at its end instead, so that its successor's wait covers them.  (It follows
  // a projection kernel that lets successors start only once all earlier work is complete.)
  if (!kOverlap) pdl_wait();  // predecessor complete: its outputs are visible and its tensor memory is free
  // fp8: the quantised queries and their scales are the preceding kernel's output; the head scales of the range's
  // first two groups are requested now, before the key stream starts (a load issued behind the stream took ~10 us)
  if constexpr (kFp8 && G == 1) {  // (the codes come by TMA, below)
    if (warp >= C::kPrepWarp0 && i_begin < i_end) {
      load_codes(g0, pre_a, false);
      if (g1 >= 0) load_codes(g1, pre_b, false);
    }
  }
  if constexpr (G == 4) {
    if ((a.gcu || kFp8) && warp >= C::kPrepWarp0 && i_begin < i_end) {
      issue_q(g0);
      load_first(g0, pre_a);
    }
  }
  if constexpr (kRopedCopy) {
    if (warp >= C::kPrepWarp0 && i_begin < i_end) {
      if (pt == 0) {
        issue_q1(g0, 0);
        if (g1 >= 0) issue_q1(g1, 1);
      }
      q_copies = true;
      g1_loaded = g1 >= 0;
    }
  }
  if (warp == 1) {
    tc::tmem_alloc(tmem_slot, C::kAcc * N);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_slot;

  bool failed = false;

  if (warp == 0) {
    // ------------------------------------------------------------ key tiles (TMA)
    // the ring starts once the query-block warps have issued their requests (issued behind a full ring of key
    // tiles, those few loads would wait in the same queues; issuing the first tiles at the programmatic wait
    // instead, or before it, measured slower)
    tc::named_bar(4, 32 + kPrepThreads);
    if (lane == 0) {
      tc::tma_prefetch(&tm_keys);
      if constexpr (kFp8) tc::tma_prefetch(&tm_ks);
      int stage = 0;
      uint32_t phase = 0;
      uint32_t used = 0, par_last = 0;  // per stage (bit s): a load was issued; parity of its last phase
      int n_items = 0;                  // fp8: items issued (scale slot n_items % kScaleSlots)
      uint32_t s_used = 0, s_par = 0;   // fp8: per scale slot, as used / par_last
      Items<G, kOverlap> itr;
      for (bool more = itr.start(a, i_begin, i_end); more; more = itr.advance(a)) {
        const int g = itr.g, t = itr.t;
        if (!tc::mbar_wait(&empty[stage], phase ^ 1)) { failed = true; break; }
        int cnt;
        const int krow = idx_seq(a, grp_first<G>(a, g, cnt)) * a.cap + t * kTileRows;  // a group's queries share
                                                                                   // a sequence
        tc::mbar_arrive_expect_tx(&full[stage], C::kTileBytes);
        tc::tma_load_2d(kbuf + stage * C::kTileBytes, &tm_keys, &full[stage], 0, krow);
        if constexpr (!kFp8)
          tc::tma_load_2d(kbuf + stage * C::kTileBytes + C::kTileBytes / 2, &tm_keys, &full[stage], 64, krow);
        if constexpr (kFp8) {
          const int ss = n_items % C::kScaleSlots;
          const uint32_t sp = (uint32_t)(n_items / C::kScaleSlots) & 1;
          tc::mbar_arrive_expect_tx(&s_full[ss], C::kScaleBytes);
          tc::tma_load_2d(sbuf + ss * C::kScaleBytes, &tm_ks, &s_full[ss], 128, krow);
          s_used |= 1u << ss;
          s_par = (s_par & ~(1u << ss)) | (sp << ss);
          ++n_items;
        }
        used |= 1u << stage;
        par_last = (par_last & ~(1u << stage)) | (phase << stage);
        if (++stage == C::kStages) { stage = 0; phase ^= 1; }
      }
      // every load issued must land before the CTA may exit
      for (int s = 0; s < C::kStages; ++s)
        if (((used >> s) & 1) && !tc::mbar_wait(&full[s], (par_last >> s) & 1)) failed = true;
      for (int s = 0; s < C::kScaleSlots; ++s)
        if (((s_used >> s) & 1) && !tc::mbar_wait(&s_full[s], (s_par >> s) & 1)) failed = true;
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = tc::idesc_bf16(128, N);
      int cur_g = -1, k = -1, stage = 0, acc = 0;
      uint32_t acc_par = 0;  // bit i: parity of accumulator i's uses so far
      uint32_t phase = 0;
      Items<G, kOverlap> itr;
      for (bool more = itr.start(a, i_begin, i_end); more; more = itr.advance(a)) {
        const int g = itr.g;
        if (g != cur_g) {
          ++k;
          cur_g = g;
          if (!tc::mbar_wait(&q_full[k % C::kQSlots], (k / C::kQSlots) & 1)) { failed = true; break; }
        }
        if (!tc::mbar_wait(&full[stage], phase)) { failed = true; break; }
        if (!tc::mbar_wait(&acc_empty[acc], ((acc_par >> acc) & 1) ^ 1)) { failed = true; break; }
        tc::fence_after_sync();
        const uint32_t a_base = tc::smem_u32(kbuf + stage * C::kTileBytes);
        const uint32_t b_base = tc::smem_u32(qbuf + (k % C::kQSlots) * C::kQBytes);
        if constexpr (kFp8) {
          // K = 128 E4M3 elements: four 32-element steps inside one 128-byte swizzled row
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint64_t ad = tc::sdesc_kmajor_sw128(a_base + kk * 32);
            const uint64_t bd = tc::sdesc_kmajor_sw128(b_base + kk * 32);
            tc::mma_f8(tmem + acc * N, ad, bd, tc::idesc_e4m3(128, N), kk > 0);
          }
        } else {
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint64_t ad = tc::sdesc_kmajor_sw128(a_base + (kk >> 2) * (C::kTileBytes / 2) + (kk & 3) * 32);
            const uint64_t bd = tc::sdesc_kmajor_sw128(b_base + (kk >> 2) * (C::kQBytes / 2) + (kk & 3) * 32);
            tc::mma_bf16(tmem + acc * N, ad, bd, idesc, kk > 0);
          }
        }
        tc::mma_commit(&empty[stage]);
        tc::mma_commit(&acc_full[acc]);
        if (itr.last_of_group()) tc::mma_commit(&q_empty[k % C::kQSlots]);
        acc_par ^= 1u << acc;
        if (++acc == C::kAcc) acc = 0;
        if (++stage == C::kStages) { stage = 0; phase ^= 1; }
      }
      // every MMA retires before tensor memory is released
      tc::mma_commit(drain);
      if (!tc::mbar_wait(drain, 0)) failed = true;
    }
  } else if (warp < C::kPrepWarp0) {
    // ------------------------------------------------------------ epilogue: warp w drains TMEM lanes 32*(w%4)
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    int cur_g = -1, k = -1, acc = 0;
    uint32_t acc_par = 0;  // bit i: parity of accumulator i's uses so far
    int nv[G], qix[G];
    int n_done = 0;  // fp8: items taken (scale slot n_done % kScaleSlots)
    Items<G, kOverlap> itr;
    for (bool more = itr.start(a, i_begin, i_end); more; more = itr.advance(a)) {
      const int g = itr.g, t = itr.t;
      if (g != cur_g) {
        ++k;
        cur_g = g;
        if (!tc::mbar_wait(&q_full[k % C::kQSlots], (k / C::kQSlots) & 1)) { failed = true; break; }
#pragma unroll
        for (int qq = 0; qq < G; ++qq) {
          qix[qq] = grp_query<G>(a, g, qq);
          nv[qq] = qix[qq] >= 0 ? scan_rows<kOverlap>(a, qix[qq]) : 0;
        }
      }
      const int j = t * kTileRows + row;
      float kscale = 1.f;  // fp8: the key row's scale, from the tile's scale slot
      if constexpr (kFp8) {
        const int ss = n_done % C::kScaleSlots;
        if (!tc::mbar_wait(&s_full[ss], (uint32_t)(n_done / C::kScaleSlots) & 1)) { failed = true; break; }
        kscale = *reinterpret_cast<const float*>(sbuf + ss * C::kScaleBytes + row * 16);
        ++n_done;
      }
      if (!tc::mbar_wait(&acc_full[acc], (acc_par >> acc) & 1)) { failed = true; break; }
      tc::fence_after_sync();
      const float4* w4 = reinterpret_cast<const float4*>(wbuf + (k % C::kQSlots) * N);
      // this warp's queries (kQPerWarp of them) in one TMEM round trip (one wait covers every load)
      {
        constexpr int kPer = C::kQPerWarp;
        const int qp = ((warp - 2) >> 2) * kPer;
        uint32_t v[kPer][64];
#pragma unroll
        for (int u = 0; u < kPer; ++u) {
          const uint32_t taddr = tmem + ((uint32_t)(quarter * 32) << 16) + acc * N + (qp + u) * 64;
          tc::tmem_ld32(taddr, v[u]);
          tc::tmem_ld32(taddr + 32, v[u] + 32);
        }
        tc::tmem_wait_ld();
#pragma unroll
        for (int u = 0; u < kPer; ++u) {
          const int qq = qp + u;
          // four partial sums (heads h = 0, 1, 2, 3 mod 4, each in increasing h) as two packed fp32 pairs, then
          // (p0 + p1) + (p2 + p3): four independent chains instead of one of 64 dependent FMAs
          float2 s01 = make_float2(0.f, 0.f), s23 = make_float2(0.f, 0.f);
#pragma unroll
          for (int h4 = 0; h4 < 16; ++h4) {
            const float4 w = w4[qq * 16 + h4];
            const float2 r01 = make_float2(fmaxf(__uint_as_float(v[u][4 * h4]), 0.f),
                                           fmaxf(__uint_as_float(v[u][4 * h4 + 1]), 0.f));
            const float2 r23 = make_float2(fmaxf(__uint_as_float(v[u][4 * h4 + 2]), 0.f),
                                           fmaxf(__uint_as_float(v[u][4 * h4 + 3]), 0.f));
            s01 = __ffma2_rn(make_float2(w.x, w.y), r01, s01);
            s23 = __ffma2_rn(make_float2(w.z, w.w), r23, s23);
          }
          float s = (s01.x + s01.y) + (s23.x + s23.y);
          if constexpr (kFp8) s *= kscale;  // ReLU(k s) = k ReLU(s) for the row's scale k >= 0
          if (j < nv[qq]) a.scores[(size_t)qix[qq] * a.cap + j] = s;
        }
      }
      tc::fence_before_sync();
      tc::mbar_arrive(&acc_empty[acc]);
      if (itr.last_of_group()) {
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&w_empty[k % C::kQSlots]);
      }
      acc_par ^= 1u << acc;
      if (++acc == C::kAcc) acc = 0;
    }
  } else {
    // ------------------------------------------------------------ query blocks (the last two warps)
    // The first group's inputs were requested before the wait above (load_first), so its preparation costs about
    // one memory round trip, overlapped with the preceding kernel.
    auto rope_store = [&](uint8_t* qb, int e0, uint4 (&raw)[kBatch], int g) {
      if constexpr (kFp8) {  // codes as they are, into the one 128-byte swizzled box of each head row
#pragma unroll
        for (int b = 0; b < kBatch; ++b) {
          const int e = e0 + b * kPrepThreads;
          if (e >= kChunks) break;
          const int row = ((e >> 9) << 6) + ((e >> 3) & 63), c = e & 7;
          *reinterpret_cast<uint4*>(qb + row * 128 + ((c ^ (row & 7)) << 4)) = raw[b];
        }
        return;
      }
#pragma unroll
      for (int b = 0; b < kBatch; ++b) {
        const int e = e0 + b * kPrepThreads;
        if (e >= kChunks) break;
        const int qq = e >> 10, h = (e >> 4) & 63, c = e & 15, row = qq * 64 + h;
        if (c * 8 >= 128 - a.R && g * G + qq < a.Q) {
          __nv_bfloat162* hv = reinterpret_cast<__nv_bfloat162*>(&raw[b]);
#pragma unroll
          for (int kq = 0; kq < 4; ++kq) {
            const int i = qq * 32 + (c * 8 - (128 - a.R)) / 2 + kq;
            const float2 x = __bfloat1622float2(hv[kq]);
            hv[kq] = __floats2bfloat162_rn(fmaf(x.x, rcos[i], -x.y * rsin[i]), fmaf(x.x, rsin[i], x.y * rcos[i]));
          }
        }
        *reinterpret_cast<uint4*>(qb + (c >> 3) * (C::kQBytes / 2) + row * 128 + (((c & 7) ^ (row & 7)) << 4)) =
            raw[b];
        if (kOverlap && g * G + qq < a.Q)  // every CTA preparing this query writes the same bytes
          *reinterpret_cast<uint4*>(a.qr_out + ((size_t)(g * G + qq) * 64 + h) * 128 + c * 8) = raw[b];
      }
    };
    // the first group of the range was requested up front (before the key stream saturates memory and stretches
    // every round trip); the second is prefetched into L2
    if (g1 >= 0) {
      int cnt1;
      const int q01 = grp_first<G>(a, g1, cnt1);
      if constexpr (kFp8) {
        for (int e = pt; e < 16 * G; e += kPrepThreads)  // 512 B a thread: 16 threads per block of codes
          if (e / 16 < cnt1) tc::prefetch_l2(a.q8 + (size_t)q01 * 8192 + e * 512, 512);
      } else {
        for (int e = pt; e < 32 * G; e += kPrepThreads)  // 512 B a thread: 32 threads per query block
          if (e / 32 < cnt1) tc::prefetch_l2(a.iq + ((size_t)q01 * 64 + e * 2) * 128, 512);
      }
    }
    tc::named_bar_arrive(4, 32 + kPrepThreads);  // releases the key-tile producer
    int k = -1;
    int q_pending = (G == 4 && i_begin < i_end) ? g0 : -1;  // G = 4: group whose block copy is in flight
    uint32_t q_waits = 0;                                  // G = 4: completed phases of q_loaded
    auto wait_q = [&]() {
      const bool ok = tc::mbar_wait(&q_loaded[0], q_waits & 1);
      ++q_waits;
      q_pending = -1;
      return ok;
    };
    Items<G, kOverlap> itr;
    for (bool more = itr.start(a, i_begin, i_end); more; more = itr.next_group(a)) {
      const int g = itr.g;
      ++k;
      const int slot = k % C::kQSlots, use = k / C::kQSlots;
      if (use > 0) {
        const bool ok = tc::mbar_wait(&q_empty[slot], (use - 1) & 1) && tc::mbar_wait(&w_empty[slot], (use - 1) & 1);
        if (tc::named_bar_any(3, kPrepThreads, !ok)) { failed = true; break; }
      } else {
        tc::named_bar(3, kPrepThreads);  // the previous group's RoPE table is no longer read
      }
      if constexpr (kRopedCopy) {
        if (k == 0) {  // both copies land before any slot is written or read
          const bool ok = tc::mbar_wait(&q_loaded[0], 0) && (!g1_loaded || tc::mbar_wait(&q_loaded[1], 0));
          if (tc::named_bar_any(3, kPrepThreads, !ok)) { failed = true; break; }
          q_copies = false;  // landed
        }
        // fp8: the head's query scale and the 1/128 of the unnormalised rotation go into its weight
        auto weight = [&](const Pre& pc) {
          return (kFp8 ? pc.wv[0] * (pc.qsv * 0.0078125f) : pc.wv[0]) * a.wscale;
        };
        if ((k == 0 && g == g0) || (k == 1 && g == g1 && g1_loaded)) {
          wbuf[slot * N + pt] = weight(k == 0 ? pre_a : pre_b);  // the block was copied into this slot
        } else {  // a range that skips its first group, or a third group: the block is built here
          load_first(g, pre_a);
          if constexpr (kFp8) load_codes(g, pre_a);
          if (!kFp8 && pt < 32) sincosf(__fmul_rn((float)pre_a.p, pre_a.th_freq), &rsin[pt], &rcos[pt]);
          tc::named_bar(3, kPrepThreads);
          rope_store(qbuf + slot * C::kQBytes, pt, pre_a.raw, g);
          wbuf[slot * N + pt] = weight(pre_a);
        }
        tc::fence_proxy_async_smem();
        tc::mbar_arrive(&q_full[slot]);
        continue;
      }
      Pre& pre = pre_a;
      if (g != g0) load_first(g, pre_a);  // a later group: request it now
      if constexpr (G == 4) {
        if (q_pending != g) {
          // the slot is free (first group, or the previous group's MMAs retired); a copy of a group without
          // tiles still in flight is drained first
          if (q_pending >= 0 && tc::named_bar_any(3, kPrepThreads, !wait_q())) { failed = true; break; }
          issue_q(g);
          q_pending = g;
        }
      }
      // RoPE table (G x 32 entries) from the preloaded position and frequency (fp8: roped before quantisation)
      for (int e = pt; !kFp8 && e < G * 32; e += kPrepThreads) {
        int p = pre.p;
        float f = pre.th_freq;
        if (e != pt) {  // G = 4: the second entry of this thread
          const int q = grp_query<G>(a, g, e / 32);
          p = q >= 0 ? idx_qpos(a, q) : 0;
          f = (e & 31) < a.R / 2 ? __ldg(a.inv_freq + (e & 31)) : 0.f;
        }
        sincosf(__fmul_rn((float)p, f), &rsin[e], &rcos[e]);
      }
      tc::named_bar(3, kPrepThreads);
      uint8_t* qb = qbuf + slot * C::kQBytes;
      if constexpr (G == 4) {
        // RoPE in place on the copied block: 16-byte chunks c >= (128 - R) / 8 of each of the N head rows (fp8:
        // the codes were roped before quantisation)
        if (tc::named_bar_any(3, kPrepThreads, !wait_q())) { failed = true; break; }
        const int c0 = (128 - a.R) / 8, nrc = 16 - c0;
        for (int e = pt; !kFp8 && e < N * nrc; e += kPrepThreads) {
          const int row = e / nrc, c = c0 + e % nrc, qq = row >> 6;
          uint4* slot_p =
              reinterpret_cast<uint4*>(qb + (c >> 3) * (C::kQBytes / 2) + row * 128 + (((c & 7) ^ (row & 7)) << 4));
          uint4 raw = *slot_p;
          __nv_bfloat162* hv = reinterpret_cast<__nv_bfloat162*>(&raw);
#pragma unroll
          for (int kq = 0; kq < 4; ++kq) {
            const int i = qq * 32 + (c * 8 - (128 - a.R)) / 2 + kq;
            const float2 x = __bfloat1622float2(hv[kq]);
            hv[kq] = __floats2bfloat162_rn(fmaf(x.x, rcos[i], -x.y * rsin[i]), fmaf(x.x, rsin[i], x.y * rcos[i]));
          }
          *slot_p = raw;
        }
      } else {
        rope_store(qb, pt, pre.raw, g);
        for (int e0 = pt + kPrepThreads * kBatch; e0 < kChunks; e0 += kPrepThreads * kBatch) {
          uint4 raw[kBatch];
#pragma unroll
          for (int b = 0; b < kBatch; ++b) {
            const int e = e0 + b * kPrepThreads;
            const int q = g * G + (e >> 10), h = (e >> 4) & 63, c = e & 15;
            raw[b] = (e < kChunks && q < a.Q)
                         ? __ldg(reinterpret_cast<const uint4*>(a.iq + ((size_t)q * 64 + h) * 128 + c * 8))
                         : make_uint4(0, 0, 0, 0);
          }
          rope_store(qb, e0, raw, g);
        }
      }
#pragma unroll
      for (int i = 0; i < G; ++i) {
        // fp8: the head's query scale and the 1/128 of the unnormalised rotation go into its weight
        // (G = 4: the folded weights already hold them)
        const float w = (kFp8 && G == 1 ? pre.wv[i] * (pre.qsv * 0.0078125f) : pre.wv[i]) * a.wscale;
        wbuf[slot * N + pt + i * kPrepThreads] = w;
        const int e = pt + i * kPrepThreads;
        if (kOverlap && g * G + e / 64 < a.Q) a.w_out[(size_t)(g * G) * 64 + e] = w;
      }
      tc::fence_proxy_async_smem();
      tc::mbar_arrive(&q_full[slot]);
    }
    // a block copy that no group used (a range without tiles) lands before the CTA exits
    if (G == 4 && q_pending >= 0 && !wait_q()) failed = true;
    if (kRopedCopy && q_copies) {
      if (!tc::mbar_wait(&q_loaded[0], 0)) failed = true;
      if (g1_loaded && !tc::mbar_wait(&q_loaded[1], 0)) failed = true;
    }
  }
  if (failed) atomicOr(a.err, tc::kErrTimeout);
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 1) tc::tmem_dealloc(tmem, C::kAcc * N);
  if (kOverlap) pdl_wait();  // complete only after the kernels it ran beside
}

int g_num_sms = 0;

// fp8 index queries (the optional key format): query q's head h, RoPE at pos[q] as for the bf16 scores, rounded
// to bf16, rotated by the unnormalised 128-point Walsh-Hadamard transform in fp32 (butterflies of span 1, 2, ..,
// 64 in that order), scaled by amax / 448 and rounded to E4M3 (nearest even, saturating): q8 [Q, 64, 128] codes,
// qs [Q, 64] scales, and (w8 non-null) the head weights with the scale and the 1/128 of the unnormalised rotation
// folded in, w8 [Q, 64] = iw qs / 128.  Query q's position as the scan takes it (pos, pos0, qps, cu: see
// idx_qpos).  Block (q, quarter): 16 warps, one head each (heads 16 quarter ..); lane l holds elements 4l .. 4l + 3.
// Everything up to the stores reads step inputs only (queries, positions, frequencies), so it runs before the
// programmatic wait, beside the preceding kernels; the stores wait for them (the workspace may still be read by an
// earlier call).
constexpr int kQuantHeads = 16;
__global__ void __launch_bounds__(32 * kQuantHeads) k_quant_iq(const __nv_bfloat16* __restrict__ iq,
                                                               const __nv_bfloat16* __restrict__ iw,
                                                               const int32_t* __restrict__ pos, int pos0, int qps,
                                                               const int32_t* __restrict__ cu, int nseq,
                                                               const float* __restrict__ inv_freq, int R,
                                                               uint8_t* __restrict__ q8, float* __restrict__ qs,
                                                               float* __restrict__ w8) {
  pdl_trigger();
  __shared__ float rc[64], rs[64];
  const int q = blockIdx.x, h = blockIdx.y * kQuantHeads + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  const uint2 raw = __ldg(reinterpret_cast<const uint2*>(iq + ((size_t)q * 64 + h) * 128 + 4 * lane));
  const float wh = w8 ? __bfloat162float(iw[(size_t)q * 64 + h]) : 0.f;
  if (threadIdx.x < R / 2) {
    int p;
    if (cu) {
      const int b = varlen_seq(cu, nseq, q);
      p = __ldg(pos + b) + q - __ldg(cu + b);
    } else {
      p = pos ? __ldg(pos + q / qps) + q % qps : pos0 + q;
    }
    sincosf(__fmul_rn((float)p, __ldg(inv_freq + threadIdx.x)), &rs[threadIdx.x], &rc[threadIdx.x]);
  }
  __syncthreads();
  const __nv_bfloat162* hv = reinterpret_cast<const __nv_bfloat162*>(&raw);
  float u[4];
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    const int i0 = 4 * lane + 2 * k;  // element pair (i0, i0 + 1)
    const float2 x = __bfloat1622float2(hv[k]);
    if (i0 >= 128 - R) {
      const int i = (i0 - (128 - R)) >> 1;
      const float2 y = __bfloat1622float2(
          __floats2bfloat162_rn(fmaf(x.x, rc[i], -x.y * rs[i]), fmaf(x.x, rs[i], x.y * rc[i])));
      u[2 * k] = y.x;
      u[2 * k + 1] = y.y;
    } else {
      u[2 * k] = x.x;
      u[2 * k + 1] = x.y;
    }
  }
  float scale;
  const uint32_t packed = fp8_rotate_quantize(u, lane, &scale);
  pdl_wait();
  *reinterpret_cast<uint32_t*>(q8 + ((size_t)q * 64 + h) * 128 + 4 * lane) = packed;
  if (lane == 0) {
    qs[(size_t)q * 64 + h] = scale;
    if (w8) w8[(size_t)q * 64 + h] = wh * (scale * 0.0078125f);
  }
}

// Roped bf16 index queries for the one-query scan: qr [Q, 64, 128], query q at pos[q / qps] + q % qps, its last R
// dims roped (the scan's arithmetic: fp32 angle, sincosf, one fused multiply-add a component, bf16).  Block (q,
// quarter): 16 warps, one head each; lane l holds elements 4l .. 4l + 3.  Everything up to the stores reads step
// inputs only, so it runs before the programmatic wait, beside the preceding kernels.
__global__ void __launch_bounds__(32 * kQuantHeads) k_rope_iq16(const __nv_bfloat16* __restrict__ iq,
                                                                const int32_t* __restrict__ pos, int qps,
                                                                const float* __restrict__ inv_freq, int R,
                                                                __nv_bfloat16* __restrict__ qr) {
  pdl_trigger();
  __shared__ float rc[64], rs[64];
  const int q = blockIdx.x, h = blockIdx.y * kQuantHeads + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  const size_t off = ((size_t)q * 64 + h) * 128 + 4 * lane;
  uint2 raw = __ldg(reinterpret_cast<const uint2*>(iq + off));
  if (threadIdx.x < R / 2) {
    const int p = __ldg(pos + q / qps) + q % qps;
    sincosf(__fmul_rn((float)p, __ldg(inv_freq + threadIdx.x)), &rs[threadIdx.x], &rc[threadIdx.x]);
  }
  __syncthreads();
  __nv_bfloat162* hv = reinterpret_cast<__nv_bfloat162*>(&raw);
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    const int i0 = 4 * lane + 2 * k;  // element pair (i0, i0 + 1)
    if (i0 >= 128 - R) {
      const int i = (i0 - (128 - R)) >> 1;
      const float2 x = __bfloat1622float2(hv[k]);
      hv[k] = __floats2bfloat162_rn(fmaf(x.x, rc[i], -x.y * rs[i]), fmaf(x.x, rs[i], x.y * rc[i]));
    }
  }
  pdl_wait();
  *reinterpret_cast<uint2*>(qr + off) = raw;
}

// gcu[b] = sum over sequences before b of ceil(T_b / 4) (T_b = cu[b+1] - cu[b], an inconsistent entry counted as
// empty), b = 0 .. nseq: one block, each thread a contiguous share of the sequences, then a block scan.
__global__ void __launch_bounds__(1024) k_varlen_groups(const int32_t* __restrict__ cu, int nseq,
                                                        int32_t* __restrict__ gcu) {
  pdl_trigger();
  pdl_wait();
  __shared__ int wsum[32];
  const int per = (nseq + blockDim.x - 1) / blockDim.x;
  const int b0 = min(nseq, (int)threadIdx.x * per), b1 = min(nseq, b0 + per);
  auto groups = [&](int b) { return (max(0, cu[b + 1] - cu[b]) + 3) / 4; };
  int mine = 0;
  for (int b = b0; b < b1; ++b) mine += groups(b);
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  int incl = mine;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += n;
  }
  if (lane == 31) wsum[wid] = incl;
  __syncthreads();
  int base = 0;
  for (int w = 0; w < wid; ++w) base += wsum[w];
  int run = base + incl - mine;
  for (int b = b0; b < b1; ++b) {
    gcu[b] = run;
    run += groups(b);
  }
  if (threadIdx.x == blockDim.x - 1) gcu[nseq] = run;
}

}  // namespace

// (RoPE on whole 16-byte chunks of a head row, with one 32-entry table per query)
bool tc_index_supported(const Dims& L) {
  return L.dtype == CSA_BF16 && L.Hi == 64 && L.Di == 128 && L.R <= 64 && L.R % 8 == 0;
}

size_t tc_index_ws(const Dims& L, int Q) {
  (void)L;
  return (size_t)Q * 64 * 128 * 2 + 256 + (size_t)Q * 64 * 4 + 256;
}

cudaError_t launch_tc_index_scores(const Dims& L, const void* iq, const void* iw, int Q, const void* ikeys, int Bk,
                                   int cap, const int32_t* n_rows, const int32_t* pos, int pos0,
                                   const float* inv_freq, void* ws, float* scores, int32_t* err, cudaStream_t s,
                                   bool overlap, const int32_t* cu, bool fp8) {
  if (!g_num_sms) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&g_num_sms, cudaDevAttrMultiProcessorCount, dev);
  }
  // queries per MMA: 4 for a prefill chunk, a packed variable-length batch (groups of four of one sequence, from a
  // group table) and verify blocks whose length is a multiple of 4 (a group's queries share every key tile, one
  // read for four), else 1 (decode)
  const int G = cu ? 4 : (!pos ? 4 : (pos0 > 1 && pos0 % 4 == 0 ? 4 : 1));
  CUtensorMap tk, tq;
  if (!make_tmap_2d_bf16(&tk, ikeys, (uint64_t)Bk * cap, 128, 256, kTileRows)) return cudaErrorInvalidValue;
  // the 4-query instance copies each group's query block (4 x 64 head rows) by TMA
  if (!make_tmap_2d_bf16(&tq, iq, (uint64_t)Q * 64, 128, 256, 64 * G)) return cudaErrorInvalidValue;
  IdxArgs a{};
  a.iq = static_cast<const __nv_bfloat16*>(iq);
  a.iw = static_cast<const __nv_bfloat16*>(iw);
  a.inv_freq = inv_freq;
  a.wscale = (float)(1.0 / sqrt((double)L.Di * (double)L.Hi));
  a.R = L.R;
  a.n_rows = n_rows; a.pos = pos; a.pos0 = pos0; a.ratio = L.ratio; a.topk = L.topk; a.cap = cap; a.Q = Q;
  a.qps = pos ? max(1, pos0) : 1;  // with device positions pos0 carries the queries per sequence
  a.cu = cu;
  a.nseq = cu ? pos0 : 0;         // ... and with a row table, the number of sequences
  if (cu && (!pos || pos0 < 1)) return cudaErrorInvalidValue;
  a.G = G; a.tiles_per_group = (cap + kTileRows - 1) / kTileRows;
  // groups: Q / G rounded up; with a row table at most (Q + 3 nseq) / 4 (every sequence's last group may be short;
  // groups past the table's total have no tiles)
  const long long n_groups = cu ? ((long long)Q + 3LL * a.nseq) / 4 : (Q + G - 1) / G;
  if (n_groups * a.tiles_per_group > INT32_MAX) return cudaErrorInvalidValue;
  a.n_items = (int)(n_groups * a.tiles_per_group);
  if (cu) {
    // the group table goes into the query-output area of ws, which only the overlapped decode scan uses
    if (!ws) return cudaErrorInvalidValue;
    a.gcu = static_cast<const int32_t*>(ws);
    CSA_LAUNCH(k_varlen_groups, dim3(1), dim3(1024), 0, s, cu, a.nseq, static_cast<int32_t*>(ws));
  }
  a.group_penalty = G == 1 ? 3 : 0;
  a.scores = scores; a.err = err;
  if (overlap) {
    if (!pos || G != 1) return cudaErrorInvalidValue;
    a.qr_out = static_cast<__nv_bfloat16*>(ws);
    a.w_out = reinterpret_cast<float*>(static_cast<char*>(ws) + (size_t)Q * 64 * 128 * 2);
  }
  const int grid = min(g_num_sms, a.n_items);
  if (fp8) {
    // the quantised queries go into the query-output area of ws (after the group table, if any): codes
    // [Q, 64, 128], scales [Q, 64] and, for 4-query groups, the folded head weights [Q, 64]; the keys are fp8 rows
    if (overlap || !ws) return cudaErrorInvalidValue;
    const size_t off = cu ? ((size_t)(a.nseq + 1) * 4 + 255) / 256 * 256 : 0;
    auto* q8 = static_cast<uint8_t*>(ws) + off;
    auto* qsc = reinterpret_cast<float*>(q8 + (size_t)Q * 64 * 128);
    float* w8 = G == 4 ? qsc + (size_t)Q * 64 : nullptr;
    CSA_LAUNCH(k_quant_iq, dim3(Q, 64 / kQuantHeads), dim3(32 * kQuantHeads), 0, s,
               static_cast<const __nv_bfloat16*>(iq), static_cast<const __nv_bfloat16*>(iw), pos, pos0, a.qps, cu,
               a.nseq, inv_freq, L.R, q8, qsc, w8);
    // the key rows' codes (bytes 0-127, swizzled) and scales (bytes 128-143) by two tensor maps; 4-query groups
    // copy their 256 code rows by TMA too
    CUtensorMap tk8, tks, tq8;
    if (!make_tmap_2d_u8(&tk8, ikeys, (uint64_t)Bk * cap, kFp8RowBytes, kFp8RowBytes, 128, kTileRows, true) ||
        !make_tmap_2d_u8(&tks, ikeys, (uint64_t)Bk * cap, kFp8RowBytes, kFp8RowBytes, 16, kTileRows, false) ||
        !make_tmap_2d_u8(&tq8, q8, (uint64_t)Q * 64, 128, 128, 128, 64 * G, true))
      return cudaErrorInvalidValue;
    a.q8 = q8;
    a.qs = qsc;
    a.w8 = w8;
    if (G == 1) {
      constexpr int smem = IdxCfg<1, true>::kSmem;
      cudaFuncSetAttribute(k_tc_index_scores<1, false, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
      CSA_LAUNCH(k_tc_index_scores<1, false, true>, dim3(grid), dim3(IdxCfg<1, true>::kThreads), smem, s, tk8, tq8,
                 tks, a);
    } else {
      constexpr int smem = IdxCfg<4, true>::kSmem;
      cudaFuncSetAttribute(k_tc_index_scores<4, false, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
      CSA_LAUNCH(k_tc_index_scores<4, false, true>, dim3(grid), dim3(IdxCfg<4, true>::kThreads), smem, s, tk8, tq8,
                 tks, a);
    }
    return cudaGetLastError();
  }
  if (G == 1 && !overlap) {
    // the queries roped by a kernel of their own into the query-output area of ws, copied into the scan by TMA
    if (!pos || !ws) return cudaErrorInvalidValue;
    auto* qr16 = static_cast<__nv_bfloat16*>(ws);
    CSA_LAUNCH(k_rope_iq16, dim3(Q, 64 / kQuantHeads), dim3(32 * kQuantHeads), 0, s,
               static_cast<const __nv_bfloat16*>(iq), pos, a.qps, inv_freq, L.R, qr16);
    CUtensorMap tqr;
    if (!make_tmap_2d_bf16(&tqr, qr16, (uint64_t)Q * 64, 128, 256, 64)) return cudaErrorInvalidValue;
    constexpr int smem = IdxCfg<1>::kSmem;
    cudaFuncSetAttribute(k_tc_index_scores<1, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    CSA_LAUNCH(k_tc_index_scores<1, false>, dim3(grid), dim3(IdxCfg<1>::kThreads), smem, s, tk, tqr, tk, a);
    return cudaGetLastError();
  }
  if (G == 1 && overlap) {
    constexpr int smem = IdxCfg<1>::kSmem;
    cudaFuncSetAttribute(k_tc_index_scores<1, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    CSA_LAUNCH(k_tc_index_scores<1, true>, dim3(grid), dim3(IdxCfg<1>::kThreads), smem, s, tk, tq, tk, a);
  } else if (G == 1) {
    constexpr int smem = IdxCfg<1>::kSmem;
    cudaFuncSetAttribute(k_tc_index_scores<1, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    CSA_LAUNCH(k_tc_index_scores<1, false>, dim3(grid), dim3(IdxCfg<1>::kThreads), smem, s, tk, tq, tk, a);
  } else {
    constexpr int smem = IdxCfg<4>::kSmem;
    cudaFuncSetAttribute(k_tc_index_scores<4, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    CSA_LAUNCH(k_tc_index_scores<4, false>, dim3(grid), dim3(IdxCfg<4>::kThreads), smem, s, tk, tq, tk, a);
  }
  return cudaGetLastError();
}

}  // namespace csa
