// Decode attention on the 5th-generation tensor cores for the Flash shapes (64
// query heads over one 512-dim latent, K = V, bf16, RoPE on the last 64 dims):
// one CTA per (query, key split) of up to 160 rows.
//
// Definitions: "DeepSeek-V4-Flash: native deepseek_v4 AR backend" (MTPLX #216),
// "What V4 adds" (MQA-shaped MLA with per-head sink logits) and "Decode path"
// (bf16 in/out, fp32 softmax state, the probability block cast to bf16 before
// the PV product); "deepseek-v41-mlx" README (inverse rope on the output, sinks
// in the denominator only).
//
// Why 160 rows: a decode query attends to topk + W = 640 rows; four splits of
// 160 put a batch of 32 on 128 CTAs, one wave of the 152 SMs, where 128-row
// splits would need 160 CTAs and a second wave.  Each CTA takes its split's rows
// as one chunk: its share of the window tokens (the newest one roped here) and
// the query block, both copied before the programmatic wait since they depend
// only on the step's inputs, then its share of the selected pool rows once the
// selection is known; all gathered with cp.async into one 160-row, 128-byte-swizzled shared tile
// that serves both as K (K-major) and as V^T (MN-major), so each row is read from
// memory once.
//   QK       S^T = K Q^T twice, M = 128 (TMEM lanes), N = 64 heads, K = 512:
//            rows 0-127, and rows 128-255 of which lanes 0-31 (rows 128-159) are
//            used (the rest read neighbouring, initialised shared memory);
//   softmax  five warps, thread = row (warp 4 reads lanes 0-31 of the second
//            product); per-head column max and sum by a warp reduce-scatter and a
//            5-warp combine;
//   PV       O^T = V^T [P_hi | P_lo]^T: M = 128 latent dims x 4 tiles, N = 2 x 64,
//            K = the chunk's rows.  Once both score products have retired, the
//            query's shared memory holds P^T as two bf16 parts side by side,
//            P_hi = bf16(P) and P_lo = bf16(P - P_hi), so one read of V serves both
//            and the epilogue adds the two halves (~16 bits of P in the product).
// With one split the epilogue finalises the output (sink, normalisation, bf16,
// inverse RoPE, bf16); with several it writes (m, l, acc) partials for the merge
// kernel.  Splits are never longer than 160 rows (the caller picks enough).
#include "common.cuh"
#include "kernels.h"
#include "tc.cuh"

namespace csa {

namespace {

constexpr int kCR = 160;                 // rows per chunk
constexpr int kAD = 512;                 // latent dims
constexpr int kAH = 64;                  // heads
constexpr int kBox = kCR * 128;          // 64 dims x 160 rows (20 KB)
constexpr int kRowsBytes = 8 * kBox;     // 160 KB
constexpr int kQBox = kAH * 128;         // 64 dims x 64 heads (8 KB)
constexpr int kQBytes = 8 * kQBox;       // 64 KB
constexpr int kPPart = kCR * 128;        // P^T part: 160 rows x 64 heads, MN-major (20 KB)
constexpr int kMainWarps = kCR / 32;     // gather / softmax threads: one per row (warps 0-4)
constexpr int kMain = 32 * kMainWarps;
constexpr int kMmaWarp = kMainWarps;     // TMEM owner and MMA issuer
constexpr int kEpiWarps = 8;             // epilogue: every warp, two per TMEM lane quarter (warps 6-7 join there)
constexpr int kThreads = 32 * kEpiWarps;
constexpr int kTmemCols = 512;           // S^T (cols 0-127), then O^T over all 512 (hi | lo per 128-dim tile)
constexpr float kLn2 = 0.6931471805599453f;

// shared memory: rows | query (after the score products: P_hi, P_lo, column reductions) | small state
constexpr int kOffQ = kRowsBytes;
constexpr int kOffRed = kOffQ + 2 * kPPart;     // [5][64] column maxima
constexpr int kOffRedSum = kOffRed + kMainWarps * 64 * 4;
static_assert(kOffRedSum + kMainWarps * 64 * 4 <= kOffQ + kQBytes, "reductions fit in the query region");
constexpr int kOffMref = kOffQ + kQBytes;
constexpr int kOffLsum = kOffMref + 64 * 4;
constexpr int kOffRope = kOffLsum + 64 * 4;     // cos[32], sin[32]
constexpr int kOffRowc = kOffRope + 64 * 4;     // [160] row codes
constexpr int kOffBars = kOffRowc + kCR * 4;    // 5 mbarriers
constexpr int kOffTmem = kOffBars + 8 * 8;
constexpr int kSmem = kOffTmem + 16 + 1024;     // + alignment slack
static_assert(kSmem <= 232448, "shared memory per block");

// row codes: >= 0 pool row (b * cap + j); kRowNone: empty; kRowNew: the new token; <= kRowRing0: ring row
constexpr int kRowNone = -1;
constexpr int kRowNew = -2;
constexpr int kRowRing0 = -3;

struct DecArgs {
  const __nv_bfloat16* q;       // [Q, 64, 512] queries before RoPE
  const __nv_bfloat16* pool;    // [B, cap, 512]
  __nv_bfloat16* ring;          // [B, W, 512]; the new token is written to slot pos % W
  const __nv_bfloat16* kv_new;  // [B, 512] the new token before RoPE
  const int32_t* sel;           // [Q, topk] or null (every visible row)
  const int32_t* n_sel;
  const int32_t* n_rows;
  const int32_t* pos;
  const float* sink;
  const float* inv_freq;
  int cap, topk, W, ratio, S;
  int Wr;                       // ring slots (W + rollback); the query attends its last W tokens
  int qps;                      // consecutive queries per sequence (a verify block; 1 for decode)
  int kv_in_ring;               // the new tokens are already in the ring (verify): none is roped here
  int cluster;                  // S in {2, 4}: the S splits of a query are one cluster and merge through DSMEM
  float scale2;                 // softmax scale * log2(e)
  float* part_ml;
  float* part_acc;
  __nv_bfloat16* out;
  int32_t* err;
};

// Reduce 64 columns over the 32 lanes of a warp; lane L returns columns 2L, 2L+1.
template <bool kMax>
__device__ __forceinline__ float2 reduce_scatter64(float (&v)[64]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int st = 0; st < 5; ++st) {
    const int half = 32 >> st, mask = 16 >> st;
    const bool upper = (lane & mask) != 0;
#pragma unroll
    for (int i = 0; i < half; ++i) {
      const float send = upper ? v[i] : v[i + half];
      const float keep = upper ? v[i + half] : v[i];
      const float recv = __shfl_xor_sync(0xffffffffu, send, mask);
      v[i] = kMax ? fmaxf(keep, recv) : keep + recv;
    }
  }
  return make_float2(v[0], v[1]);
}

// One (query, split) item.  The split's tile holds its share of the window first (known from the position alone,
// so it is gathered before the programmatic wait), then its share of the selection (known after it):
//   rows [0, nw)        window tokens w_begin .. w_begin + nw - 1 (of the query's nwin window tokens);
//   rows [nw, nw + ns)  selected rows s_begin .. s_begin + ns - 1 (of nsel).
struct Item {
  int q, s, b, p, nwin, w_begin, nw;  // before the wait
  int nrows, nsel, s_begin, ns;       // after it
};

__device__ __forceinline__ Item make_item(const DecArgs& a) {
  Item it;
  it.q = blockIdx.x / a.S;
  it.s = blockIdx.x % a.S;
  it.b = it.q / a.qps;
  it.p = a.pos[it.b] + it.q % a.qps;
  it.nwin = it.p >= 0 ? min(a.W, it.p + 1) : 0;
  const int wper = (it.nwin + a.S - 1) / a.S;
  it.w_begin = min(it.nwin, it.s * wper);
  it.nw = min(it.nwin, it.w_begin + wper) - it.w_begin;
  it.nrows = it.nsel = it.s_begin = it.ns = 0;
  return it;
}

// the selection share (reads the predecessors' outputs: call after the programmatic wait)
__device__ __forceinline__ void item_selection(const DecArgs& a, Item& it) {
  it.nrows = min(a.n_rows[it.b], a.cap);
  it.nsel = a.sel ? min(max(a.n_sel[it.q], 0), a.topk) : max(0, min(it.nrows, (it.p + 1) / a.ratio));
  const int sper = (it.nsel + a.S - 1) / a.S;
  it.s_begin = min(it.nsel, it.s * sper);
  it.ns = min(it.nsel, it.s_begin + sper) - it.s_begin;
  if (it.nw + it.ns > kCR) it.ns = max(0, kCR - it.nw);  // callers keep both shares within one tile
}

// Code of window token w (0 .. nwin-1, oldest first) and of selected row k (0 .. nsel-1; j = sel[q][k] when a
// selection is given); an out-of-range selection is reported and left empty.
__device__ __forceinline__ int window_code(const DecArgs& a, const Item& it, int w) {
  const int tok = it.p - it.nwin + 1 + w;
  if (tok == it.p && !a.kv_in_ring) return kRowNew;
  return kRowRing0 - (it.b * a.Wr + tok % a.Wr);
}
__device__ __forceinline__ int selected_code(const DecArgs& a, const Item& it, int k, int j) {
  if (!a.sel) j = k;
  if (j >= 0 && j < it.nrows) return it.b * a.cap + j;
  atomicOr(a.err, CSA_DEV_RANGE);
  return kRowNone;
}

__device__ __forceinline__ const __nv_bfloat16* code_ptr(const DecArgs& a, int code) {
  if (code >= 0) return a.pool + (size_t)code * kAD;
  if (code <= kRowRing0) return a.ring + (size_t)(kRowRing0 - code) * kAD;
  return nullptr;
}

__device__ __forceinline__ void rope8(uint4& raw, int c, const float* rcos, const float* rsin) {
  __nv_bfloat162* hv = reinterpret_cast<__nv_bfloat162*>(&raw);
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int f = (c - 56) * 4 + k;
    const float2 x = __bfloat1622float2(hv[k]);
    hv[k] = __floats2bfloat162_rn(fmaf(x.x, rcos[f], -x.y * rsin[f]), fmaf(x.x, rsin[f], x.y * rcos[f]));
  }
}

// 2^x by the hardware approximation (relative error ~2^-22; results below 2^-126 flush to zero)
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// probabilities of one row into both P^T parts (MN-major, 128-byte swizzle); returns them in pe (fp32)
__device__ __forceinline__ void write_p(uint8_t* pbuf, int row, const float (&sv)[64], const float* mref,
                                        float (&pe)[64]) {
#pragma unroll
  for (int h4 = 0; h4 < 16; ++h4) {
    const float4 r4 = reinterpret_cast<const float4*>(mref)[h4];
    const float rr[4] = {r4.x, r4.y, r4.z, r4.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int h = 4 * h4 + k;
      const float ref = rr[k] == -INFINITY ? 0.f : rr[k];
      pe[h] = sv[h] == -INFINITY ? 0.f : ex2_approx(sv[h] - ref);
    }
  }
  uint8_t* dst = pbuf + (row >> 3) * 1024 + (row & 7) * 128;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    uint4 hi, lo;
    __nv_bfloat162* hv = reinterpret_cast<__nv_bfloat162*>(&hi);
    __nv_bfloat162* lv = reinterpret_cast<__nv_bfloat162*>(&lo);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      hv[k] = __floats2bfloat162_rn(pe[8 * j + 2 * k], pe[8 * j + 2 * k + 1]);
      const float2 back = __bfloat1622float2(hv[k]);
      lv[k] = __floats2bfloat162_rn(pe[8 * j + 2 * k] - back.x, pe[8 * j + 2 * k + 1] - back.y);
    }
    const int off = (j ^ (row & 7)) << 4;
    *reinterpret_cast<uint4*>(dst + off) = hi;
    *reinterpret_cast<uint4*>(dst + kPPart + off) = lo;
  }
}

// Copy tile rows [r0, r1) from their codes (cp.async, 2 x 512 contiguous bytes per warp instruction; rows spread
// over the main warps); an empty row is zero-filled and the new token is skipped (roped separately).
__device__ __forceinline__ void gather_rows(const DecArgs& a, const int* rowc, uint32_t r_base, int r0, int r1) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
#pragma unroll 4
  for (int r = r0 + warp; r < r1; r += kMainWarps) {
    const int code = rowc[r];
    if (code == kRowNew) continue;
    const __nv_bfloat16* src = code_ptr(a, code);
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      const int ch = lane + 32 * hh;
      const uint32_t dst = r_base + (ch >> 3) * kBox + r * 128 + (((ch & 7) ^ (r & 7)) << 4);
      tc::cp_async16(dst, src ? static_cast<const void*>(src + ch * 8) : static_cast<const void*>(a.pool),
                     src ? 16u : 0u);
    }
  }
}

// S > 1 writes (m, l, acc) partials for the merge kernel; S == 1 finalises directly.
__global__ void __launch_bounds__(kThreads, 1) k_tc_attend_decode(DecArgs a) {
  pdl_trigger();
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* rows = smem;
  uint8_t* qbuf = smem + kOffQ;
  uint8_t* pbuf = qbuf;  // P^T parts reuse the query region once the score products have retired
  float* red = reinterpret_cast<float*>(smem + kOffRed);
  float* red_sum = reinterpret_cast<float*>(smem + kOffRedSum);
  float* mref = reinterpret_cast<float*>(smem + kOffMref);
  float* lsum = reinterpret_cast<float*>(smem + kOffLsum);
  float* rcos = reinterpret_cast<float*>(smem + kOffRope);
  float* rsin = rcos + 32;
  int* rowc = reinterpret_cast<int*>(smem + kOffRowc);
  uint64_t* rows_full = reinterpret_cast<uint64_t*>(smem + kOffBars);  // rows and roped query in place
  uint64_t* s_full = rows_full + 1;    // both score products retired
  uint64_t* p_full = rows_full + 2;    // both P parts written
  uint64_t* pv_done = rows_full + 3;   // PV retired
  uint64_t* drain = rows_full + 4;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffTmem);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    tc::mbar_init(rows_full, kMain);
    tc::mbar_init(s_full, 1);
    tc::mbar_init(p_full, kMain);
    tc::mbar_init(pv_done, 1);
    tc::mbar_init(drain, 1);
    tc::fence_mbar_init();
  }
  Item it = make_item(a);
  const uint32_t r_base = tc::smem_u32(rows), q_base = tc::smem_u32(qbuf);
  if (warp < kMainWarps) {
    // ---- before the programmatic wait: the query block, the RoPE table, this split's window rows and the new
    // token (step inputs and the window ring, which no kernel of this step writes before this one)
    const int row = tid;
    {
      const __nv_bfloat16* qsrc = a.q + (size_t)it.q * kAH * kAD;
#pragma unroll 8
      for (int e = tid; e < kAH * 64; e += kMain) {
        const int h = e >> 6, ch = e & 63;
        tc::cp_async16(q_base + (ch >> 3) * kQBox + h * 128 + (((ch & 7) ^ (h & 7)) << 4),
                       qsrc + (size_t)h * kAD + ch * 8, 16u);
      }
    }
    if (row < it.nw) rowc[row] = window_code(a, it, it.w_begin + row);
    if (tid < 32) {
      float cs, sn;
      rope_cs(it.p, a.inv_freq, tid, &cs, &sn);
      rcos[tid] = cs;
      rsin[tid] = sn;
    }
    tc::named_bar(1, kMain);
    gather_rows(a, rowc, r_base, 0, it.nw);
    // the new token (the window's last): RoPE at p, into the tile and into its ring slot (the slot belongs to the
    // token leaving the window, which no CTA reads)
    const int cur_row = (!a.kv_in_ring && it.nw > 0 && it.w_begin + it.nw == it.nwin) ? it.nw - 1 : -1;
    if (cur_row >= 0 && warp == cur_row % kMainWarps) {
      const __nv_bfloat16* cur = a.kv_new + (size_t)it.b * kAD;
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const int ch = lane + 32 * hh;
        uint4 raw = __ldg(reinterpret_cast<const uint4*>(cur + ch * 8));
        if (ch >= 56) rope8(raw, ch, rcos, rsin);
        *reinterpret_cast<uint4*>(rows + (ch >> 3) * kBox + cur_row * 128 + (((ch & 7) ^ (cur_row & 7)) << 4)) = raw;
        *reinterpret_cast<uint4*>(a.ring + ((size_t)it.b * a.Wr + (it.p % a.Wr)) * kAD + ch * 8) = raw;
      }
    }
    tc::cp_async_wait_all();
    tc::named_bar(1, kMain);  // every thread's share of the query block has landed
#pragma unroll
    for (int e = tid; e < kAH * 8; e += kMain) {
      const int h = e >> 3, ch = 56 + (e & 7);
      uint4* slot = reinterpret_cast<uint4*>(qbuf + (ch >> 3) * kQBox + h * 128 + (((ch & 7) ^ (h & 7)) << 4));
      uint4 raw = *slot;
      rope8(raw, ch, rcos, rsin);
      *slot = raw;
    }
  }
  pdl_wait();  // predecessors complete: the selection is visible and their tensor memory is free
  if (warp == kMmaWarp) {
    tc::tmem_alloc(tmem_slot, kTmemCols);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  const uint32_t tm_s = tmem;  // S^T: rows 0-127 in cols 0-63, rows 128-255 in cols 64-127
  const uint32_t tm_o = tmem;  // O^T tile m: cols 128m + (0-63: P_hi part, 64-127: P_lo part); overwrites S^T
  item_selection(a, it);
  const int nr = it.nw + it.ns;
  bool failed = false;

  if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && nr > 0) {
      constexpr uint32_t id_qk = tc::idesc_bf16(128, 64);
      constexpr uint32_t id_pv = tc::idesc_bf16(128, 128, true, true);
      const uint32_t p_base = tc::smem_u32(pbuf);
      do {
        if (!tc::mbar_wait(rows_full, 0)) { failed = true; break; }
        tc::fence_after_sync();
#pragma unroll 1
        for (int half = 0; half < (nr > 128 ? 2 : 1); ++half) {
          const uint32_t a_off = half ? 128 * 128 : 0;  // rows 128-255: sixteen 8-row atoms further
#pragma unroll 8
          for (int k = 0; k < 32; ++k) {
            const uint64_t ad = tc::sdesc_kmajor_sw128(r_base + (k >> 2) * kBox + a_off + (k & 3) * 32);
            const uint64_t bd = tc::sdesc_kmajor_sw128(q_base + (k >> 2) * kQBox + (k & 3) * 32);
            tc::mma_bf16(tm_s + 64 * half, ad, bd, id_qk, k > 0);
          }
        }
        tc::mma_commit(s_full);
        if (!tc::mbar_wait(p_full, 0)) { failed = true; break; }
        tc::fence_after_sync();
        // O^T tile m += V^T [P_hi | P_lo]^T: one read of V serves both parts (N = 2 x 64)
        const int ksteps = (nr + 15) >> 4;
#pragma unroll
        for (int m = 0; m < 4; ++m) {
#pragma unroll 1
          for (int kk = 0; kk < ksteps; ++kk) {
            const uint64_t ad = tc::sdesc_mnmajor_sw128(r_base + 2 * m * kBox + kk * 2048, kBox, 1024);
            const uint64_t bd = tc::sdesc_mnmajor_sw128(p_base + kk * 2048, kPPart, 1024);
            tc::mma_bf16(tm_o + 128 * m, ad, bd, id_pv, kk > 0);
          }
        }
        tc::mma_commit(pv_done);
      } while (false);
    }
    __syncwarp();
    failed = __shfl_sync(0xffffffffu, (int)failed, 0) != 0;
  } else if (warp < kMainWarps) {
    // ------------------------------------------------------------ main warps (160 threads, one per row)
    const int row = tid;
    // ---- the selection share: codes of rows nw .. 159 (empty past nr), then their copies
    if (row >= it.nw) {
      const int k = it.s_begin + (row - it.nw);
      const int j = (a.sel && row < nr) ? a.sel[(size_t)it.q * a.topk + k] : 0;
      rowc[row] = row < nr ? selected_code(a, it, k, j) : kRowNone;
    }
    tc::named_bar(1, kMain);
    gather_rows(a, rowc, r_base, it.nw, kCR);
    tc::cp_async_wait_all();
    tc::fence_proxy_async_smem();
    tc::fence_before_sync();
    tc::mbar_arrive(rows_full);
    do {
      if (nr <= 0) {
        if (tid < 64) {
          mref[tid] = -INFINITY;
          lsum[tid] = 0.f;
        }
        break;
      }
      // ---- scores of this thread's row: rows 0-127 from the first product, rows 128-159 from lanes 0-31 of
      // the second (read by warp 4, whose TMEM lane quarter is lanes 0-31)
      if (tc::named_bar_any(2, kMain, !tc::mbar_wait(s_full, 0))) { failed = true; break; }
      tc::fence_after_sync();
      float sv[64];
      if (warp < 4 || nr > 128) {
        const uint32_t ta = warp < 4 ? tm_s + ((uint32_t)(warp * 32) << 16) : tm_s + 64;
        uint32_t u[64];
        tc::tmem_ld32(ta, u);
        tc::tmem_ld32(ta + 32, u + 32);
        tc::tmem_wait_ld();
        const bool valid = row < nr && rowc[row] != kRowNone;
#pragma unroll
        for (int h = 0; h < 64; ++h) sv[h] = valid ? __uint_as_float(u[h]) * a.scale2 : -INFINITY;
      } else {
#pragma unroll
        for (int h = 0; h < 64; ++h) sv[h] = -INFINITY;
      }
      {
        float cp[64];
#pragma unroll
        for (int h = 0; h < 64; ++h) cp[h] = sv[h];
        const float2 m2 = reduce_scatter64<true>(cp);
        red[warp * 64 + 2 * lane] = m2.x;
        red[warp * 64 + 2 * lane + 1] = m2.y;
      }
      tc::named_bar(1, kMain);
      if (tid < 64) {
        float mt = red[tid];
#pragma unroll
        for (int w = 1; w < kMainWarps; ++w) mt = fmaxf(mt, red[64 * w + tid]);
        mref[tid] = mt;
      }
      tc::named_bar(1, kMain);
      // ---- probabilities (fp32 for the sums, bf16 hi + lo for the PV product)
      float pe[64];
      write_p(pbuf, row, sv, mref, pe);
      tc::fence_proxy_async_smem();
      tc::fence_before_sync();
      tc::mbar_arrive(p_full);
      {
        const float2 s2 = reduce_scatter64<false>(pe);
        red_sum[warp * 64 + 2 * lane] = s2.x;
        red_sum[warp * 64 + 2 * lane + 1] = s2.y;
      }
      tc::named_bar(1, kMain);
      if (tid < 64) {
        float st = red_sum[tid];
#pragma unroll
        for (int w = 1; w < kMainWarps; ++w) st += red_sum[64 * w + tid];
        lsum[tid] = st;
      }
      if (tc::named_bar_any(2, kMain, !tc::mbar_wait(pv_done, 0))) { failed = true; break; }
      tc::fence_after_sync();
    } while (false);
    tc::cp_async_wait_all();
    tc::named_bar(1, kMain);
  }
  // ---- epilogue (every warp, once the main warps have seen the PV product retire): warp w reads TMEM lane quarter
  // w % 4 and takes the O^T tiles {0, 1} (w < 4) or {2, 3} (w >= 4); a thread owns latent dim 128 m + 32 (w % 4) +
  // lane of each; O = hi + lo parts.  Eight warps halve the partial write of four.
  failed = __syncthreads_or(failed) != 0;
  tc::fence_after_sync();
  const int quarter = warp & 3, dl = quarter * 32 + lane, m0 = (warp >> 2) * 2;
  auto load_o = [&](int m, float (&o)[64]) {
      if (nr <= 0) {
#pragma unroll
        for (int h = 0; h < 64; ++h) o[h] = 0.f;
        return;
      }
      const uint32_t ta = tm_o + 128 * m + ((uint32_t)(quarter * 32) << 16);
      uint32_t u[64];
      tc::tmem_ld32(ta, u);
      tc::tmem_ld32(ta + 32, u + 32);
      tc::tmem_wait_ld();
#pragma unroll
      for (int h = 0; h < 64; ++h) o[h] = __uint_as_float(u[h]);
      tc::tmem_ld32(ta + 64, u);
      tc::tmem_ld32(ta + 96, u + 32);
      tc::tmem_wait_ld();
#pragma unroll
      for (int h = 0; h < 64; ++h) o[h] += __uint_as_float(u[h]);
    };
  if (a.cluster) {
    // The query's S splits are one cluster.  Each leaves its O (hi + lo, fp32), its per-head reference max (natural
    // log units) and row sum in its own row tile (free once PV retired); after a cluster barrier, rank r merges
    // dims [r D/S, (r+1) D/S) of all S with the arithmetic of the merge kernel, reading the others' shared memory.
    // A second barrier keeps every CTA's shared memory in place until the others have read it.  Every thread
    // reaches both barriers, a failed CTA too (its output is then invalid and the error word says so).
    float* accs = reinterpret_cast<float*>(rows);  // [64 heads][512]
    float* mls = accs + kAH * kAD;                 // [64][2]
    float* tab = mls + 2 * kAH;                    // [64][S + 1]: weights f_s, then 1 / Z
    const int S = a.S;
    if (!failed) {
      if (tid < 64) {
        mls[2 * tid] = mref[tid] == -INFINITY ? -INFINITY : mref[tid] * kLn2;
        mls[2 * tid + 1] = lsum[tid];
      }
      for (int m = m0; m < m0 + 2; ++m) {
        float o[64];
        load_o(m, o);
#pragma unroll
        for (int h = 0; h < 64; ++h) accs[h * kAD + 128 * m + dl] = o[h];
      }
    }
    tc::cluster_sync();
    if (tid < 64) {
      // M = max(z, m_s); f_s = e^{m_s - M} (0 for a split without rows); Z = e^{z - M} + sum_s l_s f_s
      const float z = a.sink[tid];
      float ms[4], ls[4];
      float M = z;
#pragma unroll
      for (int sp = 0; sp < 4; ++sp) {
        if (sp < S) {
          const float2 v = tc::ld_cluster_f2(tc::cluster_map(mls + 2 * tid, sp));
          ms[sp] = v.x;
          ls[sp] = v.y;
          M = fmaxf(M, v.x);
        }
      }
      float zs = 0.f;
#pragma unroll
      for (int sp = 0; sp < 4; ++sp) {
        if (sp < S) {
          const float f = ms[sp] == -INFINITY ? 0.f : expf(ms[sp] - M);
          tab[tid * (S + 1) + sp] = f;
          zs = fmaf(ls[sp], f, zs);
        }
      }
      tab[tid * (S + 1) + S] = 1.0f / (expf(z - M) + zs);
    }
    __syncthreads();
    // warp w: heads 8w .. 8w + 7, four at a time with every split's values requested together (one remote round
    // trip per four heads; one per head measured slower, and so did a remote store of every value, and fetching
    // the splits' statistics in the same round); lane: 4-dim columns of this rank's slice.  A split's values are
    // read whatever its weight (a split without rows left zeros) and added only when the weight is not zero.
    const int r = it.s, ncol = kAD / 4 / S;
    for (int c = lane; c < ncol; c += 32) {
      const int d = r * (kAD / S) + 4 * c;
#pragma unroll 1
      for (int h0 = warp * 8; h0 < warp * 8 + 8; h0 += 4) {
        float4 x[4][4];
#pragma unroll
        for (int hh = 0; hh < 4; ++hh)
#pragma unroll
          for (int sp = 0; sp < 4; ++sp)
            if (sp < S) x[hh][sp] = tc::ld_cluster_f4(tc::cluster_map(accs + (h0 + hh) * kAD + d, sp));
#pragma unroll
        for (int hh = 0; hh < 4; ++hh) {
        const int h = h0 + hh;
        float v[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int sp = 0; sp < 4; ++sp) {
          const float f = sp < S ? tab[h * (S + 1) + sp] : 0.f;
          if (f != 0.f) {
            v[0] = fmaf(x[hh][sp].x, f, v[0]);
            v[1] = fmaf(x[hh][sp].y, f, v[1]);
            v[2] = fmaf(x[hh][sp].z, f, v[2]);
            v[3] = fmaf(x[hh][sp].w, f, v[3]);
          }
        }
        const float invZ = tab[h * (S + 1) + S];
#pragma unroll
        for (int e = 0; e < 4; ++e) v[e] = rnd<__nv_bfloat16>(v[e] * invZ);
        if (d >= kAD - 64) {
#pragma unroll
          for (int e = 0; e < 4; e += 2) {
            const int i = (d + e - (kAD - 64)) >> 1;
            const float x0 = v[e], x1 = v[e + 1];
            v[e] = fmaf(x0, rcos[i], x1 * rsin[i]);
            v[e + 1] = fmaf(-x0, rsin[i], x1 * rcos[i]);
          }
        }
        uint2 pk;
        __nv_bfloat162* hv = reinterpret_cast<__nv_bfloat162*>(&pk);
        hv[0] = __floats2bfloat162_rn(v[0], v[1]);
        hv[1] = __floats2bfloat162_rn(v[2], v[3]);
        *reinterpret_cast<uint2*>(a.out + ((size_t)it.q * kAH + h) * kAD + d) = pk;
        }
      }
    }
    tc::cluster_sync();
  } else if (!failed) {
    if (a.S > 1) {
      if (tid < 64) {
        const size_t idx = ((size_t)it.q * a.S + it.s) * kAH + tid;
        a.part_ml[idx * 2] = mref[tid] == -INFINITY ? -INFINITY : mref[tid] * kLn2;
        a.part_ml[idx * 2 + 1] = lsum[tid];
      }
      if (nr > 0) {
        for (int m = m0; m < m0 + 2; ++m) {
          float o[64];
          load_o(m, o);
          float* dst = a.part_acc + (((size_t)it.q * a.S + it.s) * kAH) * kAD + 128 * m + dl;
#pragma unroll
          for (int h = 0; h < 64; ++h) dst[(size_t)h * kAD] = o[h];
        }
      }
    } else {
      for (int m = m0; m < m0 + 2; ++m) {
        const int d = 128 * m + dl;
        float o[64];
        load_o(m, o);
        __nv_bfloat16* dst = a.out + (size_t)it.q * kAH * kAD + d;
#pragma unroll
        for (int h = 0; h < 64; ++h) {
          const float z2 = a.sink[h] * 1.4426950408889634f;
          const float mr = mref[h];
          const float M2 = fmaxf(z2, mr);
          const float f = mr == -INFINITY ? 0.f : exp2f(mr - M2);
          const float Z = exp2f(z2 - M2) + lsum[h] * f;
          float v = rnd<__nv_bfloat16>(o[h] * (f / Z));
          const float partner = __shfl_xor_sync(0xffffffffu, v, 1);
          if (d >= kAD - 64) {
            const int i = (d - (kAD - 64)) >> 1;
            v = (d & 1) ? fmaf(-partner, rsin[i], v * rcos[i]) : fmaf(v, rcos[i], partner * rsin[i]);
          }
          dst[(size_t)h * kAD] = __float2bfloat16_rn(v);
        }
      }
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

int g_sms_dec = 0;

}  // namespace

bool tc_attend_decode_supported(const Dims& L) {
  return L.dtype == CSA_BF16 && L.H == kAH && L.D == kAD && L.R == 64;
}

// Splits per query: the fewest S whose window share ceil(W / S) plus selection share ceil(n_max / S) fit one
// 160-row tile, more (up to one per 128 rows) while every CTA still fits one wave of the device's SMs.  0 when
// max_splits (the workspace's partial capacity) cannot hold enough.
int tc_attend_decode_splits(int Q, int W, int n_max, int max_splits) {
  if (!g_sms_dec) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&g_sms_dec, cudaDevAttrMultiProcessorCount, dev);
  }
  auto fits = [&](int S) { return (W + S - 1) / S + (n_max + S - 1) / S <= kCR; };
  int s_min = max(1, (W + n_max + kCR - 1) / kCR);
  while (!fits(s_min)) ++s_min;
  if (s_min > max_splits) return 0;
  const int s_tiles = (W + n_max + 127) / 128;
  const int s_fit = g_sms_dec / max(1, Q);
  return min(max_splits, max(s_min, min(s_fit, s_tiles)));
}

// Whether the S splits of a query can run as one cluster (S in {2, 4}, and the device can place such a cluster of
// these CTAs); asked once per S.
bool tc_attend_decode_cluster(int S) {
  static int known[5] = {-1, -1, -1, -1, -1};
  if (S != 2 && S != 4) return false;
  if (known[S] < 0) {
    cudaFuncSetAttribute(k_tc_attend_decode, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(S);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = S;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    const cudaError_t e = cudaOccupancyMaxActiveClusters(&n, k_tc_attend_decode, &cfg);
    if (e != cudaSuccess) cudaGetLastError();  // leave no sticky error behind
    known[S] = (e == cudaSuccess && n > 0) ? 1 : 0;
  }
  return known[S] == 1;
}

cudaError_t launch_tc_attend_decode(const Dims& L, const void* q, const void* pool, void* ring, const void* kv_new,
                                    const int32_t* sel, const int32_t* n_sel, const int32_t* n_rows,
                                    const int32_t* pos, int cap, const float* sink, const float* inv_freq, int Q,
                                    int S, float* part_ml, float* part_acc, void* out, int32_t* err, cudaStream_t s,
                                    int qps, bool kv_in_ring, bool cluster) {
  DecArgs a{};
  a.cluster = cluster ? 1 : 0;
  a.qps = qps;
  a.kv_in_ring = kv_in_ring ? 1 : 0;
  a.q = static_cast<const __nv_bfloat16*>(q);
  a.pool = static_cast<const __nv_bfloat16*>(pool);
  a.ring = static_cast<__nv_bfloat16*>(ring);
  a.kv_new = static_cast<const __nv_bfloat16*>(kv_new);
  a.sel = sel; a.n_sel = n_sel; a.n_rows = n_rows; a.pos = pos; a.sink = sink; a.inv_freq = inv_freq;
  a.cap = cap; a.topk = L.topk; a.W = L.W; a.Wr = L.Wr; a.ratio = L.ratio; a.S = S;
  a.scale2 = L.scale * 1.4426950408889634f;
  a.part_ml = part_ml; a.part_acc = part_acc;
  a.out = static_cast<__nv_bfloat16*>(out);
  a.err = err;
  cudaFuncSetAttribute(k_tc_attend_decode, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
  if (cluster) {
    if (S != 2 && S != 4) return cudaErrorInvalidValue;
    const cudaError_t e = launch_pdl_cluster(k_tc_attend_decode, dim3(Q * S), dim3(kThreads), kSmem, s, S, a);
    if (e != cudaSuccess) return e;
  } else {
    CSA_LAUNCH(k_tc_attend_decode, dim3(Q * S), dim3(kThreads), kSmem, s, a);
  }
  return cudaGetLastError();
}

}  // namespace csa
