// Sparse + sliding-window attention on the 5th-generation tensor cores for the
// Flash shapes: 64 query heads over one 512-dim latent (K = V), bf16, RoPE on
// the last 64 dims.
//
// Definitions: "DeepSeek-V4-Flash: native deepseek_v4 AR backend" (MTPLX #216),
// "What V4 adds" (MQA-shaped MLA with per-head sink logits) and "Decode path"
// (bf16 in/out, fp32 softmax state, the probability block cast to bf16 before
// the PV product); "deepseek-v41-mlx" README (inverse rope on the output, sinks
// in the denominator only).
//
// One work item = (query, key split).  Its rows (selected pool rows, then the
// window tokens) are processed in tiles of 128:
//   gather   4 warps copy the tile's 128 rows (1 KB each) with cp.async into a
//            128-byte-swizzled shared tile; the same bytes serve as K (K-major)
//            and as V^T (MN-major), so each row is read from memory once;
//   QK       S^T = K Q^T: M = 128 rows (TMEM lanes), N = 64 heads, K = 512;
//   softmax  each thread owns a row; per-head column max and sum by a warp
//            reduce-scatter; the reference max is raised only when a tile
//            exceeds it by 2^8, in which case O is rescaled in TMEM;
//   PV       O^T += V^T P^T: M = 128 latent dims x 4 tiles, N = 64 heads,
//            K = 128 rows.  P^T goes to shared memory as two bf16 parts,
//            P_hi = bf16(P) and P_lo = bf16(P - P_hi), multiplied in turn, so the
//            product keeps ~16 bits of P instead of bf16's 8.
// The query is roped inside the kernel.  With one split the output is
// finalised in place (sink, normalisation, bf16, inverse RoPE, bf16); with
// several, (m, l, acc) partials go to the workspace for the merge kernel.
#include "common.cuh"
#include "kernels.h"
#include "tc.cuh"

namespace csa {

namespace {

constexpr int kAR = 128;                 // rows per tile
constexpr int kAD = 512;                 // latent dims
constexpr int kAH = 64;                  // heads
constexpr int kBox = kAR * 128;          // one 64-column box of a row tile (16 KB)
constexpr int kRowsBytes = 8 * kBox;     // 128 KB
constexpr int kQBox = kAH * 128;         // 8 KB
constexpr int kQBytes = 8 * kQBox;       // 64 KB
constexpr int kPBytes = kAR * kAH * 2;   // 16 KB
constexpr int kMain = 128;               // gather / softmax / epilogue threads (warps 0-3)
constexpr int kThreadsAt = kMain + 32;   // + warp 4: TMEM owner and MMA issuer
constexpr int kTmemCols = 512;           // S^T: cols 0-63; O^T: cols 64-319
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleAt = 8.f;        // log2 headroom before O is rescaled

// shared-memory layout after the three operand buffers (byte offsets)
constexpr int kOffRed = kRowsBytes + kQBytes + kPBytes;
constexpr int kOffRedSum = kOffRed + 4 * 64 * 4;
constexpr int kOffMref = kOffRedSum + 4 * 64 * 4;
constexpr int kOffLsum = kOffMref + 64 * 4;
constexpr int kOffAlpha = kOffLsum + 64 * 4;
constexpr int kOffRope = kOffAlpha + 64 * 4;    // cos[32], sin[32]
constexpr int kOffRowp = kOffRope + 64 * 4;     // [128] row pointers
constexpr int kOffFlag = kOffRowp + 128 * 8;
constexpr int kOffBars = kOffFlag + 16;         // 6 mbarriers + final
constexpr int kOffTmem = kOffBars + 8 * 8;
constexpr int kSmemAt = kOffTmem + 16 + 1024;   // + alignment slack

struct AtArgs {
  const __nv_bfloat16* q;     // [Q, 64, 512] queries before RoPE
  const __nv_bfloat16* pool;  // [B, cap, 512]
  const __nv_bfloat16* ring;  // [B, W, 512]
  const __nv_bfloat16* kvr;   // [T, 512] roped chunk rows (prefill) or null
  const __nv_bfloat16* kv_new;  // [B, 512] decode: the new token before RoPE (written to the ring here)
  __nv_bfloat16* ring_out;      // decode: the ring, for the new token's slot
  const int32_t* sel;         // [Q, topk] or null
  const int32_t* n_sel;
  const int32_t* n_rows;
  const int32_t* pos;         // decode positions or null (prefill: pos0 + q)
  const float* sink;
  const float* inv_freq;
  int pos0, cap, topk, W, ratio, Q, S;
  int Wr;  // window ring slots (W + rollback); a query attends its last W tokens
  float scale2;               // softmax scale * log2(e)
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

struct Item {
  int q, s, b, p, nsel, nwin, nrows, t_begin, t_end;
};

__device__ __forceinline__ Item make_item(const AtArgs& a, int item) {
  Item it;
  it.q = item / a.S;
  it.s = item % a.S;
  const bool prefill = (a.pos == nullptr);
  it.b = prefill ? 0 : it.q;
  it.p = prefill ? a.pos0 + it.q : a.pos[it.q];
  it.nrows = min(a.n_rows[it.b], a.cap);
  if (a.sel) {
    it.nsel = min(max(a.n_sel[it.q], 0), a.topk);
  } else {
    it.nsel = max(0, min(it.nrows, (it.p + 1) / a.ratio));
  }
  it.nwin = it.p >= 0 ? min(a.W, it.p + 1) : 0;
  const int ntiles = (it.nsel + it.nwin + kAR - 1) / kAR;
  const int tps = (ntiles + a.S - 1) / a.S;
  it.t_begin = min(ntiles, it.s * tps);
  it.t_end = min(ntiles, it.t_begin + tps);
  return it;
}

__global__ void __launch_bounds__(kThreadsAt, 1) k_tc_attend(AtArgs a) {
  pdl_trigger();
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* rows = smem;
  uint8_t* qbuf = smem + kRowsBytes;
  uint8_t* pbuf = qbuf + kQBytes;
  float* red = reinterpret_cast<float*>(smem + kOffRed);
  float* red_sum = reinterpret_cast<float*>(smem + kOffRedSum);
  float* mref = reinterpret_cast<float*>(smem + kOffMref);
  float* lsum = reinterpret_cast<float*>(smem + kOffLsum);
  float* alpha = reinterpret_cast<float*>(smem + kOffAlpha);
  float* rcos = reinterpret_cast<float*>(smem + kOffRope);
  float* rsin = rcos + 32;
  const __nv_bfloat16** rowp = reinterpret_cast<const __nv_bfloat16**>(smem + kOffRowp);
  int* flag = reinterpret_cast<int*>(smem + kOffFlag);
  uint64_t* rows_full = reinterpret_cast<uint64_t*>(smem + kOffBars);
  uint64_t* s_full = rows_full + 1;
  uint64_t* p_full = rows_full + 2;
  uint64_t* pv_done = rows_full + 3;
  uint64_t* drain = rows_full + 4;
  uint64_t* p_used = rows_full + 5;    // first PV product retired: P buffer may take the low part
  uint64_t* plo_full = rows_full + 6;  // low part of P written
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffTmem);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    tc::mbar_init(rows_full, kMain);
    tc::mbar_init(s_full, 1);
    tc::mbar_init(p_full, kMain);
    tc::mbar_init(pv_done, 1);
    tc::mbar_init(drain, 1);
    tc::mbar_init(p_used, 1);
    tc::mbar_init(plo_full, kMain);
    tc::fence_mbar_init();
  }
  pdl_wait();  // predecessor complete: its outputs are visible and its tensor memory is free
  if (warp == 4) {
    tc::tmem_alloc(tmem_slot, kTmemCols);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  const uint32_t tm_s = tmem;        // S^T
  const uint32_t tm_o = tmem + 64;   // O^T, 4 x 64 columns
  bool failed = false;
  uint32_t n_tiles_done = 0;         // tiles processed by this CTA: parity of every barrier

  for (int item = blockIdx.x; item < a.Q * a.S && !failed; item += gridDim.x) {
    if (warp == 4) {
      const Item it = make_item(a, item);
      // ------------------------------------------------------------ MMA issuer
      if (lane == 0) {
        constexpr uint32_t id_qk = tc::idesc_bf16(128, 64);
        constexpr uint32_t id_pv = tc::idesc_bf16(128, 64, true, true);
        const uint32_t r_base = tc::smem_u32(rows), q_base = tc::smem_u32(qbuf), p_base = tc::smem_u32(pbuf);
        for (int t = it.t_begin; t < it.t_end; ++t) {
          const uint32_t par = n_tiles_done & 1;
          if (!tc::mbar_wait(rows_full, par)) { failed = true; break; }
          tc::fence_after_sync();
#pragma unroll 8
          for (int k = 0; k < 32; ++k) {
            const uint64_t ad = tc::sdesc_kmajor_sw128(r_base + (k >> 2) * kBox + (k & 3) * 32);
            const uint64_t bd = tc::sdesc_kmajor_sw128(q_base + (k >> 2) * kQBox + (k & 3) * 32);
            tc::mma_bf16(tm_s, ad, bd, id_qk, k > 0);
          }
          tc::mma_commit(s_full);
          // P = P_hi + P_lo (both bf16): two PV products through the one P buffer
#pragma unroll 1
          for (int part = 0; part < 2; ++part) {
            if (!tc::mbar_wait(part == 0 ? p_full : plo_full, par)) { failed = true; break; }
            tc::fence_after_sync();
#pragma unroll
            for (int m = 0; m < 4; ++m) {
#pragma unroll
              for (int kk = 0; kk < 8; ++kk) {
                const uint64_t ad = tc::sdesc_mnmajor_sw128(r_base + 2 * m * kBox + kk * 2048, kBox, 1024);
                const uint64_t bd = tc::sdesc_mnmajor_sw128(p_base + kk * 2048, 8192, 1024);
                tc::mma_bf16(tm_o + 64 * m, ad, bd, id_pv, (t > it.t_begin) || (kk > 0) || (part > 0));
              }
            }
            tc::mma_commit(part == 0 ? p_used : pv_done);
          }
          if (failed) break;
          ++n_tiles_done;
        }
      }
      __syncwarp();
      n_tiles_done = __shfl_sync(0xffffffffu, n_tiles_done, 0);
      failed = __shfl_sync(0xffffffffu, (int)failed, 0) != 0;
      continue;
    }

    // ------------------------------------------------------------ main warps (128 threads)
    // The query block depends on nothing but the item, so its copy is issued first: 128-byte swizzled
    // K-major rows (one per head) by cp.async, waited for with the first tile's rows, then roped in place.
    const int qi = item / a.S, si = item % a.S;
    {
      const uint32_t q_base = tc::smem_u32(qbuf);
      const __nv_bfloat16* qsrc = a.q + (size_t)qi * kAH * kAD;
#pragma unroll 8
      for (int e = tid; e < kAH * 64; e += kMain) {
        const int h = e >> 6, c = e & 63;
        tc::cp_async16(q_base + (c >> 3) * kQBox + h * 128 + (((c & 7) ^ (h & 7)) << 4), qsrc + (size_t)h * kAD + c * 8,
                       16u);
      }
    }
    // selection of this thread's row of the split's first tile, loaded alongside the item's counters
    // (valid when the split starts at tile si, i.e. one tile per split; reloaded otherwise)
    const int spec_r = si * kAR + tid;
    const int spec_j = (a.sel && spec_r < a.topk) ? a.sel[(size_t)qi * a.topk + spec_r] : 0;
    const Item it = make_item(a, item);
    if (tid < 64) {
      mref[tid] = -INFINITY;
      lsum[tid] = 0.f;
    }
    bool q_pending = true;
    bool table_ready = false;

    for (int t = it.t_begin; t < it.t_end; ++t) {
      const uint32_t par = n_tiles_done & 1;
      const int r0 = t * kAR;
      const int nr = min(kAR, it.nsel + it.nwin - r0);
      // ---- row pointers (row = tid)
      {
        const int r = r0 + tid;
        const __nv_bfloat16* ptr = nullptr;
        if (tid < nr) {
          if (r < it.nsel) {
            const int j = !a.sel ? r : (r == spec_r ? spec_j : a.sel[(size_t)it.q * a.topk + r]);
            if (j >= 0 && j < it.nrows) ptr = a.pool + ((size_t)it.b * a.cap + j) * kAD;
            else atomicOr(a.err, CSA_DEV_RANGE);
          } else {
            const int tok = it.p - it.nwin + 1 + (r - it.nsel);
            if (a.kv_new && tok == it.p) ptr = a.kv_new + (size_t)it.b * kAD;  // roped below, also into the ring
            else
              ptr = (a.kvr && tok >= a.pos0) ? a.kvr + (size_t)(tok - a.pos0) * kAD
                                             : a.ring + ((size_t)it.b * a.Wr + (tok % a.Wr)) * kAD;
          }
        }
        rowp[tid] = ptr;
      }
      tc::named_bar(1, kMain);
      // ---- gather: warp w copies rows 32w .. 32w+31, 2 x 512 contiguous bytes per instruction
      const uint32_t r_base = tc::smem_u32(rows);
      const __nv_bfloat16* cur = (a.kv_new && it.p >= 0) ? a.kv_new + (size_t)it.b * kAD : nullptr;
#pragma unroll 4
      for (int rr = 0; rr < 32; ++rr) {
        const int r = warp * 32 + rr;
        const __nv_bfloat16* src = rowp[r];
        if (cur && src == cur) continue;  // the new token: roped below
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const int c = lane + 32 * hh;
          const uint32_t dst = r_base + (c >> 3) * kBox + r * 128 + (((c & 7) ^ (r & 7)) << 4);
          tc::cp_async16(dst, src ? static_cast<const void*>(src + c * 8) : static_cast<const void*>(a.pool),
                         src ? 16u : 0u);
        }
      }
      // RoPE table of this query's position, computed while the copies are in flight
      if (!table_ready) {
        if (tid < 32) {
          float c, sn;
          rope_cs(it.p, a.inv_freq, tid, &c, &sn);
          rcos[tid] = c;
          rsin[tid] = sn;
        }
        tc::named_bar(1, kMain);
        table_ready = true;
      }
      {
        // the new token (decode): RoPE at p, into the tile and into its ring slot (the slot belongs to the
        // token leaving the window, which no CTA reads)
        const int cur_row = it.nsel + it.nwin - 1 - r0;
        if (cur && cur_row >= 0 && cur_row < nr && rowp[cur_row] == cur && warp == (cur_row >> 5)) {
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            const int c = lane + 32 * hh;
            uint4 raw = __ldg(reinterpret_cast<const uint4*>(cur + c * 8));
            if (c >= 56) {
              __nv_bfloat162* hv = reinterpret_cast<__nv_bfloat162*>(&raw);
#pragma unroll
              for (int k = 0; k < 4; ++k) {
                const int i = (c - 56) * 4 + k;
                const float2 x = __bfloat1622float2(hv[k]);
                hv[k] = __floats2bfloat162_rn(fmaf(x.x, rcos[i], -x.y * rsin[i]), fmaf(x.x, rsin[i], x.y * rcos[i]));
              }
            }
            *reinterpret_cast<uint4*>(rows + (c >> 3) * kBox + cur_row * 128 + (((c & 7) ^ (cur_row & 7)) << 4)) = raw;
            *reinterpret_cast<uint4*>(a.ring_out + ((size_t)it.b * a.Wr + (it.p % a.Wr)) * kAD + c * 8) = raw;
          }
        }
      }
      tc::cp_async_wait_all();
      if (q_pending) {
        tc::named_bar(1, kMain);  // every thread's share of the query block has landed
#pragma unroll
        for (int e = tid; e < kAH * 8; e += kMain) {
          const int h = e >> 3, c = 56 + (e & 7);
          uint4* slot = reinterpret_cast<uint4*>(qbuf + (c >> 3) * kQBox + h * 128 + (((c & 7) ^ (h & 7)) << 4));
          uint4 raw = *slot;
          __nv_bfloat162* hv = reinterpret_cast<__nv_bfloat162*>(&raw);
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const int i = (c - 56) * 4 + k;
            const float2 x = __bfloat1622float2(hv[k]);
            hv[k] = __floats2bfloat162_rn(fmaf(x.x, rcos[i], -x.y * rsin[i]), fmaf(x.x, rsin[i], x.y * rcos[i]));
          }
          *slot = raw;
        }
        q_pending = false;
      }
      tc::fence_proxy_async_smem();
      tc::fence_before_sync();
      tc::mbar_arrive(rows_full);
      // ---- scores of this thread's row
      if (tc::named_bar_any(2, kMain, !tc::mbar_wait(s_full, par))) { failed = true; break; }
      tc::fence_after_sync();
      const int row = tid;
      float sv[64];
      {
        uint32_t u[64];
        const uint32_t ta = tm_s + ((uint32_t)(warp * 32) << 16);
        tc::tmem_ld32(ta, u);
        tc::tmem_ld32(ta + 32, u + 32);
        tc::tmem_wait_ld();
        const bool valid = row < nr && rowp[row] != nullptr;
#pragma unroll
        for (int h = 0; h < 64; ++h) sv[h] = valid ? __uint_as_float(u[h]) * a.scale2 : -INFINITY;
      }
      {
        float cp[64];
#pragma unroll
        for (int h = 0; h < 64; ++h) cp[h] = sv[h];
        const float2 m2 = reduce_scatter64<true>(cp);
        red[warp * 64 + 2 * lane] = m2.x;
        red[warp * 64 + 2 * lane + 1] = m2.y;
      }
      if (tid == 0) *flag = 0;
      tc::named_bar(1, kMain);
      if (tid < 64) {
        const float mt = fmaxf(fmaxf(red[tid], red[64 + tid]), fmaxf(red[128 + tid], red[192 + tid]));
        const float old = mref[tid];
        float nw = old;
        if (old == -INFINITY || mt > old + kRescaleAt) nw = mt;
        float al = 1.f;
        if (old != -INFINITY && nw != old) {
          al = exp2f(old - nw);
          atomicOr(flag, 1);
        }
        alpha[tid] = al;
        mref[tid] = nw;
        lsum[tid] *= al;
      }
      tc::named_bar(1, kMain);
      if (*flag) {
        // raise the reference max: O^T (previous tiles, all retired) *= alpha per head
        for (int m = 0; m < 4; ++m) {
          const uint32_t ta = tm_o + 64 * m + ((uint32_t)(warp * 32) << 16);
          uint32_t u[32];
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            tc::tmem_ld32(ta + 32 * half, u);
            tc::tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i) u[i] = __float_as_uint(__uint_as_float(u[i]) * alpha[32 * half + i]);
            tc::tmem_st32(ta + 32 * half, u);
          }
        }
        tc::tmem_wait_st();
      }
      // ---- probabilities (fp32 for the sums, bf16 for the PV product), P^T as MN-major bf16
      float pe[64];
#pragma unroll
      for (int h = 0; h < 64; ++h) {
        const float ref = mref[h] == -INFINITY ? 0.f : mref[h];
        pe[h] = sv[h] == -INFINITY ? 0.f : exp2f(sv[h] - ref);
      }
      float plo[64];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        uint4 pk;
        __nv_bfloat162* hv = reinterpret_cast<__nv_bfloat162*>(&pk);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          hv[k] = __floats2bfloat162_rn(pe[8 * j + 2 * k], pe[8 * j + 2 * k + 1]);
          const float2 back = __bfloat1622float2(hv[k]);
          plo[8 * j + 2 * k] = pe[8 * j + 2 * k] - back.x;
          plo[8 * j + 2 * k + 1] = pe[8 * j + 2 * k + 1] - back.y;
        }
        *reinterpret_cast<uint4*>(pbuf + (row >> 3) * 1024 + (row & 7) * 128 + ((j ^ (row & 7)) << 4)) = pk;
      }
      tc::fence_proxy_async_smem();
      tc::fence_before_sync();
      tc::mbar_arrive(p_full);
      {
        const float2 s2 = reduce_scatter64<false>(pe);
        red_sum[warp * 64 + 2 * lane] = s2.x;
        red_sum[warp * 64 + 2 * lane + 1] = s2.y;
      }
      // low part once the first PV product has read the buffer
      if (tc::named_bar_any(2, kMain, !tc::mbar_wait(p_used, par))) { failed = true; break; }
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        uint4 pk;
        __nv_bfloat162* hv = reinterpret_cast<__nv_bfloat162*>(&pk);
#pragma unroll
        for (int k = 0; k < 4; ++k) hv[k] = __floats2bfloat162_rn(plo[8 * j + 2 * k], plo[8 * j + 2 * k + 1]);
        *reinterpret_cast<uint4*>(pbuf + (row >> 3) * 1024 + (row & 7) * 128 + ((j ^ (row & 7)) << 4)) = pk;
      }
      tc::fence_proxy_async_smem();
      tc::fence_before_sync();
      tc::mbar_arrive(plo_full);
      tc::named_bar(1, kMain);
      if (tid < 64) lsum[tid] += (red_sum[tid] + red_sum[64 + tid]) + (red_sum[128 + tid] + red_sum[192 + tid]);
      if (tc::named_bar_any(2, kMain, !tc::mbar_wait(pv_done, par))) { failed = true; break; }
      tc::fence_after_sync();
      ++n_tiles_done;
    }
    if (failed) break;
    if (q_pending) tc::cp_async_wait_all();  // an item without rows still owns its query copy
    if (!table_ready && tid < 32) {
      float c, sn;
      rope_cs(it.p, a.inv_freq, tid, &c, &sn);
      rcos[tid] = c;
      rsin[tid] = sn;
    }
    tc::named_bar(1, kMain);
    // ---- epilogue: thread owns latent dim d = 128 m + tid of each O^T tile
    const bool any = it.t_end > it.t_begin;
    if (a.S > 1) {
      if (tid < 64) {
        const size_t idx = ((size_t)it.q * a.S + it.s) * kAH + tid;
        a.part_ml[idx * 2] = mref[tid] == -INFINITY ? -INFINITY : mref[tid] * kLn2;
        a.part_ml[idx * 2 + 1] = lsum[tid];
      }
      if (any) {
        for (int m = 0; m < 4; ++m) {
          const int d = 128 * m + tid;
          uint32_t u[64];
          const uint32_t ta = tm_o + 64 * m + ((uint32_t)(warp * 32) << 16);
          tc::tmem_ld32(ta, u);
          tc::tmem_ld32(ta + 32, u + 32);
          tc::tmem_wait_ld();
          float* dst = a.part_acc + (((size_t)it.q * a.S + it.s) * kAH) * kAD + d;
#pragma unroll
          for (int h = 0; h < 64; ++h) dst[(size_t)h * kAD] = __uint_as_float(u[h]);
        }
      }
    } else {
      for (int m = 0; m < 4; ++m) {
        const int d = 128 * m + tid;
        uint32_t u[64];
        if (any) {
          const uint32_t ta = tm_o + 64 * m + ((uint32_t)(warp * 32) << 16);
          tc::tmem_ld32(ta, u);
          tc::tmem_ld32(ta + 32, u + 32);
          tc::tmem_wait_ld();
        } else {
#pragma unroll
          for (int h = 0; h < 64; ++h) u[h] = 0u;
        }
        __nv_bfloat16* dst = a.out + (size_t)it.q * kAH * kAD + d;
#pragma unroll
        for (int h = 0; h < 64; ++h) {
          const float z2 = a.sink[h] * 1.4426950408889634f;
          const float mr = mref[h];
          const float M2 = fmaxf(z2, mr);
          const float f = mr == -INFINITY ? 0.f : exp2f(mr - M2);
          const float Z = exp2f(z2 - M2) + lsum[h] * f;
          float o = rnd<__nv_bfloat16>(__uint_as_float(u[h]) * (f / Z));
          const float partner = __shfl_xor_sync(0xffffffffu, o, 1);
          if (d >= kAD - 64) {
            const int i = (d - (kAD - 64)) >> 1;
            o = (d & 1) ? fmaf(-partner, rsin[i], o * rcos[i]) : fmaf(o, rcos[i], partner * rsin[i]);
          }
          dst[(size_t)h * kAD] = __float2bfloat16_rn(o);
        }
      }
    }
    tc::fence_before_sync();
    tc::named_bar(1, kMain);
  }
  if (failed) atomicOr(a.err, tc::kErrTimeout);
  // retire every MMA before tensor memory is released
  if (warp == 4 && lane == 0) {
    tc::mma_commit(drain);
    if (!tc::mbar_wait(drain, 0)) atomicOr(a.err, tc::kErrTimeout);
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 4) tc::tmem_dealloc(tmem, kTmemCols);
}

// Merge of S split partials for 8 heads of one query: warp w owns head 8*blockIdx.x + w, lane owns latent
// dims 16*lane .. 16*lane+15.  M = max(z, m_s); Z = e^{z-M} + sum_s l_s e^{m_s-M}; o = sum_s acc_s e^{m_s-M} / Z;
// bf16; inverse RoPE on the last 64 dims; bf16.  The first four splits' accumulators are requested together with
// the split statistics (one memory round trip for S <= 4); a split that holds no rows (m = -inf) has weight 0 and
// its accumulator, which it did not write, is not used.
__global__ void __launch_bounds__(256) k_tc_merge(const float* __restrict__ part_ml, const float* __restrict__ part_acc,
                                                  int S, const float* __restrict__ sink, const int32_t* __restrict__ pos,
                                                  int qps, const float* __restrict__ inv_freq,
                                                  __nv_bfloat16* __restrict__ out) {
  pdl_trigger();
  __shared__ float rc[32], rs[32];
  const int q = blockIdx.y, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = blockIdx.x * 8 + warp;
  const size_t base = (size_t)q * S * kAH + h;
  // before the wait: the sink and the RoPE table of the query's position (call inputs)
  const float z = sink[h];
  if (threadIdx.x < 32) rope_cs(pos[q / qps] + q % qps, inv_freq, threadIdx.x, &rc[threadIdx.x], &rs[threadIdx.x]);
  pdl_wait();
  float4 x[4][4];
  auto load_batch = [&](int s0) {
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      if (s0 + k < S) {
        const float4* pa = reinterpret_cast<const float4*>(part_acc + (base + (size_t)(s0 + k) * kAH) * kAD + lane * 16);
#pragma unroll
        for (int c = 0; c < 4; ++c) x[k][c] = __ldcg(pa + c);
      }
    }
  };
  load_batch(0);
  // split statistics: lane s holds split s (S <= 32)
  const float m_l = lane < S ? __ldcg(part_ml + (base + (size_t)lane * kAH) * 2) : -INFINITY;
  const float l_l = lane < S ? __ldcg(part_ml + (base + (size_t)lane * kAH) * 2 + 1) : 0.f;
  const float M = fmaxf(z, warp_max(m_l));
  const float f_l = m_l == -INFINITY ? 0.f : expf(m_l - M);
  const float Z = expf(z - M) + warp_sum(l_l * f_l);
  float v[16];
#pragma unroll
  for (int e = 0; e < 16; ++e) v[e] = 0.f;
  for (int s0 = 0; s0 < S; s0 += 4) {
    if (s0 > 0) load_batch(s0);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float f = __shfl_sync(0xffffffffu, f_l, (s0 + k) & 31);
      if (s0 + k < S && f != 0.f) {
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          v[4 * c] = fmaf(x[k][c].x, f, v[4 * c]);
          v[4 * c + 1] = fmaf(x[k][c].y, f, v[4 * c + 1]);
          v[4 * c + 2] = fmaf(x[k][c].z, f, v[4 * c + 2]);
          v[4 * c + 3] = fmaf(x[k][c].w, f, v[4 * c + 3]);
        }
      }
    }
  }
  __syncthreads();
  const float invZ = 1.0f / Z;
#pragma unroll
  for (int e = 0; e < 16; ++e) v[e] = rnd<__nv_bfloat16>(v[e] * invZ);
  const int d0 = lane * 16;
  if (d0 >= kAD - 64) {
#pragma unroll
    for (int e = 0; e < 16; e += 2) {
      const int i = (d0 + e - (kAD - 64)) >> 1;
      const float x0 = v[e], x1 = v[e + 1];
      v[e] = fmaf(x0, rc[i], x1 * rs[i]);
      v[e + 1] = fmaf(-x0, rs[i], x1 * rc[i]);
    }
  }
  uint4 pk[2];
  __nv_bfloat162* hv = reinterpret_cast<__nv_bfloat162*>(pk);
#pragma unroll
  for (int k = 0; k < 8; ++k) hv[k] = __floats2bfloat162_rn(v[2 * k], v[2 * k + 1]);
  uint4* dst = reinterpret_cast<uint4*>(out + ((size_t)q * kAH + h) * kAD + d0);
  dst[0] = pk[0];
  dst[1] = pk[1];
}

int g_sms_at = 0;

}  // namespace

bool tc_attend_supported(const Dims& L) { return L.dtype == CSA_BF16 && L.H == 64 && L.D == 512 && L.R == 64; }

cudaError_t launch_tc_attend(const Dims& L, const void* q, const void* pool, void* ring, const void* kvr,
                             const void* kv_new, const int32_t* sel, const int32_t* n_sel, const int32_t* n_rows,
                             const int32_t* pos, int pos0, int cap, const float* sink, const float* inv_freq, int Q,
                             int S, float* part_ml, float* part_acc, void* out, int32_t* err, cudaStream_t s) {
  if (!g_sms_at) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&g_sms_at, cudaDevAttrMultiProcessorCount, dev);
  }
  AtArgs a{};
  a.q = static_cast<const __nv_bfloat16*>(q);
  a.pool = static_cast<const __nv_bfloat16*>(pool);
  a.ring = static_cast<const __nv_bfloat16*>(ring);
  a.kvr = static_cast<const __nv_bfloat16*>(kvr);
  a.kv_new = static_cast<const __nv_bfloat16*>(kv_new);
  a.ring_out = static_cast<__nv_bfloat16*>(ring);
  a.sel = sel; a.n_sel = n_sel; a.n_rows = n_rows; a.pos = pos; a.sink = sink; a.inv_freq = inv_freq;
  a.pos0 = pos0; a.cap = cap; a.topk = L.topk; a.W = L.W; a.Wr = L.Wr; a.ratio = L.ratio; a.Q = Q; a.S = S;
  a.scale2 = L.scale * 1.4426950408889634f;
  a.part_ml = part_ml; a.part_acc = part_acc;
  a.out = static_cast<__nv_bfloat16*>(out);
  a.err = err;
  const int items = Q * S;
  const int grid = pos ? items : min(items, g_sms_at);
  cudaFuncSetAttribute(k_tc_attend, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemAt);
  CSA_LAUNCH(k_tc_attend, dim3(grid), dim3(kThreadsAt), kSmemAt, s, a);
  return cudaGetLastError();
}

cudaError_t launch_tc_merge(const Dims& L, const float* part_ml, const float* part_acc, int S, int Q,
                            const float* sink, const int32_t* pos, const float* inv_freq, void* out, cudaStream_t s,
                            int qps) {
  (void)L;
  if (S > 32) return cudaErrorNotSupported;  // callers use the generic merge beyond 32 splits
  CSA_LAUNCH(k_tc_merge, dim3(dim3(kAH / 8, Q)), dim3(256), 0, s, part_ml, part_acc, S, sink, pos, qps, inv_freq,
                                               static_cast<__nv_bfloat16*>(out));
  return cudaGetLastError();
}

}  // namespace csa
