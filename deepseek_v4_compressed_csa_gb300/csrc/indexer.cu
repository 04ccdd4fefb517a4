// Indexer: ReLU-weighted multi-head scores against the index-key pool and an
// exact top-k with lower-row tie-break.
//
// Definition: "feat: add DeepSeek-V4 (Pro/Flash) model support" (mlx-lm #1189),
// stepnoy's patch point 3 and aidiffuser's indexer: queries roped at their
// absolute position, raw head weights with Di^-1/2 * Hi^-1/2 folded in, no
// sigmoid, ReLU on the logits, sum over heads; OmarB97's visibility rule (row j
// visible to p iff (j+1)*ratio <= p+1); the selection keeps index_topk rows.
//
// Launches: rope the index queries -> scores (one block per query and 64-row
// tile) -> radix select per query (one block per query).
#include "common.cuh"
#include "fp8_row.cuh"
#include "kernels.h"

namespace csa {

IndexWs carve_index(Carver& c, const Dims& L, int Q, int cap) {
  IndexWs w;
  w.qr = c.take<float>((size_t)Q * L.Hi * L.Di);
  w.scores = c.take<float>((size_t)Q * cap);
  return w;
}

// Query q's position and sequence.  With device positions (decode, verify blocks) pos0 carries the number of
// consecutive queries per sequence (0 or 1: one; T: a verify block of T tokens): query q belongs to sequence
// q / T at position pos[q / T] + q % T.  With a packed variable-length batch (cu non-null: the row table, pos0 =
// the number of sequences) query q belongs to sequence b = varlen_seq(cu, pos0, q) at pos[b] + q - cu[b].
// Without positions (a prefill chunk of one sequence): sequence 0, pos0 + q.
__device__ __forceinline__ int query_seq(const int32_t* pos, int pos0, const int32_t* cu, int q) {
  if (cu) return varlen_seq(cu, pos0, q);
  return pos ? q / max(1, pos0) : 0;
}
__device__ __forceinline__ int query_pos(const int32_t* pos, int pos0, const int32_t* cu, int q) {
  if (cu) {
    const int b = varlen_seq(cu, pos0, q);
    return pos[b] + q - __ldg(cu + b);
  }
  const int t = max(1, pos0);
  return pos ? pos[q / t] + q % t : pos0 + q;
}

// qr[q][h][:] = RoPE(iq[q][h][:], p_q) rounded to the model dtype, held as fp32.
template <typename T>
__global__ void k_rope_iq(const T* __restrict__ iq, int Hi, int Di, int R, const int32_t* __restrict__ pos, int pos0,
                          const int32_t* __restrict__ cu, const float* __restrict__ inv_freq, float* __restrict__ qr) {
  pdl_trigger();
  pdl_wait();
  const int q = blockIdx.x;
  const int p = query_pos(pos, pos0, cu, q);
  for (int e = threadIdx.x; e < Hi * Di; e += blockDim.x) {
    const int c = e % Di;
    const T* row = iq + ((size_t)q * Hi + e / Di) * Di;
    float v = to_f(row[c]);
    if (c >= Di - R) {
      const int i = (c - (Di - R)) >> 1;
      float cs, sn;
      rope_cs(p, inv_freq, i, &cs, &sn);
      const float a = to_f(row[Di - R + 2 * i]), b = to_f(row[Di - R + 2 * i + 1]);
      v = ((c - (Di - R)) & 1) ? fmaf(a, sn, b * cs) : fmaf(a, cs, -b * sn);
    }
    qr[(size_t)q * Hi * Di + e] = rnd<T>(v);
  }
}

// scores[q][j] for the 64 rows j of tile blockIdx.x.  Thread (hq, kq) owns heads
// 4hq..4hq+3 of the current 64-head group and rows kq + 16*kk (kk < 4).
template <typename T>
__global__ void __launch_bounds__(256) k_index_scores(const float* __restrict__ qr, const T* __restrict__ iw,
                                                      int Hi, int Di, const T* __restrict__ ikeys, int cap,
                                                      const int32_t* __restrict__ n_rows,
                                                      const int32_t* __restrict__ pos, int pos0,
                                                      const int32_t* __restrict__ cu, int ratio, int topk,
                                                      float wscale, float* __restrict__ scores) {
  pdl_trigger();
  pdl_wait();
  extern __shared__ float sm_idx[];
  const int q = blockIdx.y, bseq = query_seq(pos, pos0, cu, q);
  const int p = query_pos(pos, pos0, cu, q);
  const int nvis = min(min(n_rows[bseq], cap), (p + 1) / ratio);
  const int j0 = blockIdx.x * 64;
  if (nvis <= topk || j0 >= nvis) return;
  const int KS = Di + 4;             // padded key row (floats)
  float* ks = sm_idx;                // [64][KS]
  float* qs = ks + 64 * KS;          // [64][Di] one head group
  float* part = qs + 64 * Di;        // [16][64]
  float* wts = part + 16 * 64;       // [64]
  const int tid = threadIdx.x, hq = tid >> 4, kq = tid & 15;
  const T* kbase = ikeys + ((size_t)bseq * cap + j0) * Di;
  const int nk = min(64, nvis - j0);
  for (int e = tid * 8; e < 64 * Di; e += 256 * 8) {
    const int r = e / Di, c = e % Di;
    float v[8];
    if (r < nk) load8_nc(kbase + (size_t)r * Di + c, v);
    else
      for (int i = 0; i < 8; ++i) v[i] = 0.f;
    for (int i = 0; i < 8; ++i) ks[r * KS + c + i] = v[i];
  }
  float tot[4] = {0.f, 0.f, 0.f, 0.f};
  for (int h0 = 0; h0 < Hi; h0 += 64) {
    const int hn = min(64, Hi - h0);
    __syncthreads();
    for (int e = tid; e < 64 * Di; e += 256) {
      const int h = e / Di;
      qs[e] = (h < hn) ? qr[((size_t)q * Hi + h0 + h) * Di + (e % Di)] : 0.f;
    }
    if (tid < 64) wts[tid] = (tid < hn) ? to_f(iw[(size_t)q * Hi + h0 + tid]) * wscale : 0.f;
    __syncthreads();
    float acc[4][4];
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
      for (int k = 0; k < 4; ++k) acc[a][k] = 0.f;
    for (int c = 0; c < Di; c += 4) {
      float4 qv[4], kv[4];
#pragma unroll
      for (int a = 0; a < 4; ++a) qv[a] = *reinterpret_cast<const float4*>(qs + (hq * 4 + a) * Di + c);
#pragma unroll
      for (int k = 0; k < 4; ++k) kv[k] = *reinterpret_cast<const float4*>(ks + (kq + 16 * k) * KS + c);
#pragma unroll
      for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          acc[a][k] = fmaf(qv[a].x, kv[k].x, acc[a][k]);
          acc[a][k] = fmaf(qv[a].y, kv[k].y, acc[a][k]);
          acc[a][k] = fmaf(qv[a].z, kv[k].z, acc[a][k]);
          acc[a][k] = fmaf(qv[a].w, kv[k].w, acc[a][k]);
        }
    }
#pragma unroll
    for (int k = 0; k < 4; ++k)
#pragma unroll
      for (int a = 0; a < 4; ++a) tot[k] = fmaf(wts[hq * 4 + a], fmaxf(acc[a][k], 0.f), tot[k]);
  }
#pragma unroll
  for (int k = 0; k < 4; ++k) part[hq * 64 + kq + 16 * k] = tot[k];
  __syncthreads();
  if (tid < nk) {
    float s = 0.f;
    for (int i = 0; i < 16; ++i) s += part[i * 64 + tid];
    scores[(size_t)q * cap + j0 + tid] = s;
  }
}

// Exclusive prefix count of `flag` over the block (blockDim.x == 1024) plus the block total.
__device__ __forceinline__ int block_excl_count(int flag, int* warp_tot, int* total) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const unsigned bal = __ballot_sync(0xffffffffu, flag);
  const int inwarp = __popc(bal & ((1u << lane) - 1u));
  __syncthreads();
  if (lane == 0) warp_tot[wid] = __popc(bal);
  __syncthreads();
  if (wid == 0) {
    int v = warp_tot[lane];
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int n = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += n;
    }
    warp_tot[lane] = incl - v;
    if (lane == 31) *total = incl;
  }
  __syncthreads();
  return warp_tot[wid] + inwarp;
}

// Exact top-k of scores[q][0 .. nvis) by (score desc, row asc), written in
// ascending row order.  Radix select of the k-th largest order key over four
// 8-bit digits, then one ascending pass that keeps every row above the
// threshold and the lowest-indexed rows equal to it.
__global__ void __launch_bounds__(1024) k_topk(const float* __restrict__ scores, int cap,
                                               const int32_t* __restrict__ n_rows, const int32_t* __restrict__ pos,
                                               int pos0, const int32_t* __restrict__ cu, int ratio, int topk,
                                               int32_t* __restrict__ sel, int32_t* __restrict__ n_sel) {
  pdl_trigger();
  pdl_wait();
  __shared__ int hist[256];
  __shared__ int warp_tot[32];
  __shared__ int s_total;
  __shared__ uint32_t s_prefix;
  __shared__ int s_need;
  const int q = blockIdx.x, bseq = query_seq(pos, pos0, cu, q);
  const int p = query_pos(pos, pos0, cu, q);
  const int nvis = min(min(n_rows[bseq], cap), (p + 1) / ratio);
  int32_t* out = sel + (size_t)q * topk;
  if (nvis <= topk) {
    for (int i = threadIdx.x; i < topk; i += blockDim.x) out[i] = (i < nvis) ? i : -1;
    if (threadIdx.x == 0) n_sel[q] = max(nvis, 0);
    return;
  }
  const float* sc = scores + (size_t)q * cap;
  uint32_t prefix = 0, mask = 0;
  int need = topk;  // rank (1-based, from the top) of the threshold among keys matching prefix
  for (int shift = 24; shift >= 0; shift -= 8) {
    for (int i = threadIdx.x; i < 256; i += blockDim.x) hist[i] = 0;
    __syncthreads();
    for (int j = threadIdx.x; j < nvis; j += blockDim.x) {
      const uint32_t u = ord_key(sc[j]);
      if ((u & mask) == prefix) atomicAdd(&hist[(u >> shift) & 255u], 1);
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      int c = 0, bkt = 0;
      for (bkt = 255; bkt >= 0; --bkt) {
        if (c + hist[bkt] >= need) break;
        c += hist[bkt];
      }
      s_need = need - c;
      s_prefix = prefix | ((uint32_t)bkt << shift);
    }
    __syncthreads();
    need = s_need;
    prefix = s_prefix;
    mask |= 255u << shift;
  }
  // prefix = order key of the k-th largest score; take every key above it and
  // the first `need` keys equal to it (ties to the lower row).
  int eq_base = 0, out_base = 0;
  for (int j0 = 0; j0 < nvis; j0 += blockDim.x) {
    const int j = j0 + threadIdx.x;
    uint32_t u = (j < nvis) ? ord_key(sc[j]) : 0u;
    const int eq = (j < nvis) && (u == prefix);
    const int gt = (j < nvis) && (u > prefix);
    const int eq_rank = eq_base + block_excl_count(eq, warp_tot, &s_total);
    const int eq_tot = s_total;
    const int take = gt || (eq && eq_rank < need);
    const int slot = out_base + block_excl_count(take, warp_tot, &s_total);
    const int take_tot = s_total;
    if (take && slot < topk) out[slot] = j;
    eq_base += eq_tot;
    out_base += take_tot;
  }
  for (int i = out_base + threadIdx.x; i < topk; i += blockDim.x) out[i] = -1;
  if (threadIdx.x == 0) n_sel[q] = min(out_base, topk);
}

// Inclusive prefix sum over the 1024 threads of the block (one value each).
__device__ __forceinline__ int block_incl_scan(int v, int* warp_tot) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += n;
  }
  __syncthreads();
  if (lane == 31) warp_tot[wid] = v;
  __syncthreads();
  if (wid == 0) {
    int t = warp_tot[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(0xffffffffu, t, o);
      if (lane >= o) t += n;
    }
    warp_tot[lane] = t;
  }
  __syncthreads();
  return v + (wid > 0 ? warp_tot[wid - 1] : 0);
}

// One radix-select step over a complete 2048-bin histogram h (the caller's __syncthreads() separates the
// histogram from this call, and a second one separates this call from the use of the result): the bins are taken
// in descending order (thread t owns bins 2047-2t and 2046-2t) and the bin where the running count reaches `need`
// gives *s_prefix = prefix | bin << shift, *s_need = the count still needed inside that bin and *s_count = the
// bin's count.  One block barrier: each warp scans its own 64 bins, then every warp scans the 32 warp totals
// itself.  Requires 1024 threads.
__device__ __forceinline__ void select_bin(const int* h, int need, uint32_t prefix, int shift, int* warp_tot,
                                           uint32_t* s_prefix, int* s_need, int* s_count) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const int b_hi = 2047 - 2 * threadIdx.x, b_lo = b_hi - 1;
  const int c_hi = h[b_hi], c_lo = h[b_lo];
  int v = c_hi + c_lo;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += n;
  }
  if (lane == 31) warp_tot[wid] = v;
  __syncthreads();
  int t = warp_tot[lane];
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(0xffffffffu, t, o);
    if (lane >= o) t += n;
  }
  const int before = __shfl_sync(0xffffffffu, t, (wid + 31) & 31);
  const int incl = v + (wid > 0 ? before : 0);
  const int excl = incl - c_hi - c_lo;
  if (excl < need && need <= incl) {
    if (excl + c_hi >= need) {
      *s_prefix = prefix | ((uint32_t)b_hi << shift);
      *s_need = need - excl;
      *s_count = c_hi;
    } else {
      *s_prefix = prefix | ((uint32_t)b_lo << shift);
      *s_need = need - excl - c_hi;
      *s_count = c_lo;
    }
  }
}

// The same step with every warp taking the decision itself, so that no barrier follows it: after the one barrier
// each warp scans the 32 warp totals, finds the warp whose bins hold the crossing and rescans those 64 bins (read
// from h, which must then stay unchanged until the next block barrier).  Returns the new prefix and need, and
// the selected bin's count.
__device__ __forceinline__ void select_bin_every_warp(const int* h, int& need, uint32_t& prefix, int shift,
                                                      int* warp_tot, int& bin_count) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  int v = h[2047 - 2 * threadIdx.x] + h[2046 - 2 * threadIdx.x];
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += n;
  }
  if (lane == 31) warp_tot[wid] = v;
  __syncthreads();
  int t = warp_tot[lane];
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(0xffffffffu, t, o);
    if (lane >= o) t += n;
  }
  const int cw = __ffs(__ballot_sync(0xffffffffu, t >= need)) - 1;  // the crossing warp (the total is >= need)
  const int base = cw > 0 ? __shfl_sync(0xffffffffu, t, (cw + 31) & 31) : 0;
  const int b_hi = 2047 - 2 * (32 * cw + lane);
  const int c_hi = h[b_hi], c_lo = h[b_hi - 1];
  int u = c_hi + c_lo;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(0xffffffffu, u, o);
    if (lane >= o) u += n;
  }
  const int incl = base + u, excl = incl - c_hi - c_lo;
  const int hl = __ffs(__ballot_sync(0xffffffffu, incl >= need)) - 1;  // the crossing lane
  const bool in_hi = excl + c_hi >= need;
  const int new_need = in_hi ? need - excl : need - excl - c_hi;
  const uint32_t bin = in_hi ? (uint32_t)b_hi : (uint32_t)(b_hi - 1);
  bin_count = __shfl_sync(0xffffffffu, in_hi ? c_hi : c_lo, hl);
  need = __shfl_sync(0xffffffffu, new_need, hl);
  prefix |= __shfl_sync(0xffffffffu, bin, hl) << shift;
}

// Exact top-k with the keys resident in shared memory: radix select of the
// k-th largest order key over digits of 11, 11 and 10 bits (2048-bin
// histograms; the bucket holding the k-th key is found by a block-wide scan
// over the bins in descending order), then one ascending pass that keeps the
// keys above the threshold and the lowest-indexed keys equal to it.
__global__ void __launch_bounds__(1024) k_topk_smem(const float* __restrict__ scores, int cap,
                                                    const int32_t* __restrict__ n_rows,
                                                    const int32_t* __restrict__ pos, int pos0,
                                                    const int32_t* __restrict__ cu, int ratio, int topk,
                                                    int32_t* __restrict__ sel, int32_t* __restrict__ n_sel) {
  pdl_trigger();
  pdl_wait();
  extern __shared__ uint32_t sm_keys[];  // [cap] keys, then hist[2048]
  int* hist = reinterpret_cast<int*>(sm_keys + cap);
  __shared__ int warp_tot[32];
  __shared__ int s_total;
  __shared__ uint32_t s_prefix;
  __shared__ int s_need, s_count;
  const int q = blockIdx.x, bseq = query_seq(pos, pos0, cu, q);
  const int p = query_pos(pos, pos0, cu, q);
  const int nvis = min(min(n_rows[bseq], cap), (p + 1) / ratio);
  int32_t* out = sel + (size_t)q * topk;
  if (nvis <= topk) {
    for (int i = threadIdx.x; i < topk; i += blockDim.x) out[i] = (i < nvis) ? i : -1;
    if (threadIdx.x == 0) n_sel[q] = max(nvis, 0);
    return;
  }
  const float* sc = scores + (size_t)q * cap;
  // the first digit's histogram is counted while the keys are stored
  for (int i = threadIdx.x; i < 2048; i += blockDim.x) hist[i] = 0;
  __syncthreads();
#pragma unroll 4
  for (int j = threadIdx.x; j < nvis; j += blockDim.x) {
    const uint32_t u = ord_key(__ldg(sc + j));
    sm_keys[j] = u;
    atomicAdd(&hist[u >> 21], 1);
  }
  uint32_t prefix = 0, mask = 0;
  int need = topk;
  const int shifts[3] = {21, 10, 0};
  const int widths[3] = {11, 11, 10};
#pragma unroll
  for (int pass = 0; pass < 3; ++pass) {
    const int shift = shifts[pass];
    const uint32_t dmask = (1u << widths[pass]) - 1u;
    if (pass > 0) {
      for (int i = threadIdx.x; i < 2048; i += blockDim.x) hist[i] = 0;
      __syncthreads();
#pragma unroll 4
      for (int j = threadIdx.x; j < nvis; j += blockDim.x) {
        const uint32_t u = sm_keys[j];
        if ((u & mask) == prefix) atomicAdd(&hist[(u >> shift) & dmask], 1);
      }
    }
    __syncthreads();
    select_bin(hist, need, prefix, shift, warp_tot, &s_prefix, &s_need, &s_count);
    __syncthreads();
    prefix = s_prefix;
    need = s_need;
    mask |= dmask << shift;
    // the selected bin holds exactly the keys still needed: every one is kept, the later digits decide nothing
    // (read by every thread after the barrier: the same answer everywhere)
    if (s_count == need) break;
  }
  // Compaction in ascending row order: warp w owns the contiguous keys [w*per, (w+1)*per).  Pass 1 counts
  // each warp's keys above / equal to the threshold, one warp turns the counts into output offsets (the
  // lowest-indexed equal keys are the ones kept), pass 2 writes the rows.
  __shared__ int w_gt[32], w_eq[32], w_out[32], w_eqbase[32];
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const int per = ((nvis + 31) / 32 + 31) & ~31;
  const int lo = wid * per, hi = min(nvis, lo + per);
  int gt_n = 0, eq_n = 0;
#pragma unroll 4
  for (int j0 = lo; j0 < hi; j0 += 32) {
    const int j = j0 + lane;
    const uint32_t u = j < hi ? sm_keys[j] : 0u;
    gt_n += __popc(__ballot_sync(0xffffffffu, j < hi && (u & mask) > prefix));
    eq_n += __popc(__ballot_sync(0xffffffffu, j < hi && (u & mask) == prefix));
  }
  if (lane == 0) {
    w_gt[wid] = gt_n;
    w_eq[wid] = eq_n;
  }
  __syncthreads();
  if (wid == 0) {
    const int e = w_eq[lane];
    int ei = e;  // inclusive prefix of equal keys
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(0xffffffffu, ei, o);
      if (lane >= o) ei += n;
    }
    const int eq_before = ei - e;
    const int eq_taken = max(0, min(e, need - eq_before));
    const int t = w_gt[lane] + eq_taken;
    int ti = t;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(0xffffffffu, ti, o);
      if (lane >= o) ti += n;
    }
    w_out[lane] = ti - t;
    w_eqbase[lane] = eq_before;
    if (lane == 31) s_total = ti;
  }
  __syncthreads();
  int slot = w_out[wid], eq_rank = w_eqbase[wid];
  const unsigned lt = (1u << lane) - 1u;
#pragma unroll 4
  for (int j0 = lo; j0 < hi; j0 += 32) {
    const int j = j0 + lane;
    const uint32_t u = j < hi ? sm_keys[j] : 0u;
    const bool eq = j < hi && (u & mask) == prefix;
    const unsigned eqb = __ballot_sync(0xffffffffu, eq);
    const bool take = (j < hi && (u & mask) > prefix) || (eq && eq_rank + __popc(eqb & lt) < need);
    const unsigned tb = __ballot_sync(0xffffffffu, take);
    if (take) {
      const int o = slot + __popc(tb & lt);
      if (o < topk) out[o] = j;
    }
    slot += __popc(tb);
    eq_rank += __popc(eqb);
  }
  const int total = s_total;
  for (int i2 = total + threadIdx.x; i2 < topk; i2 += blockDim.x) out[i2] = -1;
  if (threadIdx.x == 0) n_sel[q] = min(total, topk);
}

// Exact top-k with every key in registers, for up to kTopkRegKeys x 1024 visible rows: thread t owns the
// contiguous rows [K t, K t + K), K = ceil(n_vis / 1024), so the final pass writes the kept rows in ascending
// order with one block scan.  The threshold is found by the same 11/11/10-bit radix select as k_topk_smem
// (2048-bin shared histograms, one per pass, each cleared during the pass before; two block barriers a pass).
constexpr int kTopkRegKeys = 16;

// Scores of rows jr[0], jr[1] (-1: none) of query q from the roped queries qr [Q,64,128] (bf16) and the scaled
// head weights w [Q,64]: thread t takes head t/16, dims 8 (t%16) .. +7; heads are summed in order by one thread.
// Every thread of the block calls it (two block barriers).
__device__ __forceinline__ void score_rows(const __nv_bfloat16* __restrict__ qr, const float* __restrict__ w,
                                           const __nv_bfloat16* __restrict__ keys, int q, const int (&jr)[2],
                                           float (&part)[2][64], float* out) {
  const int h = threadIdx.x >> 4, sub = threadIdx.x & 15;
  float qv[8];
  load8(qr + ((size_t)q * 64 + h) * 128 + sub * 8, qv);
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    if (jr[r] < 0) continue;
    float kv[8];
    load8(keys + (size_t)jr[r] * 128 + sub * 8, kv);
    float d = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) d = fmaf(qv[i], kv[i], d);
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) d += __shfl_xor_sync(0xffffffffu, d, o);
    if (sub == 0) part[r][h] = d;
  }
  __syncthreads();
  if (threadIdx.x < 2 && jr[threadIdx.x] >= 0) {
    float sc = 0.f;
    for (int hh = 0; hh < 64; ++hh) sc = fmaf(w[(size_t)q * 64 + hh], fmaxf(part[threadIdx.x][hh], 0.f), sc);
    out[threadIdx.x] = sc;
  }
  __syncthreads();
}

// qr / w / keys non-null: the scan before this kernel covered rows < floor(p/ratio) only (it ran while the index
// pool's compress call for this token could still write); the rows that call may have written (row
// floor(p/ratio) and row n_rows-1) are scored here and replace what the score buffer holds for them.
__global__ void __launch_bounds__(1024) k_topk_reg(const float* __restrict__ scores, int cap,
                                                   const int32_t* __restrict__ n_rows, const int32_t* __restrict__ pos,
                                                   int pos0, const int32_t* __restrict__ cu, int ratio, int topk,
                                                   int32_t* __restrict__ sel,
                                                   int32_t* __restrict__ n_sel, const __nv_bfloat16* __restrict__ qr,
                                                   const float* __restrict__ w, const __nv_bfloat16* __restrict__ keys) {
  pdl_trigger();
  __shared__ int hist[3][2048];  // pass n counts into hist[n] and clears the next pass's bins
  __shared__ int warp_tot[32], warp_tot2[32];
  __shared__ float part[2][64];
  __shared__ float new_score[2];
  const int q = blockIdx.x, bseq = query_seq(pos, pos0, cu, q);
  // The position is a step input (no kernel of the step writes it), so the most rows this query can see, and so
  // this thread's rows, are known before the wait: the score loads then go out in the same round as n_rows.
  const int p = query_pos(pos, pos0, cu, q);
  const int nv_max = max(0, min(cap, (p + 1) / ratio));
  const int K = max(1, (nv_max + 1023) >> 10);
  const int r0 = threadIdx.x * K;
  const float* sc = scores + (size_t)q * cap + r0;
  pdl_wait();
  float fk[kTopkRegKeys];
#pragma unroll
  for (int i = 0; i < kTopkRegKeys; ++i) fk[i] = (i < K && r0 + i < nv_max) ? __ldg(sc + i) : 0.f;
  const int nvis = min(min(n_rows[bseq], cap), nv_max);
  int32_t* out = sel + (size_t)q * topk;
  if (nvis <= topk) {
    for (int i = threadIdx.x; i < topk; i += blockDim.x) out[i] = (i < nvis) ? i : -1;
    if (threadIdx.x == 0) n_sel[q] = max(nvis, 0);
    return;
  }
  uint32_t uk[kTopkRegKeys];
#pragma unroll
  for (int i = 0; i < kTopkRegKeys; ++i) uk[i] = (i < K && r0 + i < nvis) ? ord_key(fk[i]) : 0u;
  if (qr) {
    const int j0 = min(cap, p / ratio), jl = min(n_rows[bseq], cap) - 1;
    const int jr[2] = {j0 < nvis ? j0 : -1, (jl >= 0 && jl < nvis && jl != j0) ? jl : -1};
    score_rows(qr, w, keys + (size_t)bseq * cap * 128, q, jr, part, new_score);
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      if (jr[r] < 0) continue;
#pragma unroll
      for (int i = 0; i < kTopkRegKeys; ++i)
        if (i < K && r0 + i == jr[r]) uk[i] = ord_key(new_score[r]);
    }
  }
  hist[0][2 * threadIdx.x] = 0;
  hist[0][2 * threadIdx.x + 1] = 0;
  __syncthreads();
  uint32_t prefix = 0, mask = 0;
  int need = topk;
  const int shifts[3] = {21, 10, 0};
  const int widths[3] = {11, 11, 10};
  // two barriers a pass: the histogram is complete; the warp totals are written (every warp then decides alone,
  // and the bins it rereads are not cleared before the next pass's first barrier)
#pragma unroll
  for (int pass = 0; pass < 3; ++pass) {
    const int shift = shifts[pass];
    const uint32_t dmask = (1u << widths[pass]) - 1u;
    int* h = hist[pass];
#pragma unroll
    for (int i = 0; i < kTopkRegKeys; ++i)
      if (i < K && r0 + i < nvis && (uk[i] & mask) == prefix) atomicAdd(&h[(uk[i] >> shift) & dmask], 1);
    if (pass < 2) {  // the next pass's bins
      hist[pass + 1][2 * threadIdx.x] = 0;
      hist[pass + 1][2 * threadIdx.x + 1] = 0;
    }
    __syncthreads();
    int bin_count;
    select_bin_every_warp(h, need, prefix, shift, warp_tot, bin_count);
    mask |= dmask << shift;
    // the selected bin holds exactly the keys still needed: every one of them is kept, so the later digits
    // decide nothing (the same answer in every warp: all read the same histogram)
    if (bin_count == need) break;
  }
  // prefix = the k-th largest order key on the digits decided (mask): keep every key above it there and the
  // `need` lowest-indexed keys equal to it there, in ascending row order
  // One scan of (keys above << 16 | keys equal) per thread gives both counts before it (each < 2^16): the
  // thread's first output slot is (above before) + min(equal before, need).
  int gt = 0, eq = 0;
#pragma unroll
  for (int i = 0; i < kTopkRegKeys; ++i) {
    const bool v = i < K && r0 + i < nvis;
    gt += (v && (uk[i] & mask) > prefix) ? 1 : 0;
    eq += (v && (uk[i] & mask) == prefix) ? 1 : 0;
  }
  const int packed = (gt << 16) | eq;
  // one block barrier: every warp scans the 32 warp totals itself
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  int incl = packed;
#pragma unroll
  for (int o2 = 1; o2 < 32; o2 <<= 1) {
    const int n = __shfl_up_sync(0xffffffffu, incl, o2);
    if (lane >= o2) incl += n;
  }
  if (lane == 31) warp_tot2[wid] = incl;
  __syncthreads();
  int wt = warp_tot2[lane];
#pragma unroll
  for (int o2 = 1; o2 < 32; o2 <<= 1) {
    const int n = __shfl_up_sync(0xffffffffu, wt, o2);
    if (lane >= o2) wt += n;
  }
  const int before = (wid > 0 ? __shfl_sync(0xffffffffu, wt, (wid + 31) & 31) : 0) + incl - packed;
  const int all = __shfl_sync(0xffffffffu, wt, 31);
  const int eq_before = before & 0xffff;
  int o = (before >> 16) + min(eq_before, need);
  const int total = (all >> 16) + min(all & 0xffff, need);
  int eq_rank = eq_before;
#pragma unroll
  for (int i = 0; i < kTopkRegKeys; ++i) {
    const bool v = i < K && r0 + i < nvis;
    bool keep = v && (uk[i] & mask) > prefix;
    if (v && (uk[i] & mask) == prefix) keep = eq_rank++ < need;
    if (keep) {
      if (o < topk) out[o] = r0 + i;
      ++o;
    }
  }
  for (int i = total + threadIdx.x; i < topk; i += blockDim.x) out[i] = -1;
  if (threadIdx.x == 0) n_sel[q] = min(total, topk);
}

constexpr int kTopkSmemMaxCap = 52 * 1024;

static cudaError_t launch_topk(const Dims& L, const float* scores, int cap, const int32_t* n_rows, const int32_t* pos,
                        int pos0, const int32_t* cu, int Q, int32_t* sel, int32_t* n_sel, cudaStream_t s) {
  if (cap <= kTopkRegKeys * 1024) {
    CSA_LAUNCH(k_topk_reg, dim3(Q), dim3(1024), 0, s, scores, cap, n_rows, pos, pos0, cu, L.ratio, L.topk, sel, n_sel,
               static_cast<const __nv_bfloat16*>(nullptr), static_cast<const float*>(nullptr),
               static_cast<const __nv_bfloat16*>(nullptr));
  } else if (cap <= kTopkSmemMaxCap) {
    const size_t smem = (size_t)cap * 4 + 2048 * 4;
    cudaFuncSetAttribute(k_topk_smem, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    CSA_LAUNCH(k_topk_smem, dim3(Q), dim3(1024), smem, s, scores, cap, n_rows, pos, pos0, cu, L.ratio, L.topk, sel,
               n_sel);
  } else {
    CSA_LAUNCH(k_topk, dim3(Q), dim3(1024), 0, s, scores, cap, n_rows, pos, pos0, cu, L.ratio, L.topk, sel, n_sel);
  }
  return cudaSuccess;
}

template <typename T>
static cudaError_t index_t(const Dims& L, const void* iq, const void* iw, int Q, const void* ikeys, int cap,
                           const int32_t* n_rows, const int32_t* pos, int pos0, const int32_t* cu,
                           const float* inv_freq, int32_t* sel, int32_t* n_sel, const IndexWs& ws, int32_t* err,
                           cudaStream_t s) {
  if (L.ikey_fp8 && !tc_index_supported(L)) return cudaErrorNotSupported;  // fp8 rows: tensor-core scan only
  if (tc_index_supported(L)) {
    // sequences holding the keys: one per query group of a verify block, or the varlen batch's count (pos0)
    const int Bk = cu ? pos0 : (pos ? Q / max(1, pos0) : 1);
    cudaError_t e = launch_tc_index_scores(L, iq, iw, Q, ikeys, Bk, cap, n_rows, pos, pos0, inv_freq, ws.qr,
                                           ws.scores, err, s, false, cu, L.ikey_fp8 != 0);
    if (e != cudaSuccess) return e;
    return launch_topk(L, ws.scores, cap, n_rows, pos, pos0, cu, Q, sel, n_sel, s);
  }
  CSA_LAUNCH(k_rope_iq<T>, dim3(Q), dim3(256), 0, s, static_cast<const T*>(iq), L.Hi, L.Di, L.R, pos, pos0, cu,
             inv_freq, ws.qr);
  const float wscale = (float)(1.0 / sqrt((double)L.Di * (double)L.Hi));
  dim3 g((cap + 63) / 64, Q);
  size_t smem = (64 * (size_t)(L.Di + 4) + 64 * (size_t)L.Di + 16 * 64 + 64) * sizeof(float);
  CSA_LAUNCH(k_index_scores<T>, dim3(g), dim3(256), smem, s, ws.qr, static_cast<const T*>(iw), L.Hi, L.Di, static_cast<const T*>(ikeys),
                                         cap, n_rows, pos, pos0, cu, L.ratio, L.topk, wscale, ws.scores);
  return launch_topk(L, ws.scores, cap, n_rows, pos, pos0, cu, Q, sel, n_sel, s);
}

cudaError_t launch_index_topk_overlapped(const Dims& L, const void* iq, const void* iw, int Q, const void* ikeys,
                                         int cap, const int32_t* n_rows, const int32_t* pos, const float* inv_freq,
                                         int32_t* sel, int32_t* n_sel, const IndexWs& ws, int32_t* err,
                                         cudaStream_t s, cudaEvent_t ready) {
  if (!tc_index_supported(L) || cap > kTopkRegKeys * 1024) {
    if (ready) {
      const cudaError_t e = cudaStreamWaitEvent(s, ready, 0);
      if (e != cudaSuccess) return e;
    }
    return launch_index_topk(L, iq, iw, Q, ikeys, cap, n_rows, pos, 0, inv_freq, sel, n_sel, ws, err, s);
  }
  cudaError_t e = launch_tc_index_scores(L, iq, iw, Q, ikeys, Q, cap, n_rows, pos, 0, inv_freq, ws.qr, ws.scores,
                                         err, s, true);
  if (e != cudaSuccess) return e;
  if (ready) {
    e = cudaStreamWaitEvent(s, ready, 0);
    if (e != cudaSuccess) return e;
  }
  const auto* qr = reinterpret_cast<const __nv_bfloat16*>(ws.qr);
  const auto* w = reinterpret_cast<const float*>(reinterpret_cast<const char*>(ws.qr) + (size_t)Q * 64 * 128 * 2);
  CSA_LAUNCH(k_topk_reg, dim3(Q), dim3(1024), 0, s, ws.scores, cap, n_rows, pos, 0,
             static_cast<const int32_t*>(nullptr), L.ratio, L.topk, sel, n_sel, qr,
             w, static_cast<const __nv_bfloat16*>(ikeys));
  return cudaGetLastError();
}

// Rows of 128 bf16 values -> fp8 index rows (the format the pooling kernels write): one warp per row, lane l
// takes values 4l .. 4l+3.
__global__ void __launch_bounds__(256) k_index_rows_fp8(const __nv_bfloat16* __restrict__ src, long long n,
                                                        uint8_t* __restrict__ dst) {
  pdl_trigger();
  pdl_wait();
  const long long r = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (r >= n) return;  // a whole warp leaves together
  const uint2 raw = __ldg(reinterpret_cast<const uint2*>(src + r * 128 + 4 * lane));
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&raw);
  const float2 v0 = __bfloat1622float2(h[0]), v1 = __bfloat1622float2(h[1]);
  float u[4] = {v0.x, v0.y, v1.x, v1.y};
  float scale;
  const uint32_t packed = fp8_rotate_quantize(u, lane, &scale);
  fp8_row_store(dst + r * kFp8RowBytes, lane, packed, scale);
}

cudaError_t launch_index_rows_fp8(const void* src, long long n, void* dst, cudaStream_t s) {
  const long long blocks = (n + 7) / 8;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
  CSA_LAUNCH(k_index_rows_fp8, dim3((unsigned)blocks), dim3(256), 0, s, static_cast<const __nv_bfloat16*>(src), n,
             static_cast<uint8_t*>(dst));
  return cudaGetLastError();
}

cudaError_t launch_index_topk(const Dims& L, const void* iq, const void* iw, int Q, const void* ikeys, int cap,
                              const int32_t* n_rows, const int32_t* pos, int pos0, const float* inv_freq,
                              int32_t* sel, int32_t* n_sel, const IndexWs& ws, int32_t* err, cudaStream_t s,
                              const int32_t* cu) {
  const int smax = 227 * 1024;
  if (L.dtype == CSA_BF16) {
    cudaFuncSetAttribute(k_index_scores<__nv_bfloat16>, cudaFuncAttributeMaxDynamicSharedMemorySize, smax);
    return index_t<__nv_bfloat16>(L, iq, iw, Q, ikeys, cap, n_rows, pos, pos0, cu, inv_freq, sel, n_sel, ws, err,
                                  s);
  }
  cudaFuncSetAttribute(k_index_scores<float>, cudaFuncAttributeMaxDynamicSharedMemorySize, smax);
  return index_t<float>(L, iq, iw, Q, ikeys, cap, n_rows, pos, pos0, cu, inv_freq, sel, n_sel, ws, err, s);
}

}  // namespace csa
