// Attention of H heads over one shared latent (K = V): selected compressed rows
// plus the sliding window, per-head sink logits, split-K partial softmax and
// merge, inverse RoPE on the output.
//
// Definitions: "DeepSeek-V4-Flash: native deepseek_v4 AR backend" (MTPLX #216),
// "What V4 adds" (MQA-shaped MLA: 64 query heads over one 512-dim latent with
// per-head sink logits; 128-token sliding window) and "Decode path" (bf16
// in/out, fp32 accumulation); "deepseek-v41-mlx" README (the rope inverse on the
// attention output; sinks in the softmax denominator only); "feat: add
// DeepSeek-V4 (Pro/Flash) model support" (mlx-lm #1189), stepnoy: decode
// gathers its own top-k rows, prefill applies a per-query top-k AND-ed with
// the visibility mask.
//
// Portable SIMT path (any model dtype, D <= 1024): one block per (query,
// group of 8 heads, key split); one warp per head, rows streamed through
// shared memory in chunks of 64 with an online softmax; partials (m, l, acc)
// are merged by a second kernel, or finalised in place when there is a single
// split.
#include "common.cuh"
#include "kernels.h"

namespace csa {

static constexpr int kHG = 8;     // heads per block (one warp each)
static constexpr int kCH = 64;    // rows per shared-memory chunk
static constexpr int kSplitRows = 128;
static constexpr int kMaxC = 4;   // 8-element chunks per lane: D <= 32 * 8 * kMaxC = 1024

int attend_splits(const Dims& L, bool prefill, bool all_rows, int cap) {
  if (prefill) return 1;
  const int maxrows = (all_rows ? cap : L.topk) + L.W;
  return max(1, (maxrows + kSplitRows - 1) / kSplitRows);
}

AttendWs carve_attend(Carver& c, const Dims& L, int Q, int S, int T) {
  AttendWs w;
  w.S = S;
  w.qr = c.take<char>((size_t)Q * L.H * L.D * esize(L.dtype));
  w.kvr = T > 0 ? c.take<char>((size_t)T * L.D * esize(L.dtype)) : nullptr;
  if (S > 1) {
    w.part_ml = c.take<float>((size_t)Q * S * L.H * 2);
    w.part_acc = c.take<float>((size_t)Q * S * L.H * L.D);
  } else {
    w.part_ml = nullptr;
    w.part_acc = nullptr;
  }
  return w;
}

// dst[r][:] = RoPE(src[r][:], p(r)) in the model dtype; rows of one query are
// `rows_per_q` consecutive rows; p = pos ? pos[q] : pos0 + q.
template <typename T>
__global__ void k_rope_rows(const T* __restrict__ src, T* __restrict__ dst, int rows_per_q, int D, int R,
                            const int32_t* __restrict__ pos, int pos0, const float* __restrict__ inv_freq) {
  pdl_trigger();
  pdl_wait();
  const int q = blockIdx.x;
  const int p = pos ? pos[q] : pos0 + q;
  const size_t base = (size_t)q * rows_per_q * D;
  for (int e = threadIdx.x; e < rows_per_q * D; e += blockDim.x) {
    const int c = e % D;
    const T* row = src + base + (size_t)(e / D) * D;
    float v = to_f(row[c]);
    if (c >= D - R) {
      const int i = (c - (D - R)) >> 1;
      float cs, sn;
      rope_cs(p, inv_freq, i, &cs, &sn);
      const float a = to_f(row[D - R + 2 * i]), b = to_f(row[D - R + 2 * i + 1]);
      v = ((c - (D - R)) & 1) ? fmaf(a, sn, b * cs) : fmaf(a, cs, -b * sn);
    }
    dst[base + e] = from_f<T>(v);
  }
}

// window[b][pos[b] mod Wr] = RoPE(kv_new[b], pos[b])  (Wr: ring slots)
template <typename T>
__global__ void k_window_append(const T* __restrict__ kv, T* __restrict__ window, int W, int D, int R,
                                const int32_t* __restrict__ pos, const float* __restrict__ inv_freq) {
  pdl_trigger();
  pdl_wait();
  const int b = blockIdx.x;
  const int p = pos[b];
  if (p < 0) return;
  const T* row = kv + (size_t)b * D;
  T* dst = window + ((size_t)b * W + (p % W)) * D;
  for (int c = threadIdx.x; c < D; c += blockDim.x) {
    float v = to_f(row[c]);
    if (c >= D - R) {
      const int i = (c - (D - R)) >> 1;
      float cs, sn;
      rope_cs(p, inv_freq, i, &cs, &sn);
      const float a = to_f(row[D - R + 2 * i]), bb = to_f(row[D - R + 2 * i + 1]);
      v = ((c - (D - R)) & 1) ? fmaf(a, sn, bb * cs) : fmaf(a, cs, -bb * sn);
    }
    dst[c] = from_f<T>(v);
  }
}

// window[t mod Wr] = kvr[t - pos0] for the chunk's last min(T, Wr) tokens (Wr: ring slots, W + rollback)
template <typename T>
__global__ void k_window_store_chunk(const T* __restrict__ kvr, T* __restrict__ window, int W, int D, int T_,
                                     int pos0) {
  pdl_trigger();
  pdl_wait();
  const int keep = min(T_, W);
  const int t = pos0 + T_ - keep + blockIdx.x;
  for (int e = threadIdx.x * 8; e < D; e += blockDim.x * 8)
    copy8<T>(window + (size_t)(t % W) * D + e, kvr + (size_t)(t - pos0) * D + e);
}

// Packed variable-length chunks (row table cu [nseq + 1]): kvr[r] = RoPE(kv[r], pos[b] + r - cu[b]) for row r of
// sequence b.
template <typename T>
__global__ void k_rope_rows_varlen(const T* __restrict__ kv, T* __restrict__ kvr, int D, int R,
                                   const int32_t* __restrict__ pos, const int32_t* __restrict__ cu, int nseq,
                                   const float* __restrict__ inv_freq) {
  pdl_trigger();
  pdl_wait();
  const int r = blockIdx.x, b = varlen_seq(cu, nseq, r);
  const int p = pos[b] + r - __ldg(cu + b);
  const T* row = kv + (size_t)r * D;
  for (int c = threadIdx.x; c < D; c += blockDim.x) {
    float v = to_f(row[c]);
    if (c >= D - R) {
      const int i = (c - (D - R)) >> 1;
      float cs, sn;
      rope_cs(p, inv_freq, i, &cs, &sn);
      const float a = to_f(row[D - R + 2 * i]), bb = to_f(row[D - R + 2 * i + 1]);
      v = ((c - (D - R)) & 1) ? fmaf(a, sn, bb * cs) : fmaf(a, cs, -bb * sn);
    }
    kvr[(size_t)r * D + c] = from_f<T>(v);
  }
}

// Each sequence's last min(T_b, Wr) chunk tokens into its ring: window[b][(pos[b] + i) mod Wr] = kvr[cu[b] + i].
// A sequence whose row-table entries are inconsistent is left alone (the compress call reports the table).
template <typename T>
__global__ void k_window_store_varlen(const T* __restrict__ kvr, T* __restrict__ window, int Wr, int D, int N,
                                      const int32_t* __restrict__ pos, const int32_t* __restrict__ cu) {
  pdl_trigger();
  pdl_wait();
  const int b = blockIdx.y, c0 = cu[b], c1 = cu[b + 1];
  if (c0 < 0 || c1 > N || c1 < c0) return;
  const int Tb = c1 - c0, keep = min(Tb, Wr);
  if ((int)blockIdx.x >= keep) return;
  const int i = Tb - keep + blockIdx.x, t = pos[b] + i;
  if (t < 0) return;
  for (int e = threadIdx.x * 8; e < D; e += blockDim.x * 8)
    copy8<T>(window + ((size_t)b * Wr + t % Wr) * D + e, kvr + (size_t)(c0 + i) * D + e);
}

struct AttnArgs {
  const void* qr;       // [Q, H, D] roped queries
  const void* pool;     // [B, cap, D]
  const void* ring;     // [B, W, D]
  const void* kvr;      // [T, D] roped chunk rows (prefill) or null
  const int32_t* sel;   // [Q, topk] or null (all visible rows)
  const int32_t* n_sel; // [Q]
  const int32_t* n_rows;
  const int32_t* pos;   // decode positions [B] or null (prefill: pos0 + q)
  const float* sink;
  const float* inv_freq;
  int pos0, cap, topk, W, Wr, H, D, R, ratio;  // W attended window tokens, Wr ring slots
  float scale;
  int S;
  float* part_ml;
  float* part_acc;
  void* out;
  int32_t* err;
};

template <typename T>
__global__ void __launch_bounds__(256) k_attend_simt(AttnArgs a) {
  pdl_trigger();
  pdl_wait();
  extern __shared__ __align__(16) unsigned char sm_attn[];
  const int D = a.D, KS = D + 8;
  T* qs = reinterpret_cast<T*>(sm_attn);                 // [kHG][D]
  T* ks = qs + kHG * D;                                  // [kCH][KS]
  float* ps = reinterpret_cast<float*>(ks + kCH * KS);   // [kHG][kCH]
  const T** rowp = reinterpret_cast<const T**>(ps + kHG * kCH);  // [kCH]
  const int q = blockIdx.z, s = blockIdx.y, hg = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = hg * kHG + warp;
  const bool prefill = (a.pos == nullptr);
  const int b = prefill ? 0 : q;
  const int p = prefill ? a.pos0 + q : a.pos[q];
  const T* pool = static_cast<const T*>(a.pool) + (size_t)b * a.cap * D;
  const T* ring = static_cast<const T*>(a.ring) + (size_t)b * a.Wr * D;
  const T* kvr = static_cast<const T*>(a.kvr);
  const int nrows_b = min(a.n_rows[b], a.cap);

  int nsel;
  if (a.sel) {
    nsel = a.n_sel[q];
    if (nsel > a.topk || nsel < 0) {
      if (threadIdx.x == 0 && s == 0 && hg == 0) atomicOr(a.err, CSA_DEV_RANGE);
      nsel = min(max(nsel, 0), a.topk);
    }
  } else {
    nsel = max(0, min(nrows_b, (p + 1) / a.ratio));
  }
  const int nwin = (p >= 0) ? min(a.W, p + 1) : 0;
  const int total = nsel + nwin;
  const int per = (total + a.S - 1) / a.S;
  const int r_begin = s * per, r_end = min(total, r_begin + per);

  for (int e = threadIdx.x * 8; e < kHG * D; e += blockDim.x * 8) {
    const int hh = hg * kHG + e / D;
    if (hh < a.H) copy8<T>(qs + e, static_cast<const T*>(a.qr) + ((size_t)q * a.H + hh) * D + (e % D));
    else zero8<T>(qs + e);
  }

  float m_run = -INFINITY, l_run = 0.f;
  float acc[kMaxC][8];
#pragma unroll
  for (int c = 0; c < kMaxC; ++c)
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[c][e] = 0.f;
  const int nch8 = D / 8;

  for (int c0 = r_begin; c0 < r_end; c0 += kCH) {
    const int nr = min(kCH, r_end - c0);
    __syncthreads();
    if (threadIdx.x < kCH) {
      const int r = c0 + threadIdx.x;
      const T* ptr = nullptr;
      if (threadIdx.x < nr) {
        if (r < nsel) {
          const int j = a.sel ? a.sel[(size_t)q * a.topk + r] : r;
          if (j >= 0 && j < nrows_b) ptr = pool + (size_t)j * D;
          else if (hg == 0) atomicOr(a.err, CSA_DEV_RANGE);
        } else {
          const int t = p - nwin + 1 + (r - nsel);
          ptr = (prefill && t >= a.pos0) ? kvr + (size_t)(t - a.pos0) * D : ring + (size_t)(t % a.Wr) * D;
        }
      }
      rowp[threadIdx.x] = ptr;
    }
    __syncthreads();
    for (int e = threadIdx.x; e < kCH * nch8; e += blockDim.x) {
      const int r = e / nch8, c = (e % nch8) * 8;
      const T* src = rowp[r];
      if (src) copy8<T>(ks + r * KS + c, src + c);
      else zero8<T>(ks + r * KS + c);
    }
    __syncthreads();
    // logits of this warp's head for rows lane and lane + 32
    float lg[2];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int r = lane + 32 * u;
      float dot = 0.f;
      if (r < nr) {
        const T* kr = ks + r * KS;
        const T* qh = qs + warp * D;
        for (int c = 0; c < D; c += 8) {
          float kv8[8], q8[8];
          load8(kr + c, kv8);
          load8(qh + c, q8);
#pragma unroll
          for (int e = 0; e < 8; ++e) dot = fmaf(q8[e], kv8[e], dot);
        }
      }
      lg[u] = (r < nr && rowp[r] != nullptr) ? dot * a.scale : -INFINITY;
    }
    const float cmax = warp_max(fmaxf(lg[0], lg[1]));
    const float m_new = fmaxf(m_run, cmax);
    float pe[2];
    float alpha = 1.f;
    if (m_new == -INFINITY) {
      pe[0] = pe[1] = 0.f;
    } else {
      alpha = expf(m_run - m_new);
      pe[0] = expf(lg[0] - m_new);
      pe[1] = expf(lg[1] - m_new);
    }
    ps[warp * kCH + lane] = pe[0];
    ps[warp * kCH + lane + 32] = pe[1];
    l_run = l_run * alpha + warp_sum(pe[0] + pe[1]);
    m_run = m_new;
    __syncwarp();
#pragma unroll
    for (int c = 0; c < kMaxC; ++c)
#pragma unroll
      for (int e = 0; e < 8; ++e) acc[c][e] *= alpha;
    for (int r = 0; r < nr; ++r) {
      const float pr = ps[warp * kCH + r];
      const T* kr = ks + r * KS;
#pragma unroll
      for (int c = 0; c < kMaxC; ++c) {
        const int ci = lane + 32 * c;
        if (ci < nch8) {
          float v[8];
          load8(kr + ci * 8, v);
#pragma unroll
          for (int e = 0; e < 8; ++e) acc[c][e] = fmaf(pr, v[e], acc[c][e]);
        }
      }
    }
  }
  if (h >= a.H) return;
  if (a.S == 1) {
    // finalise: sink in the denominator only, model dtype, inverse RoPE, model dtype
    const float z = a.sink[h];
    const float M = fmaxf(z, m_run);
    const float f = (m_run == -INFINITY) ? 0.f : expf(m_run - M);
    const float Z = expf(z - M) + l_run * f;
    const float g = f / Z;
    T* o = static_cast<T*>(a.out) + ((size_t)q * a.H + h) * D;
#pragma unroll
    for (int c = 0; c < kMaxC; ++c) {
      const int ci = lane + 32 * c;
      if (ci < nch8) {
        float v[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) v[e] = rnd<T>(acc[c][e] * g);
        const int d0 = ci * 8;
#pragma unroll
        for (int e = 0; e < 8; e += 2) {
          const int dd = d0 + e;
          if (dd >= D - a.R) {
            float cs, sn;
            rope_cs(p, a.inv_freq, (dd - (D - a.R)) >> 1, &cs, &sn);
            const float x0 = v[e], x1 = v[e + 1];
            v[e] = fmaf(x0, cs, x1 * sn);
            v[e + 1] = fmaf(-x0, sn, x1 * cs);
          }
        }
#pragma unroll
        for (int e = 0; e < 8; ++e) o[d0 + e] = from_f<T>(v[e]);
      }
    }
  } else {
    const size_t idx = ((size_t)q * a.S + s) * a.H + h;
    if (lane == 0) {
      a.part_ml[idx * 2] = m_run;
      a.part_ml[idx * 2 + 1] = l_run;
    }
    float* pa = a.part_acc + idx * D;
#pragma unroll
    for (int c = 0; c < kMaxC; ++c) {
      const int ci = lane + 32 * c;
      if (ci < nch8) {
        reinterpret_cast<float4*>(pa + ci * 8)[0] = make_float4(acc[c][0], acc[c][1], acc[c][2], acc[c][3]);
        reinterpret_cast<float4*>(pa + ci * 8)[1] = make_float4(acc[c][4], acc[c][5], acc[c][6], acc[c][7]);
      }
    }
  }
}

// out[q][h] = merge of the S partials with the sink, model dtype, inverse RoPE, model dtype.
// One block per (head, query); thread i owns dims 8i .. 8i+7.
template <typename T>
__global__ void k_attend_merge(const float* __restrict__ part_ml, const float* __restrict__ part_acc, int S, int H,
                               int D, int R, const float* __restrict__ sink, const int32_t* __restrict__ pos,
                               int pos0, const float* __restrict__ inv_freq, T* __restrict__ out) {
  pdl_trigger();
  pdl_wait();
  extern __shared__ float sm_merge[];  // [S] scale factors
  const int h = blockIdx.x, q = blockIdx.y;
  const int p = pos ? pos[q] : pos0 + q;
  const float z = sink[h];
  float M = z;
  for (int s = 0; s < S; ++s) M = fmaxf(M, part_ml[(((size_t)q * S + s) * H + h) * 2]);
  float Z = expf(z - M);
  for (int s = 0; s < S; ++s) {
    const size_t idx = ((size_t)q * S + s) * H + h;
    const float m = part_ml[idx * 2];
    const float f = (m == -INFINITY) ? 0.f : expf(m - M);
    Z += part_ml[idx * 2 + 1] * f;
    if (threadIdx.x == 0) sm_merge[s] = f;
  }
  __syncthreads();
  const float invZ = 1.0f / Z;
  for (int d0 = threadIdx.x * 8; d0 < D; d0 += blockDim.x * 8) {
    float v[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    for (int s = 0; s < S; ++s) {
      const float f = sm_merge[s];
      if (f == 0.f) continue;
      const float* pa = part_acc + (((size_t)q * S + s) * H + h) * D + d0;
#pragma unroll
      for (int e = 0; e < 8; ++e) v[e] = fmaf(pa[e], f, v[e]);
    }
#pragma unroll
    for (int e = 0; e < 8; ++e) v[e] = rnd<T>(v[e] * invZ);
#pragma unroll
    for (int e = 0; e < 8; e += 2) {
      const int dd = d0 + e;
      if (dd >= D - R) {
        float cs, sn;
        rope_cs(p, inv_freq, (dd - (D - R)) >> 1, &cs, &sn);
        const float x0 = v[e], x1 = v[e + 1];
        v[e] = fmaf(x0, cs, x1 * sn);
        v[e + 1] = fmaf(-x0, sn, x1 * cs);
      }
    }
    T* o = out + ((size_t)q * H + h) * D + d0;
#pragma unroll
    for (int e = 0; e < 8; ++e) o[e] = from_f<T>(v[e]);
  }
}

template <typename T>
static size_t attend_smem(int D) {
  return (size_t)kHG * D * sizeof(T) + (size_t)kCH * (D + 8) * sizeof(T) + (size_t)kHG * kCH * sizeof(float) +
         (size_t)kCH * sizeof(void*);
}

template <typename T>
static cudaError_t run_attend(AttnArgs& a, int Q, cudaStream_t s) {
  const size_t smem = attend_smem<T>(a.D);
  cudaFuncSetAttribute(k_attend_simt<T>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  dim3 g((a.H + kHG - 1) / kHG, a.S, Q);
  CSA_LAUNCH(k_attend_simt<T>, dim3(g), dim3(256), smem, s, a);
  if (a.S > 1) {
    dim3 gm(a.H, Q);
    const int thr = max(32, min(1024, a.D / 8));
    CSA_LAUNCH(k_attend_merge<T>, dim3(gm), dim3(thr), a.S * sizeof(float), s, a.part_ml, a.part_acc, a.S, a.H, a.D, a.R, a.sink,
                                                           a.pos, a.pos0, a.inv_freq, static_cast<T*>(a.out));
  }
  return cudaGetLastError();
}

template <typename T>
static cudaError_t decode_t(const Dims& L, const void* q, const void* kv_new, const float* sink, int B, void* window,
                            const void* pool, int cap, const int32_t* n_rows, const int32_t* sel,
                            const int32_t* n_sel, const int32_t* pos, const float* inv_freq, void* out,
                            const AttendWs& ws, int32_t* err, cudaStream_t s) {
  // the workspace holds ws.S partials per query; the one-chunk decode kernel needs splits of <= 160 rows, which
  // it always has except for a layer with an indexer called without a selection (every visible row)
  const int S = tc_attend_decode_supported(L) ? tc_attend_decode_splits(B, L.W, sel ? L.topk : cap, ws.S) : 0;
  if (S > 0) {
    const bool cluster = tc_attend_decode_cluster(S);
    cudaError_t e = launch_tc_attend_decode(L, q, pool, window, kv_new, sel, n_sel, n_rows, pos, cap, sink, inv_freq,
                                            B, S, ws.part_ml, ws.part_acc, out, err, s, 1, false, cluster);
    if (e != cudaSuccess || S == 1 || cluster) return e;
    if (S <= 32) return launch_tc_merge(L, ws.part_ml, ws.part_acc, S, B, sink, pos, inv_freq, out, s);
    CSA_LAUNCH(k_attend_merge<T>, dim3(L.H, B), dim3(max(32, min(1024, L.D / 8))), S * sizeof(float), s,
               ws.part_ml, ws.part_acc, S, L.H, L.D, L.R, sink, pos, 0, inv_freq, static_cast<T*>(out));
    return cudaGetLastError();
  }
  if (tc_attend_supported(L)) {
    cudaError_t e = launch_tc_attend(L, q, pool, window, nullptr, kv_new, sel, n_sel, n_rows, pos, 0, cap, sink,
                                     inv_freq, B, ws.S, ws.part_ml, ws.part_acc, out, err, s);
    if (e != cudaSuccess || ws.S == 1) return e;
    if (ws.S <= 32) return launch_tc_merge(L, ws.part_ml, ws.part_acc, ws.S, B, sink, pos, inv_freq, out, s);
    CSA_LAUNCH(k_attend_merge<T>, dim3(L.H, B), dim3(max(32, min(1024, L.D / 8))), ws.S * sizeof(float), s,
               ws.part_ml, ws.part_acc, ws.S, L.H, L.D, L.R, sink, pos, 0, inv_freq, static_cast<T*>(out));
    return cudaGetLastError();
  }
  CSA_LAUNCH(k_window_append<T>, dim3(B), dim3(128), 0, s, static_cast<const T*>(kv_new), static_cast<T*>(window), L.Wr, L.D, L.R, pos,
                                       inv_freq);
  CSA_LAUNCH(k_rope_rows<T>, dim3(B), dim3(256), 0, s, static_cast<const T*>(q), static_cast<T*>(ws.qr), L.H, L.D, L.R, pos, 0,
                                   inv_freq);
  AttnArgs a{};
  a.qr = ws.qr; a.pool = pool; a.ring = window; a.kvr = nullptr; a.sel = sel; a.n_sel = n_sel;
  a.n_rows = n_rows; a.pos = pos; a.sink = sink; a.inv_freq = inv_freq; a.pos0 = 0; a.cap = cap;
  a.topk = L.topk; a.W = L.W; a.Wr = L.Wr; a.H = L.H; a.D = L.D; a.R = L.R; a.ratio = L.ratio; a.scale = L.scale;
  a.S = ws.S; a.part_ml = ws.part_ml; a.part_acc = ws.part_acc; a.out = out; a.err = err;
  return run_attend<T>(a, B, s);
}

template <typename T>
static cudaError_t prefill_t(const Dims& L, const void* q, const void* kv_new, const float* sink, int T_, int pos0,
                             void* window, const void* pool, int cap, const int32_t* n_rows, const int32_t* sel,
                             const int32_t* n_sel, const float* inv_freq, void* out, const AttendWs& ws,
                             int32_t* err, cudaStream_t s) {
  CSA_LAUNCH(k_rope_rows<T>, dim3(T_), dim3(256), 0, s, static_cast<const T*>(kv_new), static_cast<T*>(ws.kvr), 1, L.D, L.R, nullptr,
                                    pos0, inv_freq);
  if (tc_attend_supported(L)) {
    cudaError_t e = launch_tc_attend_prefill(L, q, pool, window, ws.kvr, sel, n_sel, n_rows, pos0, cap, sink,
                                             inv_freq, T_, out, err, s);
    if (e != cudaSuccess) return e;
    CSA_LAUNCH(k_window_store_chunk<T>, dim3(min(T_, L.Wr)), dim3(64), 0, s, static_cast<const T*>(ws.kvr), static_cast<T*>(window), L.Wr,
                                                        L.D, T_, pos0);
    return cudaGetLastError();
  }
  CSA_LAUNCH(k_rope_rows<T>, dim3(T_), dim3(256), 0, s, static_cast<const T*>(q), static_cast<T*>(ws.qr), L.H, L.D, L.R, nullptr, pos0,
                                    inv_freq);
  AttnArgs a{};
  a.qr = ws.qr; a.pool = pool; a.ring = window; a.kvr = ws.kvr; a.sel = sel; a.n_sel = n_sel;
  a.n_rows = n_rows; a.pos = nullptr; a.sink = sink; a.inv_freq = inv_freq; a.pos0 = pos0; a.cap = cap;
  a.topk = L.topk; a.W = L.W; a.Wr = L.Wr; a.H = L.H; a.D = L.D; a.R = L.R; a.ratio = L.ratio; a.scale = L.scale;
  a.S = ws.S; a.part_ml = ws.part_ml; a.part_acc = ws.part_acc; a.out = out; a.err = err;
  cudaError_t e = run_attend<T>(a, T_, s);
  if (e != cudaSuccess) return e;
  CSA_LAUNCH(k_window_store_chunk<T>, dim3(min(T_, L.Wr)), dim3(64), 0, s, static_cast<const T*>(ws.kvr), static_cast<T*>(window), L.Wr,
                                                      L.D, T_, pos0);
  return cudaGetLastError();
}

// Verify blocks: window[b][(pos[b] + i) mod Wr] = RoPE(kv_new[b][i], pos[b] + i) for the block's T tokens.  It lets
// the next kernel start only once it has written the ring (no early trigger), since the attention kernel reads
// window rows before its own programmatic wait.
template <typename T>
__global__ void k_window_append_block(const T* __restrict__ kv, T* __restrict__ window, int Wr, int D, int R, int T_,
                                      const int32_t* __restrict__ pos, const float* __restrict__ inv_freq) {
  pdl_wait();
  const int b = blockIdx.x / T_, i = blockIdx.x % T_;
  const int p = pos[b] + i;
  if (pos[b] < 0) return;
  const T* row = kv + (size_t)blockIdx.x * D;
  T* dst = window + ((size_t)b * Wr + (p % Wr)) * D;
  for (int c = threadIdx.x; c < D; c += blockDim.x) {
    float v = to_f(row[c]);
    if (c >= D - R) {
      const int k = (c - (D - R)) >> 1;
      float cs, sn;
      rope_cs(p, inv_freq, k, &cs, &sn);
      const float a = to_f(row[D - R + 2 * k]), bb = to_f(row[D - R + 2 * k + 1]);
      v = ((c - (D - R)) & 1) ? fmaf(a, sn, bb * cs) : fmaf(a, cs, -bb * sn);
    }
    dst[c] = from_f<T>(v);
  }
}

cudaError_t launch_attend_verify(const Dims& L, const void* q, const void* kv_new, const float* sink, int B, int T_,
                                 void* window, const void* pool, int cap, const int32_t* n_rows, const int32_t* sel,
                                 const int32_t* n_sel, const int32_t* pos, const float* inv_freq, void* out,
                                 const AttendWs& ws, int32_t* err, cudaStream_t s) {
  const int Q = B * T_;
  const int S = tc_attend_decode_splits(Q, L.W, L.topk, ws.S);
  if (S < 1 || S > 32) return cudaErrorNotSupported;
  CSA_LAUNCH(k_window_append_block<__nv_bfloat16>, dim3(Q), dim3(128), 0, s,
             static_cast<const __nv_bfloat16*>(kv_new), static_cast<__nv_bfloat16*>(window), L.Wr, L.D, L.R, T_, pos,
             inv_freq);
  // Many queries (more than one wave of split items): the pipelined kernel, a CTA per query streaming its tiles,
  // with no partials to merge.  Few: the split decode kernel, whose items fill the SMs.
  int sms = 0, dev = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if ((long)Q * S > sms)
    return launch_tc_attend_prefill(L, q, pool, window, nullptr, sel, n_sel, n_rows, 0, cap, sink, inv_freq, Q, out,
                                    err, s, pos, T_);
  const bool cluster = tc_attend_decode_cluster(S);
  cudaError_t e = launch_tc_attend_decode(L, q, pool, window, kv_new, sel, n_sel, n_rows, pos, cap, sink, inv_freq, Q,
                                          S, ws.part_ml, ws.part_acc, out, err, s, T_, true, cluster);
  if (e != cudaSuccess || S == 1 || cluster) return e;
  return launch_tc_merge(L, ws.part_ml, ws.part_acc, S, Q, sink, pos, inv_freq, out, s, T_);
}

// pos[b] += by: the decode loop's position advance, launched with programmatic serialisation like every kernel
// here, so it starts while the step's last kernel drains and only its store waits for it
// No early trigger: the next kernel starts once the new positions are written, since kernels read the positions
// of their step before their own programmatic wait.
__global__ void k_advance_positions(int32_t* __restrict__ pos, int B, int by) {
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  pdl_wait();
  if (b < B) pos[b] += by;
}

// csa_trim: per sequence, hw = max(hw, pos); refuse (sequence unchanged) unless 0 <= n_back, pos - n_back >= 0,
// pos - n_back >= hw - rollback and n_rows == pos / ratio; else pos -= n_back and n_rows = pos / ratio in every
// pool.  ("DeepSeek-V4-Flash: native deepseek_v4 AR backend", MTPLX #216, the MTP / speculative-lane post: an exact
// trim truncates emitted rows, rebuilds frontiers from a journal and keeps extra window rows, and refuses beyond
// its bound.)  Like the decode kernels it reads the state after its programmatic wait; it lets the next kernel
// start only once it has written pos, since kernels read positions before their own wait.
__global__ void k_trim(int B, const int32_t* __restrict__ n_back, int32_t* __restrict__ pos,
                       int32_t* __restrict__ n_rows_a, int32_t* __restrict__ n_rows_i, int32_t* __restrict__ hw,
                       int ratio, int rollback, int32_t* __restrict__ err) {
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  pdl_wait();
  if (b >= B) return;
  const int p = pos[b], n = n_back[b], h = max(hw[b], p), np = p - n;
  if (p < 0 || n_rows_a[b] != p / ratio || (n_rows_i && n_rows_i[b] != p / ratio)) {
    atomicOr(err, CSA_DEV_STATE);
    return;
  }
  if (n < 0 || np < 0 || np < h - rollback) {
    atomicOr(err, CSA_DEV_ROLLBACK);
    return;
  }
  hw[b] = h;
  pos[b] = np;
  n_rows_a[b] = np / ratio;
  if (n_rows_i) n_rows_i[b] = np / ratio;
}

cudaError_t launch_trim(const Dims& L, int B, const int32_t* n_back, int32_t* pos, int32_t* n_rows_a,
                        int32_t* n_rows_i, int32_t* hw, int32_t* err, cudaStream_t s) {
  CSA_LAUNCH(k_trim, dim3((B + 255) / 256), dim3(256), 0, s, B, n_back, pos, n_rows_a, n_rows_i, hw, L.ratio,
             L.rollback, err);
  return cudaGetLastError();
}

cudaError_t launch_advance_positions(int32_t* pos, int B, int by, cudaStream_t s) {
  CSA_LAUNCH(k_advance_positions, dim3((B + 255) / 256), dim3(256), 0, s, pos, B, by);
  return cudaGetLastError();
}

cudaError_t launch_attend_decode(const Dims& L, const void* q, const void* kv_new, const float* sink, int B,
                                 void* window, const void* pool, int cap, const int32_t* n_rows, const int32_t* sel,
                                 const int32_t* n_sel, const int32_t* pos, const float* inv_freq, void* out,
                                 const AttendWs& ws, int32_t* err, cudaStream_t s) {
  if (L.dtype == CSA_BF16)
    return decode_t<__nv_bfloat16>(L, q, kv_new, sink, B, window, pool, cap, n_rows, sel, n_sel, pos, inv_freq, out,
                                   ws, err, s);
  return decode_t<float>(L, q, kv_new, sink, B, window, pool, cap, n_rows, sel, n_sel, pos, inv_freq, out, ws, err,
                         s);
}

cudaError_t launch_attend_prefill_varlen(const Dims& L, const void* q, const void* kv_new, const float* sink, int B,
                                         const int32_t* cu, int N, int T_max, void* window, const void* pool, int cap,
                                         const int32_t* n_rows, const int32_t* sel, const int32_t* n_sel,
                                         const int32_t* pos, const float* inv_freq, void* out, const AttendWs& ws,
                                         int32_t* err, cudaStream_t s) {
  using T = __nv_bfloat16;
  if (!tc_attend_supported(L)) return cudaErrorNotSupported;
  CSA_LAUNCH(k_rope_rows_varlen<T>, dim3(N), dim3(128), 0, s, static_cast<const T*>(kv_new), static_cast<T*>(ws.kvr),
             L.D, L.R, pos, cu, B, inv_freq);
  cudaError_t e = launch_tc_attend_prefill(L, q, pool, window, ws.kvr, sel, n_sel, n_rows, 0, cap, sink, inv_freq, N,
                                           out, err, s, pos, B, cu);
  if (e != cudaSuccess) return e;
  CSA_LAUNCH(k_window_store_varlen<T>, dim3(max(1, min(T_max, L.Wr)), B), dim3(64), 0, s,
             static_cast<const T*>(ws.kvr), static_cast<T*>(window), L.Wr, L.D, N, pos, cu);
  return cudaGetLastError();
}

cudaError_t launch_attend_prefill(const Dims& L, const void* q, const void* kv_new, const float* sink, int T,
                                  int pos0, void* window, const void* pool, int cap, const int32_t* n_rows,
                                  const int32_t* sel, const int32_t* n_sel, const float* inv_freq, void* out,
                                  const AttendWs& ws, int32_t* err, cudaStream_t s) {
  if (L.dtype == CSA_BF16)
    return prefill_t<__nv_bfloat16>(L, q, kv_new, sink, T, pos0, window, pool, cap, n_rows, sel, n_sel, inv_freq,
                                    out, ws, err, s);
  return prefill_t<float>(L, q, kv_new, sink, T, pos0, window, pool, cap, n_rows, sel, n_sel, inv_freq, out, ws, err,
                          s);
}

}  // namespace csa
