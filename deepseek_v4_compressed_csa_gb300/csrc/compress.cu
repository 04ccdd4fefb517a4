// Gated-pooling compressor: projection, window pooling, RMSNorm, RoPE, emit.
//
// Definitions: "DeepSeek-V4-Flash: native deepseek_v4 AR backend" (MTPLX #216),
// "What V4 adds" (learned gated pooling, overlapping ratio-4 / non-overlapping
// ratio-128 windows, maintained incrementally) and "Decode path" (pool in fp32,
// cast back before the norm); "feat: add DeepSeek-V4 (Pro/Flash) model support"
// (mlx-lm #1189), OmarB97's RoPE fixes (a pool row is rotated when emitted, at
// its window start j*ratio) and stepnoy's "Fix" 3 (the chunk tail is carried
// across calls; the absolute position accumulates).
//
// One call = two or three launches on the caller's stream:
//   project    kv | gate rows of every new token (model dtype) -> workspace
//   pool_emit  one block per completed window: per-sequence state check
//              (n_rows == pos/ratio, capacity), softmax-weighted sum per channel,
//              RMSNorm, RoPE, store the row; for a single new token it also
//              writes the token's frontier slot and advances n_rows
//   finish     (chunks) rewrite the frontier ring with the newest tokens,
//              advance n_rows
#include "common.cuh"
#include "fp8_row.cuh"
#include "kernels.h"

namespace csa {

CompressWs carve_compress_varlen(Carver& c, const Dims& L, int d, int B, int N) {
  CompressWs w;
  w.flags = c.take<int32_t>(B);
  w.proj = c.take<char>((size_t)N * 2 * L.lanes * d * esize(L.dtype));
  w.part = nullptr;
  w.tickets = nullptr;
  if (tc_project_supported(L, d)) carve_tc_project(c, L, d, N, &w.part, &w.tickets);
  return w;
}

CompressWs carve_compress(Carver& c, const Dims& L, int d, int B, int T) {
  CompressWs w;
  w.flags = c.take<int32_t>(B);
  w.proj = c.take<char>((size_t)B * T * 2 * L.lanes * d * esize(L.dtype));
  w.part = nullptr;
  w.tickets = nullptr;
  if (tc_project_supported(L, d)) carve_tc_project(c, L, d, B * T, &w.part, &w.tickets);
  return w;
}

// out[tok][o] = sum_k W[o][k] x[tok][k]; W = [wkv ; wgate] (2*Ld rows).  One warp
// per output feature and NTOK tokens; fp32 accumulation in a fixed order.
template <typename T, int NTOK>
__global__ void __launch_bounds__(256) k_project_simt(const T* __restrict__ x, const T* __restrict__ wkv,
                                                      const T* __restrict__ wg, int ntok, int X, int Ld,
                                                      T* __restrict__ out) {
  pdl_trigger();
  pdl_wait();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int o = blockIdx.x * 8 + warp;
  if (o >= 2 * Ld) return;
  const int t0 = blockIdx.y * NTOK;
  const T* w = (o < Ld) ? wkv + (size_t)o * X : wg + (size_t)(o - Ld) * X;
  float acc[NTOK];
#pragma unroll
  for (int t = 0; t < NTOK; ++t) acc[t] = 0.f;
  for (int k = lane * 8; k < X; k += 256) {
    float wv[8];
    load8_nc(w + k, wv);
#pragma unroll
    for (int t = 0; t < NTOK; ++t) {
      if (t0 + t < ntok) {
        float xv[8];
        load8_nc(x + (size_t)(t0 + t) * X + k, xv);
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[t] = fmaf(wv[e], xv[e], acc[t]);
      }
    }
  }
#pragma unroll
  for (int t = 0; t < NTOK; ++t) {
    float v = warp_sum(acc[t]);
    if (lane == 0 && t0 + t < ntok) out[(size_t)(t0 + t) * 2 * Ld + o] = from_f<T>(v);
  }
}

// An index row of 128 values in shared memory (model dtype) -> its fp8 row at dst, written by warp 0 once every
// thread of the block has stored its values (all threads call this).
__device__ __forceinline__ void store_fp8_row(uint8_t* dst, const float* row) {
  __syncthreads();
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    const float4 v = *reinterpret_cast<const float4*>(row + 4 * lane);
    float u[4] = {v.x, v.y, v.z, v.w};
    float scale;
    const uint32_t packed = fp8_rotate_quantize(u, lane, &scale);
    fp8_row_store(dst, lane, packed, scale);
  }
}

// One block per (completed window i of this call, sequence b).
// Per-sequence state check of a compress call: n_rows == pos/ratio and every
// row the call emits fits the pool.  Returns the error bit (0 = valid).
__device__ __forceinline__ int compress_state_error(int p0, int n, int T_, int ratio, int cap) {
  if (p0 < 0 || n != p0 / ratio) return CSA_DEV_STATE;
  if ((long long)(p0 + (long long)T_) / ratio - 1 >= cap) return CSA_DEV_CAPACITY;
  return 0;
}

// One block per (completed window i of this call, sequence b).  Block (0, b)
// publishes the sequence's validity (flags[b], error word).  With fuse_finish
// (single-token calls) it also writes the new token's frontier slot and advances
// n_rows: a single new token's slot never holds a token some window still reads.
template <typename T>
__global__ void __launch_bounds__(256) k_pool_emit(int32_t* __restrict__ flags, const int32_t* __restrict__ pos,
                                                   int32_t* __restrict__ n_rows, int32_t* err, int fuse_finish,
                                                   int T_, int ratio, int lanes, int d, int R, int F,
                                                   T* __restrict__ frontier, const T* __restrict__ proj,
                                                   const float* __restrict__ ape, const float* __restrict__ norm_w,
                                                   float eps, const float* __restrict__ inv_freq,
                                                   T* __restrict__ pool, int cap, const float* __restrict__ part,
                                                   int splits, int part_stride, const int32_t* __restrict__ cu,
                                                   int N, int fp8) {
  pdl_trigger();
  pdl_wait();
  extern __shared__ float sm_pool[];  // [d] pooled, [d] normed, 32 reduction slots, [2*L*d] new token (part)
  float* u = sm_pool;
  float* y = sm_pool + d;
  float* red = sm_pool + 2 * d;
  float* cur = sm_pool + 2 * d + 32;
  const int b = blockIdx.y;
  const int p0 = pos[b];
  // a packed variable-length batch (cu non-null): this sequence's tokens are projection rows cu[b] .. cu[b+1]-1
  int row0 = b * T_, bad_table = 0;
  if (cu) {
    const int c0 = cu[b], c1 = cu[b + 1];
    bad_table = (c0 < 0 || c1 < c0 || c1 > N) ? CSA_DEV_STATE : 0;
    row0 = bad_table ? 0 : c0;
    T_ = bad_table ? 0 : c1 - c0;
  }
  const int bad = bad_table ? bad_table : compress_state_error(p0, n_rows[b], T_, ratio, cap);
  const int rowlen = 2 * lanes * d;
  if (blockIdx.x == 0) {
    __syncthreads();  // every thread of this block has read n_rows before thread 0 may advance it
    if (threadIdx.x == 0) {
      flags[b] = !bad;
      if (bad) atomicOr(err, bad);
    }
    if (fuse_finish && !bad) {
      T* dst = frontier + ((size_t)b * F + (p0 % F)) * rowlen;
      if (part) {
        // single new token with split-K partials: sum them in split order, round once to the model dtype
        for (int e = threadIdx.x * 4; e < rowlen; e += blockDim.x * 4) {
          // batches of 8 splits, each batch's loads issued before its adds; the sum stays in split order
          constexpr int kBatch = 8;
          float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
          for (int s0 = 0; s0 < splits; s0 += kBatch) {
            float4 v[kBatch];
#pragma unroll
            for (int i = 0; i < kBatch; ++i)
              if (s0 + i < splits)
                v[i] = __ldcg(reinterpret_cast<const float4*>(part + ((size_t)(s0 + i) * part_stride + b) * rowlen + e));
#pragma unroll
            for (int i = 0; i < kBatch; ++i)
              if (s0 + i < splits) {
                if (s0 + i == 0) {
                  acc = v[i];
                } else {
                  acc.x += v[i].x;
                  acc.y += v[i].y;
                  acc.z += v[i].z;
                  acc.w += v[i].w;
                }
              }
          }
          const float f[4] = {acc.x, acc.y, acc.z, acc.w};
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const T r = from_f<T>(f[i]);
            dst[e + i] = r;
            cur[e + i] = to_f(r);
          }
        }
        __syncthreads();
      } else {
        const T* src = proj + (size_t)b * rowlen;
        for (int e = threadIdx.x * 8; e < rowlen; e += blockDim.x * 8) copy8<T>(dst + e, src + e);
      }
    }
  }
  if (bad) return;
  const int first = p0 + (ratio - 1 - p0 % ratio);  // first token completing a window
  const int p = first + blockIdx.x * ratio;
  if (p >= p0 + T_) {
    if (fuse_finish && blockIdx.x == 0 && threadIdx.x == 0) n_rows[b] = (p0 + T_) / ratio;
    return;
  }
  const int j = (p + 1) / ratio - 1;
  const int Ld = lanes * d;
  const T* fr = frontier + (size_t)b * F * rowlen;
  const T* pj = proj + (size_t)row0 * rowlen;

  float ss = 0.f;
  const int t_lo = (lanes == 2) ? max(0, (j - 1) * ratio) : j * ratio;
  const int t_hi = (j + 1) * ratio;
  for (int c = threadIdx.x; c < d; c += blockDim.x) {
    // entries (token t, lane l): ratio 4 -> window j-1 via lane 0 (if j >= 1) and window j via lane 1.
    // Chunks of 8 entries: every load of a chunk is issued before its first use; online softmax across chunks.
    float m = -INFINITY, num = 0.f, den = 0.f;
    for (int t0 = t_lo; t0 < t_hi; t0 += 8) {
      float sv[8], kv[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const int t = t0 + k;
        sv[k] = -INFINITY;
        kv[k] = 0.f;
        if (t < t_hi) {
          const int l = (lanes == 2 && t >= j * ratio) ? 1 : 0;
          float g;
          if (t < p0) {
            const T* row = fr + (size_t)(t % F) * rowlen;
            g = to_f(row[Ld + l * d + c]);
            kv[k] = to_f(row[l * d + c]);
          } else if (part) {
            g = cur[Ld + l * d + c];
            kv[k] = cur[l * d + c];
          } else {
            const T* row = pj + (size_t)(t - p0) * rowlen;
            g = to_f(row[Ld + l * d + c]);
            kv[k] = to_f(row[l * d + c]);
          }
          sv[k] = g + __ldg(ape + (size_t)(t % ratio) * Ld + l * d + c);
        }
      }
      float cm = m;
#pragma unroll
      for (int k = 0; k < 8; ++k) cm = fmaxf(cm, sv[k]);
      const float al = (m == -INFINITY) ? 0.f : expf(m - cm);
      num *= al;
      den *= al;
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const float e = (sv[k] == -INFINITY) ? 0.f : expf(sv[k] - cm);
        den += e;
        num = fmaf(e, kv[k], num);
      }
      m = cm;
    }
    float uc = rnd<T>(num / den);
    u[c] = uc;
    ss = fmaf(uc, uc, ss);
  }
  ss = block_sum(ss, red);
  const float inv = 1.0f / sqrtf(ss / (float)d + eps);
  for (int c = threadIdx.x; c < d; c += blockDim.x) y[c] = rnd<T>(u[c] * inv * __ldg(norm_w + c));
  __syncthreads();
  T* dst = pool + ((size_t)b * cap + j) * d;
  for (int c = threadIdx.x; c < d; c += blockDim.x) {
    float v = y[c];
    if (c >= d - R) {
      const int i = (c - (d - R)) >> 1;
      float cs, sn;
      rope_cs(j * ratio, inv_freq, i, &cs, &sn);
      const float a = y[d - R + 2 * i], bb = y[d - R + 2 * i + 1];
      v = ((c - (d - R)) & 1) ? fmaf(a, sn, bb * cs) : fmaf(a, cs, -bb * sn);
    }
    if (fp8)
      u[c] = rnd<T>(v);  // the row in the model dtype, then rotated and quantised below
    else
      dst[c] = from_f<T>(v);
  }
  if (fp8) store_fp8_row(reinterpret_cast<uint8_t*>(pool) + ((size_t)b * cap + j) * kFp8RowBytes, u);
  if (fuse_finish && blockIdx.x == 0 && threadIdx.x == 0) n_rows[b] = (p0 + T_) / ratio;
}

// One new token per sequence, its projection as split-K partials (the decode step of a ratio-4 layer with two
// lanes): one block per sequence.  Same arithmetic as k_pool_emit, with its memory requests in two rounds:
// norm weights, APE and RoPE frequencies do not depend on the position and are requested with it; the
// partials and the window's seven older frontier entries are requested together once it is known (a token
// that completes a window has p = 3 mod 4, so its window covers tokens p-7 .. p in a fixed lane / APE order).
constexpr int kTokChans = 2;  // channels per pooling thread: d <= 512
// Threads of a single-token pooling block: all of them load the split-K partials (one round for up to 16 splits at
// the Flash shapes), the first 256 pool (so the arithmetic, the norm's reduction order included, is the chunk
// kernel's: the extra warps add zeros to the block sum).
constexpr int kTokThreads = 512;

// The bits of one element, by a load the compiler keeps where it is written, and their fp32 value (a bf16 is the
// high half of its fp32).  The single-token kernel loads the window's older entries this way, every load issued
// before any is used: converted as each arrived, the loads went out one after another.
__device__ __forceinline__ uint32_t ld_bits_now(const __nv_bfloat16* p) {
  unsigned short v;
  asm volatile("ld.global.nc.u16 %0, [%1];" : "=h"(v) : "l"(p));
  return v;
}
__device__ __forceinline__ uint32_t ld_bits_now(const float* p) {
  uint32_t v;
  asm volatile("ld.global.nc.u32 %0, [%1];" : "=r"(v) : "l"(p));
  return v;
}
__device__ __forceinline__ float bits_f(uint32_t v, const __nv_bfloat16*) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bits_f(uint32_t v, const float*) { return __uint_as_float(v); }

// One pool's side of a single-token pooling launch.
template <typename T>
struct TokPool {
  int32_t* flags;
  int32_t* n_rows;
  T* frontier;
  const float* ape;
  const float* norm_w;
  T* pool;
  const float* part;
  int d, cap, splits, part_stride;
  int fp8;  // the pool holds fp8 index rows (kFp8RowBytes each, pool then points at bytes)
};

// Blocks [0, B) serve pool pa, blocks [B, 2B) (when launched) pool pb: a ratio-4 layer's two pools of the same
// tokens in one launch.
template <typename T>
__global__ void __launch_bounds__(kTokThreads) k_pool_emit_token(TokPool<T> pa, TokPool<T> pb, int B,
                                                         const int32_t* __restrict__ pos, int32_t* err, int R, int F,
                                                         float eps, const float* __restrict__ inv_freq) {
  pdl_trigger();
  // this block's pool, field by field (a reference to one of the two parameters would move them to local memory)
  const bool second = blockIdx.x >= (unsigned)B;
  int32_t* __restrict__ flags = second ? pb.flags : pa.flags;
  int32_t* __restrict__ n_rows = second ? pb.n_rows : pa.n_rows;
  T* __restrict__ frontier = second ? pb.frontier : pa.frontier;
  const float* __restrict__ ape = second ? pb.ape : pa.ape;
  const float* __restrict__ norm_w = second ? pb.norm_w : pa.norm_w;
  T* __restrict__ pool = second ? pb.pool : pa.pool;
  const float* __restrict__ part = second ? pb.part : pa.part;
  const int d = second ? pb.d : pa.d, cap = second ? pb.cap : pa.cap;
  const int splits = second ? pb.splits : pa.splits, part_stride = second ? pb.part_stride : pa.part_stride;
  const int fp8 = second ? pb.fp8 : pa.fp8;
  constexpr int ratio = 4, lanes = 2, kEnt = ratio * lanes;
  extern __shared__ float sm_tok[];  // [2*L*d] the new token, [d] pooled, [d] normed, 32 reduction slots, [R] rope
  const int Ld = lanes * d, rowlen = 2 * Ld;
  float* cur = sm_tok;
  float* u = cur + rowlen;
  float* y = u + d;
  float* red = y + d;
  float* rc = red + 32;
  float* rs = rc + R / 2;
  const int b = blockIdx.x - (second ? B : 0), tid = threadIdx.x;
  const int cb = tid < 256 ? tid : (1 << 20);  // pooling channels cb + 256 i on threads 0-255 only
  // before the preceding kernel has completed: the position (a step input) and the layer's constants, which no
  // kernel writes
  const int p0 = pos[b];
  float nw[kTokChans], ap[kTokChans][kEnt];
#pragma unroll
  for (int i = 0; i < kTokChans; ++i) {
    const int c = cb + 256 * i;
    nw[i] = c < d ? __ldg(norm_w + c) : 0.f;
#pragma unroll
    for (int e = 0; e < kEnt; ++e)  // entry e: token p-7+e, APE row e mod ratio, lane e / ratio
      ap[i][e] = c < d ? __ldg(ape + (size_t)(e % ratio) * Ld + (e / ratio) * d + c) : 0.f;
  }
  const float fq = tid < R / 2 ? __ldg(inv_freq + tid) : 0.f;
  pdl_wait();
  // one round of requests: n_rows, the partials of the new token and, if it completes window j, the window's
  // older entries (their bits, converted where the pooling uses them; this kernel writes no slot it reads them
  // from); nothing is written before the state check
  const int n = n_rows[b];
  const bool completes = (p0 + 1) % ratio == 0;
  const int j = (p0 + 1) / ratio - 1;
  const T* fr = frontier + (size_t)b * F * rowlen;
  uint32_t g[kTokChans][kEnt - 1], kv[kTokChans][kEnt - 1];
  if (completes) {
#pragma unroll
    for (int i = 0; i < kTokChans; ++i) {
      const int c = cb + 256 * i;
#pragma unroll
      for (int e = 0; e < kEnt - 1; ++e) {
        const int t = p0 - (kEnt - 1) + e;
        g[i][e] = 0u;
        kv[i][e] = 0u;
        if (c < d && t >= 0) {
          const T* row = fr + (size_t)(t % F) * rowlen + (e / ratio) * d + c;
          g[i][e] = ld_bits_now(row + Ld);
          kv[i][e] = ld_bits_now(row);
        }
      }
    }
  }
  for (int e = tid * 4; e < rowlen; e += kTokThreads * 4) {
    // batches of 16 splits, each batch's loads issued before its adds; the sum stays in split order
    constexpr int kBatch = 16;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int s0 = 0; s0 < splits; s0 += kBatch) {
      float4 v[kBatch];
#pragma unroll
      for (int i = 0; i < kBatch; ++i)
        if (s0 + i < splits)
          v[i] = __ldcg(reinterpret_cast<const float4*>(part + ((size_t)(s0 + i) * part_stride + b) * rowlen + e));
#pragma unroll
      for (int i = 0; i < kBatch; ++i)
        if (s0 + i < splits) {
          if (s0 + i == 0) {
            acc = v[i];
          } else {
            acc.x += v[i].x;
            acc.y += v[i].y;
            acc.z += v[i].z;
            acc.w += v[i].w;
          }
        }
    }
    const float f[4] = {acc.x, acc.y, acc.z, acc.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) cur[e + i] = to_f(from_f<T>(f[i]));  // the token in the model dtype
  }
  if (tid < R / 2) {
    float cs, sn;
    sincosf(__fmul_rn((float)(j * ratio), fq), &sn, &cs);
    rc[tid] = cs;
    rs[tid] = sn;
  }
  const int bad = compress_state_error(p0, n, 1, ratio, cap);
  __syncthreads();  // every thread has read n_rows before thread 0 may advance it; the token is in shared memory
  if (tid == 0) {
    flags[b] = !bad;
    if (bad) atomicOr(err, bad);
  }
  if (bad) return;
  {
    T* dst = frontier + ((size_t)b * F + (p0 % F)) * rowlen;
    for (int e = tid; e < rowlen; e += kTokThreads) dst[e] = from_f<T>(cur[e]);
  }
  if (!completes) {
    if (tid == 0) n_rows[b] = (p0 + 1) / ratio;
    return;
  }
  // window j: entries p-7 .. p (lane 0 for window j-1, lane 1 for window j); the last is the new token
  float ss = 0.f;
#pragma unroll
  for (int i = 0; i < kTokChans; ++i) {
    const int c = cb + 256 * i;
    if (c >= d) continue;
    float sv[kEnt], kk[kEnt];
#pragma unroll
    for (int e = 0; e < kEnt; ++e) {
      const int t = p0 - (kEnt - 1) + e;
      if (t < 0) {
        sv[e] = -INFINITY;
        kk[e] = 0.f;
      } else if (e == kEnt - 1) {
        sv[e] = cur[Ld + d + c] + ap[i][e];
        kk[e] = cur[d + c];
      } else {
        sv[e] = bits_f(g[i][e], fr) + ap[i][e];
        kk[e] = bits_f(kv[i][e], fr);
      }
    }
    float m = -INFINITY;
#pragma unroll
    for (int e = 0; e < kEnt; ++e) m = fmaxf(m, sv[e]);
    float num = 0.f, den = 0.f;
#pragma unroll
    for (int e = 0; e < kEnt; ++e) {
      const float x = (sv[e] == -INFINITY) ? 0.f : expf(sv[e] - m);
      den += x;
      num = fmaf(x, kk[e], num);
    }
    const float uc = rnd<T>(num / den);
    u[c] = uc;
    ss = fmaf(uc, uc, ss);
  }
  ss = block_sum(ss, red);
  const float inv = 1.0f / sqrtf(ss / (float)d + eps);
#pragma unroll
  for (int i = 0; i < kTokChans; ++i) {
    const int c = cb + 256 * i;
    if (c < d) y[c] = rnd<T>(u[c] * inv * nw[i]);
  }
  __syncthreads();
  T* dst = pool + ((size_t)b * cap + j) * d;
  for (int c = tid; c < d; c += kTokThreads) {
    float v = y[c];
    if (c >= d - R) {
      const int i = (c - (d - R)) >> 1;
      const float a = y[d - R + 2 * i], bb = y[d - R + 2 * i + 1];
      v = ((c - (d - R)) & 1) ? fmaf(a, rs[i], bb * rc[i]) : fmaf(a, rc[i], -bb * rs[i]);
    }
    if (fp8)
      u[c] = rnd<T>(v);  // the row in the model dtype, then rotated and quantised below
    else
      dst[c] = from_f<T>(v);
  }
  if (fp8) store_fp8_row(reinterpret_cast<uint8_t*>(pool) + ((size_t)b * cap + j) * kFp8RowBytes, u);
  if (tid == 0) n_rows[b] = (p0 + 1) / ratio;
}

// A block of 2 <= T <= kBlockMax new tokens per sequence whose projections are split-K partials (a verify block of
// a ratio-4 layer with two lanes): one CTA per sequence and pool.  The CTA sums each token's partials in split
// order and rounds it to the model dtype (what the projection's own fix-up would store), holding the block's
// tokens and the seven frontier entries before it in shared memory, so the frontier is read before any slot is
// rewritten, whatever its length.  It then writes the newest min(T, F) tokens' frontier slots and pools every
// window the block completes with the arithmetic of k_pool_emit_token (entries p-7 .. p in lane / APE order):
// threads 0-255 pool (the others add zeros to the norm's reduction, which leaves it unchanged); all 1024 load,
// so the partials take about two memory round trips.
constexpr int kBlockMax = 16;
constexpr int kBlockOld = 7;  // frontier entries before the block that a window it completes can need
constexpr int kBlockThreads = 1024;

template <typename T>
__global__ void __launch_bounds__(kBlockThreads) k_pool_block(TokPool<T> pa, TokPool<T> pb, int B, int T_,
                                                    const int32_t* __restrict__ pos, int32_t* err, int R, int F,
                                                    float eps, const float* __restrict__ inv_freq, int ext_stride) {
  pdl_trigger();
  const bool second = blockIdx.x >= (unsigned)B;
  int32_t* __restrict__ flags = second ? pb.flags : pa.flags;
  int32_t* __restrict__ n_rows = second ? pb.n_rows : pa.n_rows;
  T* __restrict__ frontier = second ? pb.frontier : pa.frontier;
  const float* __restrict__ ape = second ? pb.ape : pa.ape;
  const float* __restrict__ norm_w = second ? pb.norm_w : pa.norm_w;
  T* __restrict__ pool = second ? pb.pool : pa.pool;
  const float* __restrict__ part = second ? pb.part : pa.part;
  const int d = second ? pb.d : pa.d, cap = second ? pb.cap : pa.cap;
  const int splits = second ? pb.splits : pa.splits, part_stride = second ? pb.part_stride : pa.part_stride;
  constexpr int ratio = 4, lanes = 2, kEnt = ratio * lanes;
  // shared: [kBlockOld + T][ext_stride] entries (model dtype) from token p0 - 7 on, [d] pooled, [d] normed,
  // 32 reduction slots
  extern __shared__ float sm_blk[];
  const int Ld = lanes * d, rowlen = 2 * Ld;
  T* ext = reinterpret_cast<T*>(sm_blk);
  float* u = reinterpret_cast<float*>(ext + (size_t)(kBlockOld + T_) * ext_stride);
  float* y = u + d;
  float* red = y + d;
  const int b = blockIdx.x - (second ? B : 0), tid = threadIdx.x;
  const int p0 = pos[b];
  pdl_wait();
  const int n = n_rows[b];
  const int bad = compress_state_error(p0, n, T_, ratio, cap);
  if (!bad) {
    // the seven older entries (rows of tokens p0-7 .. p0-1 that exist) and the block's tokens
    const T* fr = frontier + (size_t)b * F * rowlen;
    for (int e = tid * 8; e < kBlockOld * rowlen; e += kBlockThreads * 8) {
      const int k = e / rowlen, c = e % rowlen, t = p0 - kBlockOld + k;
      if (t >= 0) copy8<T>(ext + (size_t)k * ext_stride + c, fr + (size_t)(t % F) * rowlen + c);
    }
    for (int e = tid * 4; e < T_ * rowlen; e += kBlockThreads * 4) {
      const int i = e / rowlen, c = e % rowlen;
      // batches of 8 splits, each batch's loads issued before its adds; the sum stays in split order
      constexpr int kBatch = 8;
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int s0 = 0; s0 < splits; s0 += kBatch) {
        float4 v[kBatch];
#pragma unroll
        for (int k = 0; k < kBatch; ++k)
          if (s0 + k < splits)
            v[k] = __ldcg(reinterpret_cast<const float4*>(part + ((size_t)(s0 + k) * part_stride + b * T_ + i) *
                                                                 rowlen + c));
#pragma unroll
        for (int k = 0; k < kBatch; ++k)
          if (s0 + k < splits) {
            if (s0 + k == 0) {
              acc = v[k];
            } else {
              acc.x += v[k].x;
              acc.y += v[k].y;
              acc.z += v[k].z;
              acc.w += v[k].w;
            }
          }
      }
      T* dst = ext + (size_t)(kBlockOld + i) * ext_stride + c;
      dst[0] = from_f<T>(acc.x);
      dst[1] = from_f<T>(acc.y);
      dst[2] = from_f<T>(acc.z);
      dst[3] = from_f<T>(acc.w);
    }
  }
  __syncthreads();  // every thread has read n_rows and the frontier before either is written
  if (tid == 0) {
    flags[b] = !bad;
    if (bad) atomicOr(err, bad);
  }
  if (bad) return;
  {
    const int keep = min(T_, F);
    for (int e = tid * 8; e < keep * rowlen; e += kBlockThreads * 8) {
      const int i = T_ - keep + e / rowlen, c = e % rowlen;
      copy8<T>(frontier + ((size_t)b * F + (p0 + i) % F) * rowlen + c, ext + (size_t)(kBlockOld + i) * ext_stride + c);
    }
  }
  // windows j completed by the block: token 4j + 3 in [p0, p0 + T), the first j = floor(p0 / 4)
  for (int j = p0 / ratio; ratio * j + ratio - 1 < p0 + T_; ++j) {
    float ss = 0.f;
#pragma unroll
    for (int i = 0; i < kTokChans; ++i) {
      const int c = tid + 256 * i;
      if (tid >= 256 || c >= d) continue;
      float sv[kEnt], kk[kEnt];
#pragma unroll
      for (int e = 0; e < kEnt; ++e) {  // entry e: token 4j-4+e, APE row e mod 4, lane e / 4
        const int t = ratio * j + ratio - kEnt + e;
        if (t < 0) {
          sv[e] = -INFINITY;
          kk[e] = 0.f;
        } else {
          const T* row = ext + (size_t)(t - (p0 - kBlockOld)) * ext_stride + (e / ratio) * d + c;
          sv[e] = to_f(row[Ld]) + __ldg(ape + (size_t)(e % ratio) * Ld + (e / ratio) * d + c);
          kk[e] = to_f(row[0]);
        }
      }
      float m = -INFINITY;
#pragma unroll
      for (int e = 0; e < kEnt; ++e) m = fmaxf(m, sv[e]);
      float num = 0.f, den = 0.f;
#pragma unroll
      for (int e = 0; e < kEnt; ++e) {
        const float x = (sv[e] == -INFINITY) ? 0.f : expf(sv[e] - m);
        den += x;
        num = fmaf(x, kk[e], num);
      }
      const float uc = rnd<T>(num / den);
      u[c] = uc;
      ss = fmaf(uc, uc, ss);
    }
    ss = block_sum(ss, red);
    const float inv = 1.0f / sqrtf(ss / (float)d + eps);
#pragma unroll
    for (int i = 0; i < kTokChans; ++i) {
      const int c = tid + 256 * i;
      if (tid < 256 && c < d) y[c] = rnd<T>(u[c] * inv * __ldg(norm_w + c));
    }
    __syncthreads();
    T* dst = pool + ((size_t)b * cap + j) * d;
    for (int c = tid; c < d; c += kBlockThreads) {
      float v = y[c];
      if (c >= d - R) {
        const int i = (c - (d - R)) >> 1;
        float cs, sn;
        rope_cs(j * ratio, inv_freq, i, &cs, &sn);
        const float a = y[d - R + 2 * i], bb = y[d - R + 2 * i + 1];
        v = ((c - (d - R)) & 1) ? fmaf(a, sn, bb * cs) : fmaf(a, cs, -bb * sn);
      }
      dst[c] = from_f<T>(v);
    }
    __syncthreads();  // y is rewritten by the next window
  }
  if (tid == 0) n_rows[b] = (p0 + T_) / ratio;
}

// Rewrite the frontier slots of the newest min(T, F) tokens; block (0, b) advances n_rows.
template <typename T>
__global__ void k_compress_finish(const int32_t* __restrict__ flags, const int32_t* __restrict__ pos, int T_,
                                  int ratio, int F, int rowlen, const T* __restrict__ proj, T* __restrict__ frontier,
                                  int32_t* __restrict__ n_rows, const int32_t* __restrict__ cu) {
  pdl_trigger();
  pdl_wait();
  const int b = blockIdx.y;
  if (!flags[b]) return;  // also set for an inconsistent row-table entry
  const int p0 = pos[b];
  int row0 = b * T_;
  if (cu) {
    row0 = cu[b];
    T_ = cu[b + 1] - row0;
  }
  const int keep = min(T_, F);
  if (cu && (int)blockIdx.x >= keep) {
    if (blockIdx.x == 0 && threadIdx.x == 0) n_rows[b] = (p0 + T_) / ratio;
    return;
  }
  const int t = p0 + T_ - keep + blockIdx.x;
  const T* src = proj + ((size_t)row0 + (t - p0)) * rowlen;
  T* dst = frontier + ((size_t)b * F + (t % F)) * rowlen;
  for (int e = threadIdx.x * 8; e < rowlen; e += blockDim.x * 8) copy8<T>(dst + e, src + e);
  if (blockIdx.x == 0 && threadIdx.x == 0) n_rows[b] = (p0 + T_) / ratio;
}

template <typename T>
static cudaError_t compress_t(const Dims& L, const csa_compressor& comp, const void* x, int B, int T_,
                              const int32_t* pos, void* frontier, void* pool, int cap, int32_t* n_rows,
                              const float* inv_freq, const CompressWs& ws, int32_t* err, cudaStream_t s) {
  const int d = comp.d, Ld = L.lanes * d, rowlen = 2 * Ld;
  const int fp8 = L.ikey_fp8 && d == L.Di;  // the index pool of a layer with fp8 index rows
  const int ntok = B * T_;
  const int fuse = (T_ == 1);
  // single new token per sequence with split-K partials: the pooling kernel sums them (no fix-up pass)
  const float* part = nullptr;
  int splits = 1, part_stride = 0;
  if (tc_project_supported(L, d)) {
    splits = tc_project_splits(L, d, ntok);
    const bool consumer_sums = fuse && splits > 1;
    if (consumer_sums) {
      part = ws.part;
      part_stride = tc_project_cols(L, d, ntok);
    }
    cudaError_t e = launch_tc_project(L, d, x, ntok, comp.wkv, comp.wgate, ws.proj, ws.part, ws.tickets,
                                      !consumer_sums, err, s);
    if (e != cudaSuccess) return e;
  } else {
    dim3 gp((2 * Ld + 7) / 8, (ntok + 7) / 8);
    CSA_LAUNCH(k_project_simt<T, 8>, dim3(gp), dim3(256), 0, s, static_cast<const T*>(x), static_cast<const T*>(comp.wkv),
                                             static_cast<const T*>(comp.wgate), ntok, L.X, Ld,
                                             static_cast<T*>(ws.proj));
  }
  if (part && L.ratio == 4 && L.lanes == 2 && L.F >= 8 && d <= 256 * kTokChans) {
    const size_t smem = ((size_t)rowlen + 2 * (size_t)d + 32 + L.R) * sizeof(float);
    const TokPool<T> tp{ws.flags, n_rows, static_cast<T*>(frontier), comp.ape, comp.norm_w, static_cast<T*>(pool),
                        part, d, cap, splits, part_stride, fp8};
    CSA_LAUNCH(k_pool_emit_token<T>, dim3(B), dim3(kTokThreads), smem, s, tp, tp, B, pos, err, L.R, L.F, L.eps,
               inv_freq);
    return cudaGetLastError();
  }
  const int maxwin = (T_ + L.ratio - 1) / L.ratio;
  dim3 ge(maxwin, B);
  const size_t smem = (2 * (size_t)d + 32 + (part ? (size_t)rowlen : 0)) * sizeof(float);
  CSA_LAUNCH(k_pool_emit<T>, dim3(ge), dim3(256), smem, s, ws.flags, pos, n_rows, err, fuse, T_, L.ratio, L.lanes, d,
             L.R, L.F, static_cast<T*>(frontier), static_cast<const T*>(ws.proj), comp.ape, comp.norm_w, L.eps,
             inv_freq, static_cast<T*>(pool), cap, part, splits, part_stride, static_cast<const int32_t*>(nullptr),
             0, fp8);
  if (!fuse) {
    dim3 gf(min(T_, L.F), B);
    CSA_LAUNCH(k_compress_finish<T>, dim3(gf), dim3(128), 0, s, ws.flags, pos, T_, L.ratio, L.F, rowlen,
                                            static_cast<const T*>(ws.proj), static_cast<T*>(frontier), n_rows,
               static_cast<const int32_t*>(nullptr));
  }
  return cudaGetLastError();
}

// A packed variable-length batch: x [N, X] holds B chunks back to back (row table cu, the longest T_max tokens).
// One projection over the N rows, then per sequence the windows its chunk completes and its frontier slots.
template <typename T>
static cudaError_t compress_varlen_t(const Dims& L, const csa_compressor& comp, const void* x, int B,
                                     const int32_t* cu, int N, int T_max, const int32_t* pos, void* frontier,
                                     void* pool, int cap, int32_t* n_rows, const float* inv_freq,
                                     const CompressWs& ws, int32_t* err, cudaStream_t s) {
  const int d = comp.d, Ld = L.lanes * d, rowlen = 2 * Ld;
  const int fp8 = L.ikey_fp8 && d == L.Di;
  if (tc_project_supported(L, d)) {
    cudaError_t e = launch_tc_project(L, d, x, N, comp.wkv, comp.wgate, ws.proj, ws.part, ws.tickets, true, err, s);
    if (e != cudaSuccess) return e;
  } else {
    dim3 gp((2 * Ld + 7) / 8, (N + 7) / 8);
    CSA_LAUNCH(k_project_simt<T, 8>, dim3(gp), dim3(256), 0, s, static_cast<const T*>(x),
               static_cast<const T*>(comp.wkv), static_cast<const T*>(comp.wgate), N, L.X, Ld,
               static_cast<T*>(ws.proj));
  }
  // windows a chunk of T_max tokens can complete: ceil(T_max / ratio), one more when it starts mid-window
  const int maxwin = (T_max + L.ratio - 1) / L.ratio + 1;
  const size_t smem = (2 * (size_t)d + 32) * sizeof(float);
  CSA_LAUNCH(k_pool_emit<T>, dim3(maxwin, B), dim3(256), smem, s, ws.flags, pos, n_rows, err, 0, 0, L.ratio, L.lanes,
             d, L.R, L.F, static_cast<T*>(frontier), static_cast<const T*>(ws.proj), comp.ape, comp.norm_w, L.eps,
             inv_freq, static_cast<T*>(pool), cap, static_cast<const float*>(nullptr), 1, 0, cu, N, fp8);
  CSA_LAUNCH(k_compress_finish<T>, dim3(max(1, min(T_max, L.F)), B), dim3(128), 0, s, ws.flags, pos, 0, L.ratio, L.F,
             rowlen, static_cast<const T*>(ws.proj), static_cast<T*>(frontier), n_rows, cu);
  return cudaGetLastError();
}

cudaError_t launch_compress_varlen(const Dims& L, const csa_compressor& comp, const void* x, int B,
                                   const int32_t* cu, int N, int T_max, const int32_t* pos, void* frontier,
                                   void* pool, int cap, int32_t* n_rows, const float* inv_freq,
                                   const CompressWs& ws, int32_t* err, cudaStream_t s) {
  if (L.dtype == CSA_BF16)
    return compress_varlen_t<__nv_bfloat16>(L, comp, x, B, cu, N, T_max, pos, frontier, pool, cap, n_rows, inv_freq,
                                            ws, err, s);
  return compress_varlen_t<float>(L, comp, x, B, cu, N, T_max, pos, frontier, pool, cap, n_rows, inv_freq, ws, err,
                                  s);
}

// Both pools of a ratio-4 layer.  One token per sequence on the tensor-core path: the two projections as one
// grid and the two pooling steps as one launch; otherwise the two calls in turn.
static cudaError_t compress_pair_token(const Dims& L, const csa_compressor& ca, const csa_compressor& ci,
                                       const void* x, int B, const int32_t* pos, void* fa, void* pa, int cap_a,
                                       int32_t* na, void* fi, void* pi, int cap_i, int32_t* ni,
                                       const float* inv_freq, const CompressWs& wa, const CompressWs& wi,
                                       int32_t* err, cudaStream_t s, int sa, int si) {
  using T = __nv_bfloat16;
  cudaError_t e = launch_tc_project_pair(L, ca.d, ca.wkv, ca.wgate, wa.part, ci.d, ci.wkv, ci.wgate, wi.part, x, B,
                                         sa, si, err, s);
  if (e != cudaSuccess) return e;
  const TokPool<T> ta{wa.flags, na, static_cast<T*>(fa), ca.ape, ca.norm_w, static_cast<T*>(pa), wa.part, ca.d,
                      cap_a, sa, tc_project_cols(L, ca.d, B), 0};
  const TokPool<T> tb{wi.flags, ni, static_cast<T*>(fi), ci.ape, ci.norm_w, static_cast<T*>(pi), wi.part, ci.d,
                      cap_i, si, tc_project_cols(L, ci.d, B), L.ikey_fp8};
  const int dm = max(ca.d, ci.d);
  const size_t smem = ((size_t)2 * L.lanes * dm + 2 * (size_t)dm + 32 + L.R) * sizeof(float);
  CSA_LAUNCH(k_pool_emit_token<T>, dim3(2 * B), dim3(kTokThreads), smem, s, ta, tb, B, pos, err, L.R, L.F, L.eps,
             inv_freq);
  return cudaGetLastError();
}

// A verify block (2 <= T <= kBlockMax tokens per sequence, one token tile in all): the two projections as one
// grid, then k_pool_block for both pools in one launch.
static cudaError_t compress_pair_block(const Dims& L, const csa_compressor& ca, const csa_compressor& ci,
                                       const void* x, int B, int T_, const int32_t* pos, void* fa, void* pa,
                                       int cap_a, int32_t* na, void* fi, void* pi, int cap_i, int32_t* ni,
                                       const float* inv_freq, const CompressWs& wa, const CompressWs& wi,
                                       int32_t* err, cudaStream_t s, int sa, int si) {
  using T = __nv_bfloat16;
  const int ntok = B * T_;
  cudaError_t e = launch_tc_project_pair(L, ca.d, ca.wkv, ca.wgate, wa.part, ci.d, ci.wkv, ci.wgate, wi.part, x, ntok,
                                         sa, si, err, s);
  if (e != cudaSuccess) return e;
  const TokPool<T> ta{wa.flags, na, static_cast<T*>(fa), ca.ape, ca.norm_w, static_cast<T*>(pa), wa.part, ca.d,
                      cap_a, sa, tc_project_cols(L, ca.d, ntok), 0};
  const TokPool<T> tb{wi.flags, ni, static_cast<T*>(fi), ci.ape, ci.norm_w, static_cast<T*>(pi), wi.part, ci.d,
                      cap_i, si, tc_project_cols(L, ci.d, ntok), 0};
  const int dm = max(ca.d, ci.d), stride = 2 * L.lanes * dm;
  const size_t smem = (size_t)(kBlockOld + T_) * stride * sizeof(T) + (2 * (size_t)dm + 32) * sizeof(float);
  cudaFuncSetAttribute(k_pool_block<T>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  CSA_LAUNCH(k_pool_block<T>, dim3(2 * B), dim3(kBlockThreads), smem, s, ta, tb, B, T_, pos, err, L.R, L.F, L.eps,
             inv_freq, stride);
  return cudaGetLastError();
}

cudaError_t launch_compress_pair(const Dims& L, const csa_compressor& ca, const csa_compressor& ci, const void* x,
                                 int B, int T, const int32_t* pos, void* fa, void* pa, int cap_a, int32_t* na,
                                 void* fi, void* pi, int cap_i, int32_t* ni, const float* inv_freq,
                                 const CompressWs& wa, const CompressWs& wi, int32_t* err, cudaStream_t s) {
  int sa = 0, si = 0;
  const bool fused = T <= kBlockMax && L.dtype == CSA_BF16 && L.ratio == 4 && L.lanes == 2 && L.F >= 8 &&
                     ca.d <= 512 && ci.d <= 512 && tc_project_supported(L, ca.d) && tc_project_supported(L, ci.d) &&
                     wa.part && wi.part && plan_project_pair(L, ca.d, ci.d, B * T, &sa, &si);
  if (fused && T == 1)
    return compress_pair_token(L, ca, ci, x, B, pos, fa, pa, cap_a, na, fi, pi, cap_i, ni, inv_freq, wa, wi, err, s,
                               sa, si);
  if (fused && !L.ikey_fp8)  // the block kernel writes model-dtype rows only
    return compress_pair_block(L, ca, ci, x, B, T, pos, fa, pa, cap_a, na, fi, pi, cap_i, ni, inv_freq, wa, wi, err,
                               s, sa, si);
  cudaError_t e = launch_compress(L, ca, x, B, T, pos, fa, pa, cap_a, na, inv_freq, wa, err, s);
  if (e != cudaSuccess) return e;
  return launch_compress(L, ci, x, B, T, pos, fi, pi, cap_i, ni, inv_freq, wi, err, s);
}

cudaError_t launch_compress(const Dims& L, const csa_compressor& comp, const void* x, int B, int T,
                            const int32_t* pos, void* frontier, void* pool, int cap, int32_t* n_rows,
                            const float* inv_freq, const CompressWs& ws, int32_t* err, cudaStream_t s) {
  if (L.dtype == CSA_BF16)
    return compress_t<__nv_bfloat16>(L, comp, x, B, T, pos, frontier, pool, cap, n_rows, inv_freq, ws, err, s);
  return compress_t<float>(L, comp, x, B, T, pos, frontier, pool, cap, n_rows, inv_freq, ws, err, s);
}

}  // namespace csa
