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
// One persistent CTA per SM, 6 warps: warp 0 issues TMA loads (a resident
// query block plus a 4-stage ring of 32 KB key tiles), warp 1 owns tensor
// memory and issues the MMAs from one thread, warps 2-5 drain the two TMEM
// accumulators and write fp32 scores.
#include "common.cuh"
#include "kernels.h"
#include "tc.cuh"

namespace csa {

namespace {

constexpr int kStages = 4;
constexpr int kTileRows = 128;
constexpr int kTileBytes = kTileRows * 128 * 2;  // 128 rows x 128 bf16
constexpr int kThreads = 192;

struct IdxArgs {
  const int32_t* n_rows;
  const int32_t* pos;  // decode positions [Q] or null (prefill: pos0 + q)
  int pos0, ratio, topk, cap, Q, G, n_items, tiles_per_group;
  const float* wts;  // [Q, 64] head weights (iw * scale)
  float* scores;     // [Q, cap]
  int32_t* err;
};

__device__ __forceinline__ int idx_qpos(const IdxArgs& a, int q) { return a.pos ? a.pos[q] : a.pos0 + q; }
__device__ __forceinline__ int idx_nvis(const IdxArgs& a, int q) {
  const int b = a.pos ? q : 0;
  return min(min(a.n_rows[b], a.cap), (idx_qpos(a, q) + 1) / a.ratio);
}
// rows that group g must score (its last query sees the most rows); 0 if the
// group's queries keep every visible row anyway
__device__ __forceinline__ int group_rows(const IdxArgs& a, int g) {
  const int qlast = min(a.Q - 1, g * a.G + a.G - 1);
  const int nv = idx_nvis(a, qlast);
  return nv > a.topk ? nv : 0;
}

template <int G>
__global__ void __launch_bounds__(kThreads, 1)
    k_tc_index_scores(const __grid_constant__ CUtensorMap tm_keys, const __grid_constant__ CUtensorMap tm_q,
                      IdxArgs a) {
  pdl_trigger();
  constexpr int N = 64 * G;
  constexpr int QBYTES = N * 128 * 2;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* qbuf = smem;                  // [2 boxes][N rows][128 B]
  uint8_t* kbuf = smem + QBYTES;         // [kStages][2 boxes][128 rows][128 B]
  uint64_t* bars = reinterpret_cast<uint64_t*>(kbuf + kStages * kTileBytes);
  uint64_t* full = bars;                 // [kStages]
  uint64_t* empty = bars + kStages;      // [kStages]
  uint64_t* q_full = bars + 2 * kStages;
  uint64_t* q_empty = q_full + 1;
  uint64_t* acc_full = q_full + 2;       // [2]
  uint64_t* acc_empty = q_full + 4;      // [2]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(q_full + 6);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      tc::mbar_init(&full[s], 1);
      tc::mbar_init(&empty[s], 1);
    }
    tc::mbar_init(q_full, 1);
    tc::mbar_init(q_empty, 1);
    for (int i = 0; i < 2; ++i) {
      tc::mbar_init(&acc_full[i], 1);
      tc::mbar_init(&acc_empty[i], 128);
    }
    tc::fence_mbar_init();
  }
  pdl_wait();  // predecessor complete: its outputs are visible and its tensor memory is free
  if (warp == 1) {
    tc::tmem_alloc(tmem_slot, 2 * N);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_slot;

  const int per = (a.n_items + gridDim.x - 1) / gridDim.x;
  const int i_begin = blockIdx.x * per, i_end = min(a.n_items, i_begin + per);
  bool failed = false;

  if (warp == 0) {
    if (lane == 0) {
      tc::tma_prefetch(&tm_keys);
      tc::tma_prefetch(&tm_q);
      int cur_g = -1, stage = 0, n_q = 0;
      uint32_t phase = 0;
      int issued[kStages] = {0, 0, 0, 0};
      for (int it = i_begin; it < i_end && !failed; ++it) {
        const int g = it / a.tiles_per_group, t = it % a.tiles_per_group;
        if (t * kTileRows >= group_rows(a, g)) continue;
        if (g != cur_g) {
          if (cur_g >= 0 && !tc::mbar_wait(q_empty, (n_q - 1) & 1)) { failed = true; break; }
          tc::mbar_arrive_expect_tx(q_full, QBYTES);
          tc::tma_load_2d(qbuf, &tm_q, q_full, 0, g * N);
          tc::tma_load_2d(qbuf + QBYTES / 2, &tm_q, q_full, 64, g * N);
          cur_g = g;
          ++n_q;
        }
        if (!tc::mbar_wait(&empty[stage], phase ^ 1)) { failed = true; break; }
        const int krow = (a.pos ? g : 0) * a.cap + t * kTileRows;
        tc::mbar_arrive_expect_tx(&full[stage], kTileBytes);
        tc::tma_load_2d(kbuf + stage * kTileBytes, &tm_keys, &full[stage], 0, krow);
        tc::tma_load_2d(kbuf + stage * kTileBytes + kTileBytes / 2, &tm_keys, &full[stage], 64, krow);
        ++issued[stage];
        if (++stage == kStages) { stage = 0; phase ^= 1; }
      }
      // drain: every load issued must land before the CTA may exit
      for (int s = 0; s < kStages; ++s)
        if (issued[s] && !tc::mbar_wait(&full[s], (issued[s] - 1) & 1)) failed = true;
      if (n_q && !tc::mbar_wait(q_full, (n_q - 1) & 1)) failed = true;
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc = tc::idesc_bf16(128, N);
      int cur_g = -1, stage = 0, acc = 0, n_q = 0, n_acc[2] = {0, 0};
      uint32_t phase = 0;
      for (int it = i_begin; it < i_end; ++it) {
        const int g = it / a.tiles_per_group, t = it % a.tiles_per_group;
        if (t * kTileRows >= group_rows(a, g)) continue;
        if (g != cur_g) {
          if (cur_g >= 0) tc::mma_commit(q_empty);
          if (!tc::mbar_wait(q_full, n_q & 1)) { failed = true; break; }
          cur_g = g;
          ++n_q;
        }
        if (!tc::mbar_wait(&full[stage], phase)) { failed = true; break; }
        if (!tc::mbar_wait(&acc_empty[acc], (n_acc[acc] & 1) ^ 1)) { failed = true; break; }
        tc::fence_after_sync();
        const uint32_t a_base = tc::smem_u32(kbuf + stage * kTileBytes);
        const uint32_t b_base = tc::smem_u32(qbuf);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const uint64_t ad = tc::sdesc_kmajor_sw128(a_base + (k >> 2) * (kTileBytes / 2) + (k & 3) * 32);
          const uint64_t bd = tc::sdesc_kmajor_sw128(b_base + (k >> 2) * (QBYTES / 2) + (k & 3) * 32);
          tc::mma_bf16(tmem + acc * N, ad, bd, idesc, k > 0);
        }
        tc::mma_commit(&empty[stage]);
        tc::mma_commit(&acc_full[acc]);
        ++n_acc[acc];
        acc ^= 1;
        if (++stage == kStages) { stage = 0; phase ^= 1; }
      }
      // make sure every MMA has retired before tensor memory is released
      if (n_q > 0) {
        tc::mma_commit(q_empty);
        if (!tc::mbar_wait(q_empty, (n_q - 1) & 1)) failed = true;
      }
    }
  } else {
    // epilogue: warp w drains TMEM lanes 32*(w%4) .. +31
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    int acc = 0, n_acc[2] = {0, 0};
    for (int it = i_begin; it < i_end; ++it) {
      const int g = it / a.tiles_per_group, t = it % a.tiles_per_group;
      if (t * kTileRows >= group_rows(a, g)) continue;
      if (!tc::mbar_wait(&acc_full[acc], n_acc[acc] & 1)) { failed = true; break; }
      tc::fence_after_sync();
      const int j = t * kTileRows + row;
#pragma unroll
      for (int qq = 0; qq < G; ++qq) {
        const int q = g * G + qq;
        uint32_t v[64];
        const uint32_t taddr = tmem + ((uint32_t)(quarter * 32) << 16) + acc * N + qq * 64;
        tc::tmem_ld32(taddr, v);
        tc::tmem_ld32(taddr + 32, v + 32);
        tc::tmem_wait_ld();
        if (q < a.Q) {
          const float* w = a.wts + (size_t)q * 64;
          float s = 0.f;
#pragma unroll
          for (int h = 0; h < 64; ++h) s = fmaf(__ldg(w + h), fmaxf(__uint_as_float(v[h]), 0.f), s);
          if (j < idx_nvis(a, q)) a.scores[(size_t)q * a.cap + j] = s;
        }
      }
      tc::fence_before_sync();
      tc::mbar_arrive(&acc_empty[acc]);
      ++n_acc[acc];
      acc ^= 1;
    }
  }
  if (failed) atomicOr(a.err, tc::kErrTimeout);
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 1) tc::tmem_dealloc(tmem, 2 * N);
}

// qr[q][h][:] = RoPE(iq[q][h][:], p_q) (bf16), wts[q][h] = iw[q][h] * scale.
// Block (q, head group of 8): one 16-byte chunk of 8 dims per thread.
__global__ void __launch_bounds__(128) k_tc_index_prep(const __nv_bfloat16* __restrict__ iq,
                                                       const __nv_bfloat16* __restrict__ iw,
                                                       const int32_t* __restrict__ pos, int pos0, int R,
                                                       const float* __restrict__ inv_freq, float wscale,
                                                       __nv_bfloat16* __restrict__ qr, float* __restrict__ wts) {
  pdl_trigger();
  pdl_wait();
  constexpr int Hi = 64, Di = 128;
  __shared__ float rc[64], rs[64];
  const int q = blockIdx.x, h0 = blockIdx.y * 8;
  const int p = pos ? pos[q] : pos0 + q;
  if (threadIdx.x < R / 2) rope_cs(p, inv_freq, threadIdx.x, &rc[threadIdx.x], &rs[threadIdx.x]);
  __syncthreads();
  const int h = h0 + (threadIdx.x >> 4), c = threadIdx.x & 15;  // 16 chunks of 8 dims per head row
  const size_t off = ((size_t)q * Hi + h) * Di + c * 8;
  uint4 raw = __ldg(reinterpret_cast<const uint4*>(iq + off));
  if (c * 8 >= Di - R) {
    __nv_bfloat162* hv = reinterpret_cast<__nv_bfloat162*>(&raw);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int i = (c * 8 - (Di - R)) / 2 + k;
      const float2 x = __bfloat1622float2(hv[k]);
      hv[k] = __floats2bfloat162_rn(fmaf(x.x, rc[i], -x.y * rs[i]), fmaf(x.x, rs[i], x.y * rc[i]));
    }
  }
  *reinterpret_cast<uint4*>(qr + off) = raw;
  if (threadIdx.x < 8) wts[(size_t)q * Hi + h0 + threadIdx.x] = __bfloat162float(iw[(size_t)q * Hi + h0 + threadIdx.x]) * wscale;
}

int g_num_sms = 0;

}  // namespace

bool tc_index_supported(const Dims& L) { return L.dtype == CSA_BF16 && L.Hi == 64 && L.Di == 128; }

size_t tc_index_ws(const Dims& L, int Q) {
  (void)L;
  return (size_t)Q * 64 * 128 * 2 + 256 + (size_t)Q * 64 * 4 + 256;
}

cudaError_t launch_tc_index_scores(const Dims& L, const void* iq, const void* iw, int Q, const void* ikeys, int Bk,
                                   int cap, const int32_t* n_rows, const int32_t* pos, int pos0,
                                   const float* inv_freq, void* ws, float* scores, int32_t* err, cudaStream_t s) {
  if (!g_num_sms) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&g_num_sms, cudaDevAttrMultiProcessorCount, dev);
  }
  Carver c(ws);
  __nv_bfloat16* qr = c.take<__nv_bfloat16>((size_t)Q * 64 * 128);
  float* wts = c.take<float>((size_t)Q * 64);
  const float wscale = (float)(1.0 / sqrt((double)L.Di * (double)L.Hi));
  CSA_LAUNCH(k_tc_index_prep, dim3(dim3(Q, 8)), dim3(128), 0, s, static_cast<const __nv_bfloat16*>(iq),
                                              static_cast<const __nv_bfloat16*>(iw), pos, pos0, L.R, inv_freq,
                                              wscale, qr, wts);
  const int G = pos ? 1 : 4;
  CUtensorMap tk, tq;
  if (!make_tmap_2d_bf16(&tk, ikeys, (uint64_t)Bk * cap, 128, 256, kTileRows)) return cudaErrorInvalidValue;
  if (!make_tmap_2d_bf16(&tq, qr, (uint64_t)Q * 64, 128, 256, 64 * G)) return cudaErrorInvalidValue;
  IdxArgs a{};
  a.n_rows = n_rows; a.pos = pos; a.pos0 = pos0; a.ratio = L.ratio; a.topk = L.topk; a.cap = cap; a.Q = Q;
  a.G = G; a.tiles_per_group = (cap + kTileRows - 1) / kTileRows;
  a.n_items = ((Q + G - 1) / G) * a.tiles_per_group;
  a.wts = wts; a.scores = scores; a.err = err;
  const int grid = min(g_num_sms, a.n_items);
  const size_t smem = 1024 + (size_t)64 * G * 128 * 2 + (size_t)kStages * kTileBytes + 256;
  if (G == 1) {
    cudaFuncSetAttribute(k_tc_index_scores<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    CSA_LAUNCH(k_tc_index_scores<1>, dim3(grid), dim3(kThreads), smem, s, tk, tq, a);
  } else {
    cudaFuncSetAttribute(k_tc_index_scores<4>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    CSA_LAUNCH(k_tc_index_scores<4>, dim3(grid), dim3(kThreads), smem, s, tk, tq, a);
  }
  
  return cudaGetLastError();
}

}  // namespace csa
