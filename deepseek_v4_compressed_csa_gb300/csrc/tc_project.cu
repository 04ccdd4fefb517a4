// Compressor projections on the 5th-generation tensor cores:
//   proj[tok][o] = sum_k W[o][k] x[tok][k],  W = [wkv ; wgate]  (2*L*d rows), bf16 out.
// ("DeepSeek-V4-Flash: native deepseek_v4 AR backend", MTPLX #216, "Decode path":
// projections kept at the model dtype; "feat: add DeepSeek-V4 (Pro/Flash) model
// support", mlx-lm #1189, Thump604: wkv/wgate (1024, 4096) on ratio-4 layers.)
//
// Computed transposed, C^T = W x^T: M = 128 output features per tile (TMEM lane =
// feature), N = up to 256 tokens, K = hidden size streamed by TMA in 64-wide
// blocks through a ring of stages.  Decode has few tokens (one per sequence), so
// the hidden axis is split across CTAs until ~150 CTAs stream the weights; each
// split writes fp32 partials and the last CTA of a tile (atomic ticket) sums
// them in split order, so the result does not depend on arrival order.
#include "common.cuh"
#include "kernels.h"
#include "tc.cuh"

namespace csa {

namespace {

constexpr int kPThreads = 192;  // warp 0 TMA, warp 1 MMA + TMEM, warps 2-5 epilogue
constexpr int kABytes = 128 * 128;  // 128 rows x 64 bf16
constexpr int kMaxSplits = 16;

struct PjArgs {
  int ntok, X, Ld, N, n_kblk, splits;  // n_kblk: 64-wide K blocks per split
  __nv_bfloat16* proj;                 // [ntok, 2*Ld]
  float* part;                         // [splits, n_tiles*N, 2*Ld] fp32 (splits > 1)
  int* tickets;                        // [m_tiles * n_tiles] zeroed before the launch
  int n_cols;                          // n_tiles * N
  int fixup;                           // splits > 1: 1 = sum the partials here; 0 = the consumer sums them
  int32_t* err;
};

// One (feature tile m, token tile n, split) of one projection: TMA ring, MMA, epilogue to proj or partials.
// Returns after the CTA's TMEM is released.
__device__ __forceinline__ void project_tile(const CUtensorMap* tm_wkv, const CUtensorMap* tm_wg,
                                             const CUtensorMap* tm_x, const PjArgs& a, int m, int n, int split,
                                             int stages, uint8_t* smem) {
  const int N = a.N;
  const int stage_bytes = kABytes + N * 128;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + stages * stage_bytes);
  uint64_t* empty = full + stages;
  uint64_t* acc_full = empty + stages;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acc_full + 1);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t tcols = N <= 32 ? 32 : (N <= 64 ? 64 : (N <= 128 ? 128 : 256));

  if (threadIdx.x == 0) {
    for (int s = 0; s < stages; ++s) {
      tc::mbar_init(&full[s], 1);
      tc::mbar_init(&empty[s], 1);
    }
    tc::mbar_init(acc_full, 1);
    tc::fence_mbar_init();
  }
  const int k0 = split * a.n_kblk;
  const CUtensorMap* wmap = (m * 128 < a.Ld) ? tm_wkv : tm_wg;
  const int wrow = (m * 128 < a.Ld) ? m * 128 : m * 128 - a.Ld;
  // The first fill of the ring is issued before the wait on the preceding kernel (by the thread that initialised
  // the barriers): weights and tokens are the call's inputs, which no kernel of this library writes.
  const int n_first = min(stages, a.n_kblk);
  if (threadIdx.x == 0) {
    tc::tma_prefetch(wmap);
    tc::tma_prefetch(tm_x);
    for (int kb = 0; kb < n_first; ++kb) {
      uint8_t* st = smem + kb * stage_bytes;
      tc::mbar_arrive_expect_tx(&full[kb], stage_bytes);
      tc::tma_load_2d(st, wmap, &full[kb], (k0 + kb) * 64, wrow);
      tc::tma_load_2d(st + kABytes, tm_x, &full[kb], (k0 + kb) * 64, n * N);
    }
  }
  pdl_wait();  // predecessor complete: its outputs are visible and its tensor memory is free
  // Successors may start only now: everything enqueued before this kernel is complete, so a successor that does
  // not wait for this kernel (the overlapped index scan) may write scratch memory an earlier call still read.
  pdl_trigger();
  if (warp == 1) {
    tc::tmem_alloc(tmem_slot, tcols);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  bool failed = false;

  if (warp == 0) {
    if (lane == 0) {
      int issued[8] = {0, 0, 0, 0, 0, 0, 0, 0};
      for (int kb = 0; kb < n_first; ++kb) ++issued[kb];
      for (int kb = n_first; kb < a.n_kblk; ++kb) {
        const int s = kb % stages;
        const uint32_t ph = (kb / stages) & 1;
        if (!tc::mbar_wait(&empty[s], ph ^ 1)) { failed = true; break; }
        uint8_t* st = smem + s * stage_bytes;
        tc::mbar_arrive_expect_tx(&full[s], stage_bytes);
        tc::tma_load_2d(st, wmap, &full[s], (k0 + kb) * 64, wrow);
        tc::tma_load_2d(st + kABytes, tm_x, &full[s], (k0 + kb) * 64, n * N);
        ++issued[s];
      }
      for (int s = 0; s < stages; ++s)
        if (issued[s] && !tc::mbar_wait(&full[s], (issued[s] - 1) & 1)) failed = true;
    }
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t idesc = tc::idesc_bf16(128, N);
      for (int kb = 0; kb < a.n_kblk; ++kb) {
        const int s = kb % stages;
        if (!tc::mbar_wait(&full[s], (kb / stages) & 1)) { failed = true; break; }
        tc::fence_after_sync();
        const uint32_t ab = tc::smem_u32(smem + s * stage_bytes);
#pragma unroll
        for (int k = 0; k < 4; ++k)
          tc::mma_bf16(tmem, tc::sdesc_kmajor_sw128(ab + k * 32), tc::sdesc_kmajor_sw128(ab + kABytes + k * 32),
                       idesc, (kb > 0 || k > 0) ? 1u : 0u);
        tc::mma_commit(&empty[s]);
      }
      tc::mma_commit(acc_full);  // also retires every MMA before the epilogue and the dealloc
    }
  } else {
    const int quarter = warp & 3;
    const int o = m * 128 + quarter * 32 + lane;  // output feature of this thread
    if (!tc::mbar_wait(acc_full, 0)) failed = true;
    tc::fence_after_sync();
    if (!failed) {
      for (int c0 = 0; c0 < N; c0 += 32) {
        uint32_t u[32];
        tc::tmem_ld32(tmem + ((uint32_t)(quarter * 32) << 16) + c0, u);
        tc::tmem_wait_ld();
        if (a.splits == 1) {
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const int tok = n * N + c0 + i;
            if (tok < a.ntok) a.proj[(size_t)tok * 2 * a.Ld + o] = __float2bfloat16_rn(__uint_as_float(u[i]));
          }
        } else {
          float* dst = a.part + ((size_t)split * a.n_cols + n * N + c0) * 2 * a.Ld + o;
#pragma unroll
          for (int i = 0; i < 32; ++i) dst[(size_t)i * 2 * a.Ld] = __uint_as_float(u[i]);
        }
      }
    }
  }
  if (failed) atomicOr(a.err, tc::kErrTimeout);
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 1) tc::tmem_dealloc(tmem, tcols);
}

__global__ void __launch_bounds__(kPThreads, 1)
    k_tc_project(const __grid_constant__ CUtensorMap tm_wkv, const __grid_constant__ CUtensorMap tm_wg,
                 const __grid_constant__ CUtensorMap tm_x, PjArgs a, int stages) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int m = blockIdx.x, n = blockIdx.y;
  project_tile(&tm_wkv, &tm_wg, &tm_x, a, m, n, blockIdx.z, stages, smem);
  if (a.splits == 1 || !a.fixup) return;
  int* s_last = reinterpret_cast<int*>(smem + stages * (kABytes + a.N * 128) + (2 * stages + 1) * 8 + 4);
  const int N = a.N;
  // split-K fix-up: the last CTA of the tile sums every split's partials in split order
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    const int t = atomicAdd(&a.tickets[m * gridDim.y + n], 1);
    *s_last = (t == a.splits - 1);
  }
  __syncthreads();
  if (!*s_last) return;
  __threadfence();
  // 4 features per task; every split's float4 is loaded before the (split-ordered) sum
  for (int e = threadIdx.x; e < N * 32; e += blockDim.x) {
    const int c = e / 32, o = m * 128 + (e % 32) * 4, tok = n * N + c;
    if (tok >= a.ntok) continue;
    constexpr int kBatch = 8;  // each batch's loads are issued before its adds; the sum stays in split order
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int s0 = 0; s0 < a.splits; s0 += kBatch) {
      float4 v[kBatch];
#pragma unroll
      for (int i = 0; i < kBatch; ++i)
        if (s0 + i < a.splits)
          v[i] = __ldcg(reinterpret_cast<const float4*>(a.part + ((size_t)(s0 + i) * a.n_cols + tok) * 2 * a.Ld + o));
#pragma unroll
      for (int i = 0; i < kBatch; ++i)
        if (s0 + i < a.splits) {
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
    __nv_bfloat16* dst = a.proj + (size_t)tok * 2 * a.Ld + o;
    *reinterpret_cast<__nv_bfloat162*>(dst) = __floats2bfloat162_rn(acc.x, acc.y);
    *reinterpret_cast<__nv_bfloat162*>(dst + 2) = __floats2bfloat162_rn(acc.z, acc.w);
  }
}

// The two projections of one token per sequence (attention pool and index pool, one token tile) in one grid:
// blocks [0, tiles0) are problem 0 (block = split * m_tiles0 + m), the rest problem 1.  Partials only: the pooling
// kernel sums them.
__global__ void __launch_bounds__(kPThreads, 1)
    k_tc_project_pair(const __grid_constant__ CUtensorMap tm_wkv0, const __grid_constant__ CUtensorMap tm_wg0,
                      const __grid_constant__ CUtensorMap tm_wkv1, const __grid_constant__ CUtensorMap tm_wg1,
                      const __grid_constant__ CUtensorMap tm_x, PjArgs a0, PjArgs a1, int m_tiles0, int m_tiles1,
                      int stages) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int tiles0 = m_tiles0 * a0.splits;
  const int bx = blockIdx.x;
  if (bx < tiles0)
    project_tile(&tm_wkv0, &tm_wg0, &tm_x, a0, bx % m_tiles0, 0, bx / m_tiles0, stages, smem);
  else
    project_tile(&tm_wkv1, &tm_wg1, &tm_x, a1, (bx - tiles0) % m_tiles1, 0, (bx - tiles0) / m_tiles1, stages, smem);
}

struct PjPlan {
  int N, n_tiles, m_tiles, splits;
};

PjPlan plan_project(const Dims& L, int d, int ntok) {
  PjPlan p;
  const int Ld = L.lanes * d;
  p.N = ntok >= 256 ? 256 : ((ntok + 31) / 32) * 32;  // multiple of 32: the epilogue drains 32 columns at a time
  p.n_tiles = (ntok + p.N - 1) / p.N;
  p.m_tiles = 2 * Ld / 128;
  const int base = p.m_tiles * p.n_tiles;
  const int kblk = L.X / 64;
  p.splits = 1;
  while (base * p.splits * 2 <= 160 && p.splits * 2 <= kMaxSplits && (kblk % (p.splits * 2)) == 0) p.splits *= 2;
  return p;
}

}  // namespace

bool tc_project_supported(const Dims& L, int d) {
  return L.dtype == CSA_BF16 && L.X % 64 == 0 && (2 * L.lanes * d) % 128 == 0;
}

void carve_tc_project(Carver& c, const Dims& L, int d, int ntok, float** part, int** tickets) {
  const PjPlan p = plan_project(L, d, ntok);
  if (p.splits > 1) {
    *part = c.take<float>((size_t)p.splits * 2 * L.lanes * d * p.n_tiles * p.N);
    *tickets = c.take<int>((size_t)p.m_tiles * p.n_tiles);
  } else {
    *part = nullptr;
    *tickets = nullptr;
  }
}

int tc_project_splits(const Dims& L, int d, int ntok) { return plan_project(L, d, ntok).splits; }
int tc_project_cols(const Dims& L, int d, int ntok) {
  const PjPlan p = plan_project(L, d, ntok);
  return p.n_tiles * p.N;
}

// The pair's CTAs run two per SM (their TMA rings sized to fit), so that both weight streams are in flight at
// once.  Measured on GB300 for the Flash shapes (B = 32): two CTAs per SM with a 5-stage ring took the decode
// step from 12.6k to 12.8k layer-steps/s against one CTA per SM with 8 stages.
constexpr int kPairCtasPerSm = 2;

int pair_stages(int N, int n_kblk_min) {
  const int stage_bytes = kABytes + N * 128;
  const int budget = 233472 / kPairCtasPerSm - 1024 - 1024 - 256;  // per-SM shared memory, reserve, slack
  return max(1, min(8, min(n_kblk_min, budget / stage_bytes)));
}

// Split counts for the two single-token projections run as one grid: powers of two no larger than each one's own
// plan (its workspace holds that many partials), at most kPairCtasPerSm CTAs per SM in total, the largest
// per-CTA weight share as small as possible.  False when the pair does not fit one wave even unsplit, or has
// more than one token tile.
bool plan_project_pair(const Dims& L, int d0, int d1, int ntok, int* s0, int* s1) {
  const PjPlan p0 = plan_project(L, d0, ntok), p1 = plan_project(L, d1, ntok);
  if (p0.n_tiles != 1 || p1.n_tiles != 1) return false;
  int sms = 0, dev = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  long best = -1;
  for (int a = 1; a <= p0.splits; a *= 2)
    for (int b = 1; b <= p1.splits; b *= 2) {
      if (p0.m_tiles * a + p1.m_tiles * b > kPairCtasPerSm * sms) continue;
      const long share = max((long)L.X / a, (long)L.X / b);  // K per CTA of the heavier problem
      if (best < 0 || share < best || (share == best && a * p0.m_tiles + b * p1.m_tiles > *s0 * p0.m_tiles + *s1 * p1.m_tiles)) {
        best = share;
        *s0 = a;
        *s1 = b;
      }
    }
  return best >= 0;
}

cudaError_t launch_tc_project_pair(const Dims& L, int d0, const void* wkv0, const void* wg0, float* part0, int d1,
                                   const void* wkv1, const void* wg1, float* part1, const void* x, int ntok, int s0,
                                   int s1, int32_t* err, cudaStream_t s) {
  const PjPlan p0 = plan_project(L, d0, ntok), p1 = plan_project(L, d1, ntok);
  const int Ld0 = L.lanes * d0, Ld1 = L.lanes * d1;
  CUtensorMap tw0, tg0, tw1, tg1, tx;
  if (!make_tmap_2d_bf16(&tw0, wkv0, Ld0, L.X, (uint64_t)L.X * 2, 128) ||
      !make_tmap_2d_bf16(&tg0, wg0, Ld0, L.X, (uint64_t)L.X * 2, 128) ||
      !make_tmap_2d_bf16(&tw1, wkv1, Ld1, L.X, (uint64_t)L.X * 2, 128) ||
      !make_tmap_2d_bf16(&tg1, wg1, Ld1, L.X, (uint64_t)L.X * 2, 128) ||
      !make_tmap_2d_bf16(&tx, x, ntok, L.X, (uint64_t)L.X * 2, p0.N))
    return cudaErrorInvalidValue;
  PjArgs a0{}, a1{};
  a0.ntok = ntok; a0.X = L.X; a0.Ld = Ld0; a0.N = p0.N; a0.splits = s0; a0.n_kblk = L.X / 64 / s0;
  a0.part = part0; a0.n_cols = p0.N; a0.fixup = 0; a0.err = err;
  a1 = a0;
  a1.Ld = Ld1; a1.splits = s1; a1.n_kblk = L.X / 64 / s1; a1.part = part1;
  const int stage_bytes = kABytes + p0.N * 128;
  const int stages = pair_stages(p0.N, min(a0.n_kblk, a1.n_kblk));
  const size_t smem = 1024 + (size_t)stages * stage_bytes + 256;
  cudaFuncSetAttribute(k_tc_project_pair, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  CSA_LAUNCH(k_tc_project_pair, dim3(p0.m_tiles * s0 + p1.m_tiles * s1), dim3(kPThreads), smem, s, tw0, tg0, tw1,
             tg1, tx, a0, a1, p0.m_tiles, p1.m_tiles, stages);
  return cudaGetLastError();
}

cudaError_t launch_tc_project(const Dims& L, int d, const void* x, int ntok, const void* wkv, const void* wgate,
                              void* proj, float* part, int* tickets, bool fixup, int32_t* err, cudaStream_t s) {
  const PjPlan p = plan_project(L, d, ntok);
  const int Ld = L.lanes * d;
  CUtensorMap tw, tg, tx;
  if (!make_tmap_2d_bf16(&tw, wkv, Ld, L.X, (uint64_t)L.X * 2, 128)) return cudaErrorInvalidValue;
  if (!make_tmap_2d_bf16(&tg, wgate, Ld, L.X, (uint64_t)L.X * 2, 128)) return cudaErrorInvalidValue;
  if (!make_tmap_2d_bf16(&tx, x, ntok, L.X, (uint64_t)L.X * 2, p.N)) return cudaErrorInvalidValue;
  PjArgs a{};
  a.ntok = ntok; a.X = L.X; a.Ld = Ld; a.N = p.N; a.splits = p.splits; a.n_kblk = L.X / 64 / p.splits;
  a.proj = static_cast<__nv_bfloat16*>(proj); a.part = part; a.tickets = tickets;
  a.n_cols = p.n_tiles * p.N; a.fixup = fixup ? 1 : 0; a.err = err;
  if (p.splits > 1 && fixup) {
    cudaMemsetAsync(tickets, 0, (size_t)p.m_tiles * p.n_tiles * sizeof(int), s);
  }
  const int stage_bytes = kABytes + p.N * 128;
  const int stages = min(8, min(a.n_kblk, (200 * 1024) / stage_bytes));
  const size_t smem = 1024 + (size_t)stages * stage_bytes + 256;
  cudaFuncSetAttribute(k_tc_project, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  dim3 grid(p.m_tiles, p.n_tiles, p.splits);
  CSA_LAUNCH(k_tc_project, dim3(grid), dim3(kPThreads), smem, s, tw, tg, tx, a, stages);
  return cudaGetLastError();
}

}  // namespace csa
