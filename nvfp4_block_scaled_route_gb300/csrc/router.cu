// Router front-end: the step before the routing permutation.  For every
// token, logits = x W_r^T (bf16 inputs, fp32 sums), the k largest logits
// (ties to the lower expert id; slot j in descending-logit order), and their
// weights from a softmax (over the k selected logits, or the full softmax's
// probabilities of the selected experts).  The pages keep the router
// ("gate") weight in BF16 ("NVFP4 MegaMoE Debug Log", Checkpoint Layers) and
// the workloads route top-k with softmax weights; the rest is the plain
// reading of a top-k softmax router.
//
// Two launches.
//  * router_tc_kernel: the logits on the 5th-generation tensor cores.  A CTA
//    takes a tile of 128 tokens and one range of K: TMA brings the x tile
//    (128 x 64 bf16) and the router weight (E padded to a multiple of 16
//    rows x 64 bf16) stage by stage in the 128-byte-swizzled K-major layout,
//    one thread issues tcgen05.mma.kind::f16 (M = 128, N = E padded, K = 16)
//    into an fp32 accumulator in TMEM, and the four warps read it back
//    (tcgen05.ld) into the workspace as that range's partial logits.  The
//    logits are HBM-bound (48 flops per byte of x at E = 48), so the grid is
//    sized to stream from every SM: about two CTAs per SM, small batches
//    splitting K over several CTAs (the weight is then most of the bytes).
//  * router_topk_kernel: one warp per token sums the partials in range order
//    (deterministic), selects the top k and normalises.
#include <cuda_bf16.h>

#include "internal.h"
#include "ptx.cuh"

namespace nvmoe {
namespace {

constexpr int kSms = 152;                 // grid sizing target (GB300)
constexpr int kRtRows = 128;              // tokens per tile (MMA M)
constexpr int kRtK = 64;                  // K elements per stage (128 bytes of bf16)
constexpr int kRtStages = 4;
constexpr int kRtMinStages = 4;           // stages per CTA at least (fewer partials)
constexpr int kRtThreads = 128;
constexpr int kRtXBytes = kRtRows * 128;  // 16 KB

struct RtBars {
  uint64_t full[kRtStages];
  uint64_t empty[kRtStages];
  uint64_t done;
  uint32_t tmem;
  int abort;
};

__host__ __device__ inline int rt_npad(int E) { return (E + 15) / 16 * 16; }
__host__ __device__ inline int rt_stage_bytes(int E) { return kRtXBytes + rt_npad(E) * 128; }
inline size_t rt_smem_bytes(int E) {
  return static_cast<size_t>(kRtStages) * rt_stage_bytes(E) + 1024 + sizeof(RtBars);
}

// TMEM columns for the accumulator: a power of two >= max(32, N).
__device__ __forceinline__ uint32_t rt_tmem_cols(int n) {
  uint32_t c = 32;
  while (c < static_cast<uint32_t>(n)) c <<= 1;
  return c;
}

__global__ void __launch_bounds__(kRtThreads) router_tc_kernel(
    const __grid_constant__ CUtensorMap map_x, const __grid_constant__ CUtensorMap map_w,
    int64_t T, int E, int stages_total, int stages_per_split, float* __restrict__ partials,
    int* status) {
  extern __shared__ uint8_t raw[];
  uint8_t* smem = raw + ((1024u - (smem_u32(raw) & 1023u)) & 1023u);
  const int n_pad = rt_npad(E);
  const int stage_bytes = rt_stage_bytes(E);
  RtBars* bars = reinterpret_cast<RtBars*>(smem + kRtStages * stage_bytes);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tile = blockIdx.x, split = blockIdx.y;
  const int ks0 = split * stages_per_split;
  const int ks1 = min(stages_total, ks0 + stages_per_split);
  const uint32_t ncols = rt_tmem_cols(n_pad);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kRtStages; ++s) {
      mbar_init(&bars->full[s], 1);
      mbar_init(&bars->empty[s], 1);
    }
    mbar_init(&bars->done, 1);
    bars->abort = 0;
    fence_mbarrier_init();
    prefetch_tensormap(&map_x);
    prefetch_tensormap(&map_w);
  }
  if (warp == 1) {
    tmem_alloc(&bars->tmem, ncols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem;
  volatile int* abort = &bars->abort;

  if (warp == 0 && lane == 0) {
    // producer: x tile and the weight rows of each stage of this K range
    const uint64_t pol_x = policy_evict_first();
    const uint64_t pol_w = policy_evict_last();
    int stage = 0;
    uint32_t phase = 0;
    for (int ks = ks0; ks < ks1; ++ks) {
      if (!mbar_wait(&bars->empty[stage], phase ^ 1u, status, abort)) break;
      uint8_t* xs = smem + stage * stage_bytes;
      mbar_arrive_expect_tx(&bars->full[stage], static_cast<uint32_t>(stage_bytes));
      tma_load_2d(xs, &map_x, ks * 128, tile * kRtRows, &bars->full[stage], pol_x);
      tma_load_2d(xs + kRtXBytes, &map_w, ks * 128, 0, &bars->full[stage], pol_w);
      if (++stage == kRtStages) {
        stage = 0;
        phase ^= 1u;
      }
    }
  } else if (warp == 1 && lane == 0) {
    // MMA issuer: four K = 16 steps per stage, in K order
    const uint32_t idesc = idesc_bf16_f32(kRtRows, n_pad);
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    for (int ks = ks0; ks < ks1 && ok; ++ks) {
      if (!mbar_wait(&bars->full[stage], phase, status, abort)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t xa = smem_u32(smem + stage * stage_bytes);
      const uint32_t wa = xa + kRtXBytes;
#pragma unroll
      for (int kk = 0; kk < kRtK / 16; ++kk)
        mma_f16(tmem, smem_desc(xa + kk * 32, 16, 1024, 2), smem_desc(wa + kk * 32, 16, 1024, 2),
                idesc, (ks != ks0 || kk != 0) ? 1u : 0u);
      tc_commit(&bars->empty[stage]);
      if (++stage == kRtStages) {
        stage = 0;
        phase ^= 1u;
      }
    }
    tc_commit(&bars->done);
  }
  // epilogue: every warp reads its 32 TMEM lanes (token rows)
  __syncwarp();
  const bool ok = mbar_wait(&bars->done, 0, status, abort);
  tc_fence_after();
  if (ok) {
    const int64_t t = static_cast<int64_t>(tile) * kRtRows + warp * 32 + lane;
    float* out = partials + (static_cast<int64_t>(split) * T + t) * E;
    const uint32_t trow = tmem + (static_cast<uint32_t>(warp * 32) << 16);
    for (int c = 0; c < n_pad; c += 16) {
      uint32_t r[16];
      tmem_ld_32x32b_x16(trow + c, r);
      tmem_ld_wait();
      if (t < T) {
#pragma unroll
        for (int j = 0; j < 16; ++j)
          if (c + j < E) out[c + j] = __uint_as_float(r[j]);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, ncols);
  }
}

// (value, index) pair ordering of the selection: larger value first, the
// lower index on equal values.
__device__ __forceinline__ bool better(float v, int i, float bv, int bi) {
  return v > bv || (v == bv && i < bi);
}

__global__ void router_topk_kernel(const float* __restrict__ partials, int splits, int64_t T,
                                   int E, int k, int mode, int32_t* __restrict__ ids,
                                   float* __restrict__ weights) {
  const int lane = threadIdx.x & 31;
  const int64_t t = static_cast<int64_t>(blockIdx.x) * (blockDim.x / 32) + (threadIdx.x >> 5);
  if (t >= T) return;
  constexpr int kPer = kMaxExperts / 32;
  float l[kPer];
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    const int e = lane + 32 * i;
    float s = 0.0f;
    if (e < E) {
      // loads in batches of 8 (independent), adds in range order
      for (int p0 = 0; p0 < splits; p0 += 8) {
        float v[8];
#pragma unroll
        for (int q = 0; q < 8; ++q)
          v[q] = p0 + q < splits ? __ldg(partials + (static_cast<int64_t>(p0 + q) * T + t) * E + e)
                                 : 0.0f;
#pragma unroll
        for (int q = 0; q < 8; ++q)
          if (p0 + q < splits) s += v[q];
      }
    }
    l[i] = e < E ? s : -INFINITY;
  }
  // full softmax denominator needs the maximum over all experts
  float mx = -INFINITY;
#pragma unroll
  for (int i = 0; i < kPer; ++i) mx = fmaxf(mx, l[i]);
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, o));
  float den_all = 0.0f;
  if (mode == 1) {
#pragma unroll
    for (int i = 0; i < kPer; ++i)
      if (lane + 32 * i < E) den_all += expf(l[i] - mx);
    for (int o = 16; o > 0; o >>= 1) den_all += __shfl_xor_sync(0xFFFFFFFFu, den_all, o);
  }
  bool taken[kPer];
#pragma unroll
  for (int i = 0; i < kPer; ++i) taken[i] = lane + 32 * i >= E;
  float sel_v = 0.0f;       // lane j keeps the j-th selection
  int sel_i = 0;
  for (int j = 0; j < k; ++j) {
    float bv = -INFINITY;
    int bi = 0x7FFFFFFF;
#pragma unroll
    for (int i = 0; i < kPer; ++i)
      if (!taken[i] && better(l[i], lane + 32 * i, bv, bi)) {
        bv = l[i];
        bi = lane + 32 * i;
      }
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xFFFFFFFFu, bv, o);
      const int oi = __shfl_xor_sync(0xFFFFFFFFu, bi, o);
      if (better(ov, oi, bv, bi)) {
        bv = ov;
        bi = oi;
      }
    }
#pragma unroll
    for (int i = 0; i < kPer; ++i)
      if (bi == lane + 32 * i) taken[i] = true;
    if (lane == j) {
      sel_v = bv;
      sel_i = bi;
    }
  }
  // softmax weights: the largest selected logit is the first
  const float top = __shfl_sync(0xFFFFFFFFu, sel_v, 0);
  const float ex = lane < k ? expf(sel_v - top) : 0.0f;
  float den = ex;
  for (int o = 16; o > 0; o >>= 1) den += __shfl_xor_sync(0xFFFFFFFFu, den, o);
  if (lane < k) {
    ids[t * k + lane] = sel_i;
    weights[t * k + lane] =
        mode == 1 ? __fdiv_rn(expf(sel_v - mx), den_all) : __fdiv_rn(ex, den);
  }
}

// K ranges: about two CTAs per SM over (token tiles x ranges), whole stages
// per range, at least kRtMinStages of them (the top-k adds every range's
// partials).
int router_splits(int64_t T, int H) {
  const int64_t tiles = (T + kRtRows - 1) / kRtRows;
  const int stages = H / kRtK;
  int64_t s = (2 * kSms) / (tiles > 0 ? tiles : 1);
  const int64_t max_s = stages / kRtMinStages > 0 ? stages / kRtMinStages : 1;
  if (s > max_s) s = max_s;
  if (s < 1) s = 1;
  const int per = static_cast<int>((stages + s - 1) / s);
  return (stages + per - 1) / per;
}

PerDeviceOnce g_router_attr;

}  // namespace

size_t router_workspace_bytes(int64_t T, int H, int E) {
  return static_cast<size_t>(router_splits(T, H)) * static_cast<size_t>(T) * E * sizeof(float);
}

cudaError_t launch_router(const CUtensorMap& map_x, const CUtensorMap& map_w, int64_t T, int H,
                          int E, int k, int mode, int32_t* ids, float* weights, float* partials,
                          int* status, cudaStream_t stream) {
  const int stages = H / kRtK;
  const int splits = router_splits(T, H);
  const int per = (stages + splits - 1) / splits;
  const size_t smem = rt_smem_bytes(E);
  // the attribute is the largest any E takes (set once per device)
  cudaError_t e = set_smem_attr_once(g_router_attr,
                                     reinterpret_cast<const void*>(router_tc_kernel),
                                     static_cast<int>(rt_smem_bytes(kMaxExperts)));
  if (e != cudaSuccess) return e;
  const dim3 grid(static_cast<unsigned>((T + kRtRows - 1) / kRtRows), static_cast<unsigned>(splits));
  router_tc_kernel<<<grid, kRtThreads, smem, stream>>>(map_x, map_w, T, E, stages, per, partials,
                                                       status);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int warps = 8;
  router_topk_kernel<<<static_cast<unsigned>((T + warps - 1) / warps), warps * 32, 0, stream>>>(
      partials, splits, T, E, k, mode, ids, weights);
  return cudaGetLastError();
}

}  // namespace nvmoe
