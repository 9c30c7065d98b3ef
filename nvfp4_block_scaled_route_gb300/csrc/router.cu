// Router front-end: the step before the routing permutation.  For every
// token, logits = x W_r^T (bf16 inputs, fp32 products and sums), the k
// largest logits (ties to the lower expert id; slot j in descending-logit
// order), and their weights from a softmax (over the k selected logits, or
// the full softmax's probabilities of the selected experts).
// The pages keep the router ("gate") weight in BF16 (NVFP4 MegaMoE Debug
// Log, Checkpoint Layers) and the workloads route top-k with softmax
// weights; the rest is the plain reading of a top-k softmax router.
//
// Two launches.  router_logits_kernel: a CTA takes 32 tokens x all experts
// x one K range and accumulates in K order; small batches split K over many
// CTAs (the router weight is the bulk of the bytes), each range's partial
// logits go to the workspace.  router_topk_kernel: one warp per token sums
// the partials in range order (deterministic), selects and normalises.
#include <cuda_bf16.h>

#include "internal.h"

namespace nvmoe {
namespace {

constexpr int kRouterThreads = 256;
constexpr int kTokPerCta = 32;
constexpr int kChunkK = 128;          // K elements staged per step
constexpr int kXStride = kChunkK + 2; // padded row (bf16): no bank conflicts across tokens

__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// partials[split][t][e] = sum over this split's K range, ascending k.
// NE: experts per thread (compile-time, so the accumulators stay in
// registers); thread group eg takes experts eg, eg + 8, ...
template <int NE>
__global__ void __launch_bounds__(kRouterThreads) router_logits_kernel(
    const __nv_bfloat16* __restrict__ x, const __nv_bfloat16* __restrict__ w, int64_t T, int H,
    int E, int k_per_split, float* __restrict__ partials) {
  extern __shared__ __align__(16) uint8_t smem[];
  __nv_bfloat16* xs = reinterpret_cast<__nv_bfloat16*>(smem);                    // [32][kXStride]
  __nv_bfloat16* ws = xs + kTokPerCta * kXStride;                                 // [E][kChunkK]
  const int t_local = threadIdx.x & 31;
  const int eg = threadIdx.x >> 5;                 // expert group 0..7: experts eg, eg+8, ...
  const int64_t t0 = static_cast<int64_t>(blockIdx.x) * kTokPerCta;
  const int k0 = blockIdx.y * k_per_split;
  const int k1 = min(H, k0 + k_per_split);
  constexpr int kMaxPerThread = NE;
  float acc[kMaxPerThread];
#pragma unroll
  for (int i = 0; i < kMaxPerThread; ++i) acc[i] = 0.0f;
  const int n_e = (E - eg + 7) / 8;                // experts of this thread's group
  for (int kc = k0; kc < k1; kc += kChunkK) {
    __syncthreads();
    // stage x[t0..t0+31][kc..kc+127] (pairs of bf16) and W[0..E-1][kc..kc+127]
    for (int i = threadIdx.x; i < kTokPerCta * (kChunkK / 2); i += kRouterThreads) {
      const int r = i / (kChunkK / 2), c = (i % (kChunkK / 2)) * 2;
      uint32_t v = 0;
      if (t0 + r < T)
        v = *reinterpret_cast<const uint32_t*>(x + (t0 + r) * H + kc + c);
      *reinterpret_cast<uint32_t*>(xs + r * kXStride + c) = v;
    }
    for (int i = threadIdx.x; i < E * (kChunkK / 8); i += kRouterThreads) {
      const int r = i / (kChunkK / 8), c = (i % (kChunkK / 8)) * 8;
      *reinterpret_cast<uint4*>(ws + r * kChunkK + c) =
          __ldg(reinterpret_cast<const uint4*>(w + static_cast<int64_t>(r) * H + kc + c));
    }
    __syncthreads();
    const uint32_t* xr = reinterpret_cast<const uint32_t*>(xs + t_local * kXStride);
    for (int c = 0; c < kChunkK / 2; ++c) {
      const uint32_t xv = xr[c];
      const float xa = bf_lo(xv), xb = bf_hi(xv);
#pragma unroll
      for (int i = 0; i < kMaxPerThread; ++i) {
        if (i < n_e) {
          const uint32_t wv =
              reinterpret_cast<const uint32_t*>(ws + (eg + 8 * i) * kChunkK)[c];
          acc[i] = __fmaf_rn(xa, bf_lo(wv), acc[i]);
          acc[i] = __fmaf_rn(xb, bf_hi(wv), acc[i]);
        }
      }
    }
  }
  const int64_t t = t0 + t_local;
  if (t < T) {
    float* out = partials + (static_cast<int64_t>(blockIdx.y) * T + t) * E;
#pragma unroll
    for (int i = 0; i < kMaxPerThread; ++i)
      if (i < n_e) out[eg + 8 * i] = acc[i];
  }
}

// Small batches (T <= kSmallT): one CTA per expert streams that expert's
// weight row once; thread i owns the 8-element groups i, i + 128, ... of H
// and accumulates every token over them; the 128 partial sums of a logit are
// then added in a fixed tree (warp shuffles, then the four warps in order).
constexpr int kSmallT = 32;
constexpr int kSms = 152;               // grid sizing target (GB300)
constexpr int kMmaMinT = 1024;          // tensor-core logits from this many tokens
constexpr int kSmallThreads = 128;

template <int TT>
__global__ void __launch_bounds__(kSmallThreads) router_logits_small_kernel(
    const __nv_bfloat16* __restrict__ x, const __nv_bfloat16* __restrict__ w, int T, int H,
    int E, float* __restrict__ logits) {
  __shared__ float red[kSmallThreads / 32][TT];
  const int e = blockIdx.x;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  float acc[TT];
#pragma unroll
  for (int t = 0; t < TT; ++t) acc[t] = 0.0f;
  const uint4* wr = reinterpret_cast<const uint4*>(w + static_cast<int64_t>(e) * H);
  const int groups = H / 8;
  // blocks of 8 groups per thread: all loads of a block are issued before
  // any is used (one memory round trip per block, not per group)
  for (int g0 = threadIdx.x; g0 < groups; g0 += 8 * kSmallThreads) {
    uint4 wv[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int g = g0 + j * kSmallThreads;
      wv[j] = g < groups ? __ldg(wr + g) : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int t = 0; t < TT; ++t) {
      if (t < T) {
        const uint4* xr = reinterpret_cast<const uint4*>(x + static_cast<int64_t>(t) * H);
        uint4 xv[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int g = g0 + j * kSmallThreads;
          xv[j] = g < groups ? __ldg(xr + g) : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const uint32_t w4[4] = {wv[j].x, wv[j].y, wv[j].z, wv[j].w};
          const uint32_t x4[4] = {xv[j].x, xv[j].y, xv[j].z, xv[j].w};
#pragma unroll
          for (int m = 0; m < 4; ++m) {
            acc[t] = __fmaf_rn(bf_lo(x4[m]), bf_lo(w4[m]), acc[t]);
            acc[t] = __fmaf_rn(bf_hi(x4[m]), bf_hi(w4[m]), acc[t]);
          }
        }
      }
    }
  }
#pragma unroll
  for (int t = 0; t < TT; ++t) {
    float v = acc[t];
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
    if (lane == 0) red[warp][t] = v;
  }
  __syncthreads();
  if (threadIdx.x < T) {
    const int t = threadIdx.x;
    float v = 0.0f;
#pragma unroll
    for (int q = 0; q < kSmallThreads / 32; ++q) v += red[q][t];
    logits[static_cast<int64_t>(t) * E + e] = v;
  }
}

// Larger batches: the logits as a tensor-core contraction.  A CTA takes 128
// tokens (8 warps x 16 rows) and a column tile of NT x 8 experts
// (blockIdx.y), and walks H in chunks of 64 that cp.async stages into a
// four-deep shared-memory ring (three chunks in flight while one is used);
// each warp issues mma.sync.m16n8k16 (bf16 in, fp32 accumulate) over its 16
// rows.  The K order is fixed, so the logits do not depend on timing.
constexpr int kMmaRows = 128;
constexpr int kMmaK = 64;
constexpr int kMmaStride = kMmaK + 8;   // bf16 per staged row (+16 B: no bank conflicts)

__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], const uint32_t (&a)[4],
                                               const uint32_t (&b)[2]) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
      "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

__device__ __forceinline__ void cp_async16(void* smem_dst, const void* src, bool valid) {
  // 16 bytes global -> shared, zero-filled when !valid (src is then not read)
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(
                   static_cast<uint32_t>(__cvta_generic_to_shared(smem_dst))),
               "l"(src), "r"(valid ? 16 : 0)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

constexpr int kMmaStages = 4;

template <int NT>
__global__ void __launch_bounds__(256) router_logits_mma_kernel(
    const __nv_bfloat16* __restrict__ x, const __nv_bfloat16* __restrict__ w, int64_t T, int H,
    int E, float* __restrict__ logits) {
  extern __shared__ __align__(16) uint8_t smem[];
  constexpr int kStageElems = (kMmaRows + NT * 8) * kMmaStride;
  __nv_bfloat16* stage_base = reinterpret_cast<__nv_bfloat16*>(smem);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int grp = lane >> 2, tig = lane & 3;
  const int64_t t0 = static_cast<int64_t>(blockIdx.x) * kMmaRows;
  const int e0 = blockIdx.y * NT * 8;     // first expert of this CTA's column tile
  const int chunks = H / kMmaK;
  // chunk c -> stage c % kMmaStages: 128 token rows then NT*8 expert rows
  auto load = [&](int c) {
    __nv_bfloat16* xs = stage_base + (c % kMmaStages) * kStageElems;
    __nv_bfloat16* ws = xs + kMmaRows * kMmaStride;
    const int kc = c * kMmaK;
    for (int i = threadIdx.x; i < kMmaRows * (kMmaK / 8); i += 256) {
      const int r = i / (kMmaK / 8), col = (i % (kMmaK / 8)) * 8;
      const bool ok = t0 + r < T;
      cp_async16(xs + r * kMmaStride + col, x + (ok ? (t0 + r) * H + kc + col : 0), ok);
    }
    for (int i = threadIdx.x; i < NT * 8 * (kMmaK / 8); i += 256) {
      const int r = i / (kMmaK / 8), col = (i % (kMmaK / 8)) * 8;
      const bool ok = e0 + r < E;
      cp_async16(ws + r * kMmaStride + col,
                 w + (ok ? static_cast<int64_t>(e0 + r) * H + kc + col : 0), ok);
    }
  };
  float acc[NT][4];
#pragma unroll
  for (int n = 0; n < NT; ++n)
#pragma unroll
    for (int i = 0; i < 4; ++i) acc[n][i] = 0.0f;
#pragma unroll
  for (int c = 0; c < kMmaStages - 1; ++c) {
    if (c < chunks) load(c);
    cp_async_commit();
  }
  for (int c = 0; c < chunks; ++c) {
    cp_async_wait<kMmaStages - 2>();          // chunk c has landed (this thread's part)
    __syncthreads();                           // ... and everyone's; stage of c-1 is free
    if (c + kMmaStages - 1 < chunks) load(c + kMmaStages - 1);
    cp_async_commit();
    const __nv_bfloat16* xs = stage_base + (c % kMmaStages) * kStageElems;
    const __nv_bfloat16* ws = xs + kMmaRows * kMmaStride;
    const __nv_bfloat16* xw = xs + (warp * 16) * kMmaStride;
#pragma unroll
    for (int k16 = 0; k16 < kMmaK; k16 += 16) {
      uint32_t a[4];
      a[0] = *reinterpret_cast<const uint32_t*>(xw + grp * kMmaStride + k16 + 2 * tig);
      a[1] = *reinterpret_cast<const uint32_t*>(xw + (grp + 8) * kMmaStride + k16 + 2 * tig);
      a[2] = *reinterpret_cast<const uint32_t*>(xw + grp * kMmaStride + k16 + 8 + 2 * tig);
      a[3] = *reinterpret_cast<const uint32_t*>(xw + (grp + 8) * kMmaStride + k16 + 8 + 2 * tig);
#pragma unroll
      for (int n = 0; n < NT; ++n) {
        const __nv_bfloat16* wr = ws + (n * 8 + grp) * kMmaStride + k16 + 2 * tig;
        uint32_t b[2];
        b[0] = *reinterpret_cast<const uint32_t*>(wr);
        b[1] = *reinterpret_cast<const uint32_t*>(wr + 8);
        mma_bf16_16816(acc[n], a, b);
      }
    }
  }
  cp_async_wait<0>();
  // D fragment: rows grp / grp + 8 of the warp's 16, columns 2*tig, 2*tig + 1
#pragma unroll
  for (int n = 0; n < NT; ++n) {
    const int e = e0 + n * 8 + 2 * tig;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int64_t t = t0 + warp * 16 + grp + 8 * h;
      if (t < T) {
        if (e < E) logits[t * E + e] = acc[n][2 * h];
        if (e + 1 < E) logits[t * E + e + 1] = acc[n][2 * h + 1];
      }
    }
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

int splits_for(int64_t T, int H) {
  if (T <= kSmallT || T >= kMmaMinT) return 1;
  const int64_t tiles = (T + kTokPerCta - 1) / kTokPerCta;
  int64_t s = (2 * kSms) / (tiles > 0 ? tiles : 1);
  const int max_s = H / kChunkK;
  if (s > max_s) s = max_s;
  if (s < 1) s = 1;
  return static_cast<int>(s);
}

}  // namespace

size_t router_workspace_bytes(int64_t T, int H, int E) {
  return static_cast<size_t>(splits_for(T, H)) * static_cast<size_t>(T) * E * sizeof(float);
}

cudaError_t launch_router(const void* x, const void* w, int64_t T, int H, int E, int k, int mode,
                          int32_t* ids, float* weights, float* partials, cudaStream_t stream) {
  const int warps = 8;
  if (T <= kSmallT) {
    const auto* xb = static_cast<const __nv_bfloat16*>(x);
    const auto* wb = static_cast<const __nv_bfloat16*>(w);
    const int t = static_cast<int>(T);
    if (T <= 4)
      router_logits_small_kernel<4><<<E, kSmallThreads, 0, stream>>>(xb, wb, t, H, E, partials);
    else if (T <= 8)
      router_logits_small_kernel<8><<<E, kSmallThreads, 0, stream>>>(xb, wb, t, H, E, partials);
    else if (T <= 16)
      router_logits_small_kernel<16><<<E, kSmallThreads, 0, stream>>>(xb, wb, t, H, E, partials);
    else
      router_logits_small_kernel<32><<<E, kSmallThreads, 0, stream>>>(xb, wb, t, H, E, partials);
    cudaError_t err = cudaGetLastError();
    if (err != cudaSuccess) return err;
    router_topk_kernel<<<static_cast<unsigned>((T + warps - 1) / warps), warps * 32, 0, stream>>>(
        partials, 1, T, E, k, mode, ids, weights);
    return cudaGetLastError();
  }
  if (T >= kMmaMinT && H % kMmaK == 0) {
    const auto* xb = static_cast<const __nv_bfloat16*>(x);
    const auto* wb = static_cast<const __nv_bfloat16*>(w);
    // column tile: all experts in one CTA, halved (down to 64 experts) while
    // the grid would leave SMs idle; x tiles are then re-read from L2
    const int nt_all = (E + 7) / 8;
    int nt = nt_all <= 2 ? 2 : nt_all <= 4 ? 4 : nt_all <= 6 ? 6 : nt_all <= 8 ? 8
           : nt_all <= 16 ? 16 : 32;
    const int64_t row_tiles = (T + kMmaRows - 1) / kMmaRows;
    while (nt > 8 && row_tiles * ((nt_all + nt - 1) / nt) < kSms) nt /= 2;
    const size_t smem =
        static_cast<size_t>(kMmaStages) * (kMmaRows + nt * 8) * kMmaStride * 2;
    const dim3 grid(static_cast<unsigned>(row_tiles),
                    static_cast<unsigned>((nt_all + nt - 1) / nt));
    auto run = [&](auto kernel) -> cudaError_t {
      if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(smem));
        if (e != cudaSuccess) return e;
      }
      kernel<<<grid, 256, smem, stream>>>(xb, wb, T, H, E, partials);
      return cudaGetLastError();
    };
    cudaError_t err = nt == 2 ? run(router_logits_mma_kernel<2>)
                    : nt == 4 ? run(router_logits_mma_kernel<4>)
                    : nt == 6 ? run(router_logits_mma_kernel<6>)
                    : nt == 8 ? run(router_logits_mma_kernel<8>)
                    : nt == 16 ? run(router_logits_mma_kernel<16>)
                               : run(router_logits_mma_kernel<32>);
    if (err != cudaSuccess) return err;
    router_topk_kernel<<<static_cast<unsigned>((T + warps - 1) / warps), warps * 32, 0, stream>>>(
        partials, 1, T, E, k, mode, ids, weights);
    return cudaGetLastError();
  }
  const int splits = splits_for(T, H);
  // K range per split: whole chunks
  const int chunks = H / kChunkK;
  const int k_per_split = ((chunks + splits - 1) / splits) * kChunkK;
  const int used = (H + k_per_split - 1) / k_per_split;
  const size_t smem = (kTokPerCta * kXStride + static_cast<size_t>(E) * kChunkK) * 2;
  dim3 grid(static_cast<unsigned>((T + kTokPerCta - 1) / kTokPerCta), used);
  auto run = [&](auto kernel) -> cudaError_t {
    if (smem > 48 * 1024) {
      cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(smem));
      if (e != cudaSuccess) return e;
    }
    kernel<<<grid, kRouterThreads, smem, stream>>>(
        static_cast<const __nv_bfloat16*>(x), static_cast<const __nv_bfloat16*>(w), T, H, E,
        k_per_split, partials);
    return cudaGetLastError();
  };
  const int per = (E + 7) / 8;
  cudaError_t err = per <= 2 ? run(router_logits_kernel<2>)
                  : per <= 4 ? run(router_logits_kernel<4>)
                  : per <= 6 ? run(router_logits_kernel<6>)
                  : per <= 8 ? run(router_logits_kernel<8>)
                  : per <= 16 ? run(router_logits_kernel<16>)
                              : run(router_logits_kernel<32>);
  if (err != cudaSuccess) return err;
  router_topk_kernel<<<static_cast<unsigned>((T + warps - 1) / warps), warps * 32, 0, stream>>>(
      partials, used, T, E, k, mode, ids, weights);
  return cudaGetLastError();
}

}  // namespace nvmoe
