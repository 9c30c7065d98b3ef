// Top-k routing permutation ("NVFP4 MegaMoE Debug Log", Pipeline Trace: the
// per-expert slot counts of the grouped GEMM; NVFP4 MoE Pipeline, the
// grouped layout the L1/L2 GEMMs run over): per-expert histogram, prefix sum
// over experts with 128-row aligned segments, and a stable slot assignment
// (ascending flat index t*k + j within an expert).  Deterministic: counts come from
// per-chunk histograms, ranks from warp match + per-warp counts; no global
// atomics decide any position.
#include "internal.h"
#include "ptx.cuh"

namespace nvmoe {

namespace {

constexpr int kRouteThreads = 1024;
constexpr int kWarps = kRouteThreads / 32;
constexpr int kPerWarp = 128;                       // elements per warp
constexpr int kChunk = kWarps * kPerWarp;           // 4096 elements per CTA
constexpr int kRounds = kPerWarp / 32;

__global__ void __launch_bounds__(kRouteThreads) route_count_kernel(
    const int32_t* __restrict__ ids, int64_t S, int E, int32_t* __restrict__ chunk_counts,
    int32_t* __restrict__ row_token, int64_t rows_bound, int* status) {
  pdl_trigger();
  pdl_wait();
  __shared__ int hist[kMaxExperts];
  for (int e = threadIdx.x; e < E; e += blockDim.x) hist[e] = 0;
  __syncthreads();
  const int64_t c0 = static_cast<int64_t>(blockIdx.x) * kChunk;
  for (int i = threadIdx.x; i < kChunk; i += blockDim.x) {
    const int64_t idx = c0 + i;
    if (idx >= S) break;
    const int e = ids[idx];
    if (e >= 0 && e < E) {
      atomicAdd(&hist[e], 1);
    } else {
      record_status(status, kErrBadIndex);
    }
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x)
    chunk_counts[static_cast<int64_t>(blockIdx.x) * E + e] = hist[e];
  // mark every row as padding; the assign pass overwrites the slots in use
  for (int64_t r = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; r < rows_bound;
       r += (int64_t)gridDim.x * blockDim.x)
    row_token[r] = -1;
}

__global__ void __launch_bounds__(kRouteThreads) route_assign_kernel(
    const int32_t* __restrict__ ids, int64_t S, int k, int E,
    const int32_t* __restrict__ chunk_counts, int n_chunks, int32_t* __restrict__ expert_offsets,
    int32_t* __restrict__ expert_counts, int32_t* __restrict__ row_token,
    int32_t* __restrict__ slot_of, int64_t rows_bound, int* status) {
  pdl_trigger();
  pdl_wait();
  __shared__ int base[kMaxExperts];        // first row of this chunk's slots per expert
  __shared__ int total[kMaxExperts];
  __shared__ int whist[kWarps][kMaxExperts];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (chunk_counts == nullptr) {
    // single CTA (S <= one chunk): histogram here, no counting launch
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
      total[e] = 0;
      base[e] = 0;
    }
    for (int64_t r = threadIdx.x; r < rows_bound; r += blockDim.x) row_token[r] = -1;
    __syncthreads();
    for (int64_t i = threadIdx.x; i < S; i += blockDim.x) {
      const int e = ids[i];
      if (e >= 0 && e < E)
        atomicAdd(&total[e], 1);
      else
        record_status(status, kErrBadIndex);
    }
  } else {
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
      int tot = 0, pre = 0;
      for (int c = 0; c < n_chunks; ++c) {
        const int v = chunk_counts[static_cast<int64_t>(c) * E + e];
        tot += v;
        if (c < static_cast<int>(blockIdx.x)) pre += v;
      }
      total[e] = tot;
      base[e] = pre;
    }
  }
  for (int i = threadIdx.x; i < kWarps * kMaxExperts; i += blockDim.x)
    (&whist[0][0])[i] = 0;
  __syncthreads();
  if (threadIdx.x == 0) {
    int off = 0;
    for (int e = 0; e < E; ++e) {
      const int t = total[e];
      if (blockIdx.x == 0) {
        expert_offsets[e] = off;
        expert_counts[e] = t;
      }
      base[e] += off;
      off += (t + kTileRows - 1) / kTileRows * kTileRows;
    }
    if (blockIdx.x == 0) expert_offsets[E] = off;
  }
  __syncthreads();

  // pass 1: rank of each element among equal experts inside its warp's range
  const int64_t w0 = static_cast<int64_t>(blockIdx.x) * kChunk + warp * kPerWarp;
  int my_e[kRounds], my_pos[kRounds];
  const unsigned lt_mask = (1u << lane) - 1u;
#pragma unroll
  for (int r = 0; r < kRounds; ++r) {
    const int64_t idx = w0 + r * 32 + lane;
    int e = -1;
    if (idx < S) {
      e = ids[idx];
      if (e < 0 || e >= E) e = -1;
    }
    const unsigned peers = __match_any_sync(0xFFFFFFFFu, e);
    const int rank = __popc(peers & lt_mask);
    int before = 0;
    if (e >= 0) before = whist[warp][e];
    __syncwarp();
    const bool last = (peers >> lane) == 1u;       // highest lane of its group
    if (e >= 0 && last) whist[warp][e] = before + rank + 1;
    __syncwarp();
    my_e[r] = e;
    my_pos[r] = before + rank;
  }
  __syncthreads();
  // exclusive prefix over warps, per expert
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int run = 0;
    for (int w = 0; w < kWarps; ++w) {
      const int v = whist[w][e];
      whist[w][e] = run;
      run += v;
    }
  }
  __syncthreads();
#pragma unroll
  for (int r = 0; r < kRounds; ++r) {
    const int64_t idx = w0 + r * 32 + lane;
    if (idx >= S) continue;
    const int e = my_e[r];
    if (e < 0) {
      slot_of[idx] = -1;
      continue;
    }
    const int row = base[e] + whist[warp][e] + my_pos[r];
    if (!NVMOE_BOUNDS(row >= 0 && row < rows_bound, status)) {
      slot_of[idx] = -1;
      continue;
    }
    slot_of[idx] = row;
    row_token[row] = static_cast<int32_t>(idx / k);
  }
}

}  // namespace

int route_chunk_elems() { return kChunk; }

cudaError_t launch_route(const int32_t* topk_ids, int64_t T, int k, int E,
                         int32_t* expert_offsets, int32_t* expert_counts, int32_t* row_token,
                         int64_t rows_bound, int32_t* slot_of, int32_t* chunk_counts,
                         int n_chunks, int* status, cudaStream_t stream) {
  const int64_t S = T * k;
  if (n_chunks == 1) {
    // one chunk: histogram, prefix sum and assignment in a single CTA
    (void)launch_pdl(route_assign_kernel, dim3(1), dim3(kRouteThreads), 0, stream, topk_ids, S, k, E, nullptr, 1,
                                                         expert_offsets, expert_counts,
                                                         row_token, slot_of, rows_bound, status);
    return cudaGetLastError();
  }
  (void)launch_pdl(route_count_kernel, dim3(n_chunks), dim3(kRouteThreads), 0, stream, topk_ids, S, E, chunk_counts,
                                                             row_token, rows_bound, status);
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  (void)launch_pdl(route_assign_kernel, dim3(n_chunks), dim3(kRouteThreads), 0, stream, 
      topk_ids, S, k, E, chunk_counts, n_chunks, expert_offsets, expert_counts, row_token,
      slot_of, rows_bound, status);
  return cudaGetLastError();
}

}  // namespace nvmoe

// ------------------------------------------------------------- no-alloc ----
// Routing without a caller workspace: the per-chunk histograms go to a fixed
// array in this library (every GPU that loads it holds the array until the
// process exits).  Host code cannot use the array's name as a device address,
// so the address is looked up once per device with cudaGetSymbolAddress.
#include <mutex>

#include "nvfp4moe.h"

namespace {

static __device__ __align__(256) int32_t g_noalloc_route_counts[NVMOE_NOALLOC_ROUTE_WORDS];

constexpr int kNoAllocMaxDevices = 64;
std::mutex g_noalloc_mu;
int32_t* g_noalloc_ptr[kNoAllocMaxDevices] = {};

// Device address of the array on the current device (looked up on first use).
int noalloc_counts(int32_t** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kNoAllocMaxDevices)
    return NVMOE_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (g_noalloc_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_route_counts) != cudaSuccess || p == nullptr)
      return NVMOE_ERR_CUDA;
    g_noalloc_ptr[dev] = static_cast<int32_t*>(p);
  }
  *out = g_noalloc_ptr[dev];
  return NVMOE_OK;
}

}  // namespace

extern "C" int moe_route_permute_noalloc(const int32_t* topk_ids, int64_t T, int k, int E,
                                         int32_t* expert_offsets, int32_t* expert_counts,
                                         int32_t* row_token, int32_t* slot_of,
                                         cudaStream_t stream) {
  using namespace nvmoe;
  if (T < 0 || k < 1 || k > kMaxTopK || E < 1 || E > kMaxExperts) return NVMOE_ERR_INVALID_ARG;
  // T*k < 2^31, tested without forming the product (T may be any int64)
  if (T > int64_t{INT32_MAX} / k) return NVMOE_ERR_UNSUPPORTED_SHAPE;
  if (expert_offsets == nullptr || expert_counts == nullptr) return NVMOE_ERR_INVALID_ARG;
  if (T > 0 && (topk_ids == nullptr || row_token == nullptr || slot_of == nullptr))
    return NVMOE_ERR_INVALID_ARG;
  const int64_t S = T * k;
  const int64_t n_chunks = S > 0 ? ceil_div(S, kChunk) : 1;
  if (n_chunks * E > NVMOE_NOALLOC_ROUTE_WORDS) return NVMOE_ERR_UNSUPPORTED_SHAPE;
  int32_t* counts = nullptr;
  const int st = noalloc_counts(&counts);
  if (st != NVMOE_OK) return st;
  // every word a launch reads is written by the same launch's counting pass
  // (one chunk needs no histogram words at all), so nothing is cleared here
  const int64_t S_pad = S + (S < E ? S : E) * (kTileRows - 1);
  const int64_t rows = (S_pad + kTileRows - 1) / kTileRows * kTileRows;
  const cudaError_t e = launch_route(topk_ids, T, k, E, expert_offsets, expert_counts, row_token,
                                     rows, slot_of, counts, static_cast<int>(n_chunks), nullptr,
                                     stream);
  if (e != cudaSuccess) return NVMOE_ERR_CUDA;
  note_launches(n_chunks == 1 ? 1 : 2);
  return NVMOE_OK;
}
