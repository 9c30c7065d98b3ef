// Expert-parallel dispatch and combine: the data movement around the
// all-to-all exchanges when the E experts are split over G ranks (E/G
// consecutive experts per rank).  The pages treat the 48-expert layer as one
// tensor-parallel rank's share of a larger MoE ("NVFP4 MoE Debug Log
// (early)", Symptoms; Hypotheses section 7, the per-rank table); the
// exchange itself is a collective of the caller's communicator.
//
//   dispatch  each slot (t, j) goes to the rank owning expert topk_ids[t, j]:
//             the slot's quantised token row (H/2 bytes of E2M1 nibbles,
//             then H/16 row-major E4M3 scale bytes) and the expert's index
//             on that rank are packed at send_pos[t*k + j]; the rows for rank
//             d occupy [sum_{d'<d} counts[d'], ...) in ascending t*k + j.
//   scatter   received rows into the slot layout of the owner's forward
//             (nibbles to xq[slot_of[i]], scales to their staged offsets).
//   gather    the owner's slot outputs back into received-row order, for
//             the return exchange; the source then reduces the returned
//             rows with slot_of = send_pos (moe_unpermute_reduce).
#include <cuda_runtime.h>
#include <cstdint>

#include "internal.h"
#include "ptx.cuh"
#include "quant.cuh"

namespace nvmoe {

namespace {

// Destination rank of every slot: id / (E / G); an id outside [0, E) is
// recorded (bad index) and its slot sent nowhere (dest -1).
__global__ void ep_dest_kernel(const int32_t* __restrict__ ids, int64_t S, int E, int G,
                               int32_t* __restrict__ dest, int* status) {
  const int per = E / G;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < S;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int e = ids[i];
    if (e >= 0 && e < E) {
      dest[i] = e / per;
    } else {
      dest[i] = -1;
      record_status(status, kErrBadIndex);
    }
  }
}

// One warp per slot: the unpadded send position (the padded position from
// the counting sort by destination, minus the destination's padded offset,
// plus the exclusive prefix of the true counts), then the row and the local
// expert index.  row_bytes = H/2 + H/16 is a multiple of 16 (H % 256 == 0).
__global__ void ep_pack_kernel(const int32_t* __restrict__ ids, const int32_t* __restrict__ padded,
                               const int32_t* __restrict__ dest,
                               const int32_t* __restrict__ offsets,
                               const int32_t* __restrict__ counts, int64_t S, int k, int E, int G,
                               const uint8_t* __restrict__ q_tok,
                               const uint8_t* __restrict__ sf_tok, int H,
                               int32_t* __restrict__ send_pos, uint8_t* __restrict__ send_rows,
                               int32_t* __restrict__ send_expert) {
  __shared__ int s_prefix[kMaxExperts + 1];
  if (threadIdx.x == 0) {
    int p = 0;
    for (int d = 0; d < G; ++d) {
      s_prefix[d] = p;
      p += counts[d];
    }
    s_prefix[G] = p;
  }
  __syncthreads();
  const int lane = threadIdx.x & 31;
  const int warps = blockDim.x >> 5;
  const int per = E / G;
  const int qb = H / 2, sb = H / 16;
  const int64_t row_bytes = qb + sb;
  for (int64_t i = blockIdx.x * (int64_t)warps + (threadIdx.x >> 5); i < S;
       i += (int64_t)gridDim.x * warps) {
    const int d = dest[i];
    if (d < 0) {
      if (lane == 0) send_pos[i] = -1;
      continue;
    }
    const int64_t pos = padded[i] - offsets[d] + s_prefix[d];
    const int64_t t = i / k;
    if (lane == 0) {
      send_pos[i] = static_cast<int32_t>(pos);
      send_expert[pos] = ids[i] - d * per;
    }
    const uint4* qs = reinterpret_cast<const uint4*>(q_tok + t * qb);
    uint4* dst = reinterpret_cast<uint4*>(send_rows + pos * row_bytes);
    for (int c = lane; c < qb / 16; c += 32) dst[c] = qs[c];
    const uint4* ss = reinterpret_cast<const uint4*>(sf_tok + t * sb);
    uint4* dsf = reinterpret_cast<uint4*>(send_rows + pos * row_bytes + qb);
    for (int c = lane; c < sb / 16; c += 32) dsf[c] = ss[c];
  }
}

// One warp per received row: nibbles to xq[slot_of[i]], the H/16 scale
// bytes to their staged offsets (4 consecutive groups form one 32-bit word).
__global__ void ep_scatter_kernel(const uint8_t* __restrict__ rows, int64_t n, int H,
                                  const int32_t* __restrict__ slot_of, int64_t out_rows,
                                  uint8_t* __restrict__ xq, uint8_t* __restrict__ xsf,
                                  int k_atoms, int* status) {
  const int lane = threadIdx.x & 31;
  const int warps = blockDim.x >> 5;
  const int qb = H / 2, sb = H / 16;
  const int64_t row_bytes = qb + sb;
  for (int64_t i = blockIdx.x * (int64_t)warps + (threadIdx.x >> 5); i < n;
       i += (int64_t)gridDim.x * warps) {
    const int64_t r = slot_of[i];
    if (r < 0 || !NVMOE_BOUNDS(r < out_rows, status)) continue;
    const uint4* src = reinterpret_cast<const uint4*>(rows + i * row_bytes);
    uint4* dst = reinterpret_cast<uint4*>(xq + r * qb);
    for (int c = lane; c < qb / 16; c += 32) dst[c] = src[c];
    const uint32_t* s4 = reinterpret_cast<const uint32_t*>(rows + i * row_bytes + qb);
    for (int w = lane; w < sb / 4; w += 32)
      *reinterpret_cast<uint32_t*>(xsf + staged_offset(r, 4 * w, k_atoms)) = s4[w];
  }
}

// out[i] = slot_out[slot_of[i]] (row_bytes per row, a multiple of 16).
__global__ void ep_gather_kernel(const uint8_t* __restrict__ slot_out, int64_t row_bytes,
                                 int64_t slot_rows, const int32_t* __restrict__ slot_of, int64_t n,
                                 uint8_t* __restrict__ out, int* status) {
  const int lane = threadIdx.x & 31;
  const int warps = blockDim.x >> 5;
  for (int64_t i = blockIdx.x * (int64_t)warps + (threadIdx.x >> 5); i < n;
       i += (int64_t)gridDim.x * warps) {
    const int64_t r = slot_of[i];
    uint4* dst = reinterpret_cast<uint4*>(out + i * row_bytes);
    if (r < 0 || !NVMOE_BOUNDS(r < slot_rows, status)) {
      for (int c = lane; c < row_bytes / 16; c += 32) dst[c] = make_uint4(0u, 0u, 0u, 0u);
      continue;
    }
    const uint4* src = reinterpret_cast<const uint4*>(slot_out + r * row_bytes);
    for (int c = lane; c < row_bytes / 16; c += 32) dst[c] = src[c];
  }
}

// out[0] = max of partial[0..n) (non-negative values; 0 for n == 0).
__global__ void max_reduce_kernel(const float* __restrict__ partial, int n, float* out) {
  __shared__ float s[32];
  float m = 0.0f;
  for (int i = threadIdx.x; i < n; i += blockDim.x) m = fmaxf(m, __ldcg(partial + i));
  m = warp_max(m);
  if ((threadIdx.x & 31) == 0) s[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x < 32) {
    float r = threadIdx.x < (blockDim.x >> 5) ? s[threadIdx.x] : 0.0f;
    r = warp_max(r);
    if (threadIdx.x == 0) *out = r;
  }
}

constexpr int kEpThreads = 256;

int ep_blocks(int64_t items_per_warp_unit) {
  int64_t b = (items_per_warp_unit + (kEpThreads / 32) - 1) / (kEpThreads / 32);
  if (b > 152 * 8) b = 152 * 8;
  return static_cast<int>(b < 1 ? 1 : b);
}

}  // namespace

cudaError_t launch_ep_dest(const int32_t* ids, int64_t S, int E, int G, int32_t* dest, int* status,
                           cudaStream_t stream) {
  int64_t b = (S + kEpThreads - 1) / kEpThreads;
  if (b > 152 * 8) b = 152 * 8;
  ep_dest_kernel<<<static_cast<int>(b < 1 ? 1 : b), kEpThreads, 0, stream>>>(ids, S, E, G, dest,
                                                                            status);
  return cudaGetLastError();
}

cudaError_t launch_ep_pack(const int32_t* ids, const int32_t* padded, const int32_t* dest,
                           const int32_t* offsets, const int32_t* counts, int64_t S, int k, int E,
                           int G, const uint8_t* q_tok, const uint8_t* sf_tok, int H,
                           int32_t* send_pos, uint8_t* send_rows, int32_t* send_expert,
                           cudaStream_t stream) {
  ep_pack_kernel<<<ep_blocks(S), kEpThreads, 0, stream>>>(ids, padded, dest, offsets, counts, S, k,
                                                         E, G, q_tok, sf_tok, H, send_pos,
                                                         send_rows, send_expert);
  return cudaGetLastError();
}

cudaError_t launch_ep_scatter(const uint8_t* rows, int64_t n, int H, const int32_t* slot_of,
                              int64_t out_rows, uint8_t* xq, uint8_t* xsf, int k_atoms,
                              int* status, cudaStream_t stream) {
  ep_scatter_kernel<<<ep_blocks(n), kEpThreads, 0, stream>>>(rows, n, H, slot_of, out_rows, xq,
                                                            xsf, k_atoms, status);
  return cudaGetLastError();
}

cudaError_t launch_ep_gather(const void* slot_out, int64_t row_bytes, int64_t slot_rows,
                             const int32_t* slot_of, int64_t n, void* out, int* status,
                             cudaStream_t stream) {
  ep_gather_kernel<<<ep_blocks(n), kEpThreads, 0, stream>>>(
      static_cast<const uint8_t*>(slot_out), row_bytes, slot_rows, slot_of, n,
      static_cast<uint8_t*>(out), status);
  return cudaGetLastError();
}

cudaError_t launch_max_reduce(const float* partial, int n, float* out, cudaStream_t stream) {
  max_reduce_kernel<<<1, 1024, 0, stream>>>(partial, n, out);
  return cudaGetLastError();
}

}  // namespace nvmoe
