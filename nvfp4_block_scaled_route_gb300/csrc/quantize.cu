// Dynamic NVFP4 quantisation (activations, the SiLU*up intermediate, and
// offline fp32 weights).
//
// Arithmetic ("NVFP4 MegaMoE Debug Log", Hypotheses §6 steps 1-5; commit
// message "Three bugs fixed" on src), IEEE fp32 round-to-nearest-even:
//   gs = amax / 2688 (1 if amax == 0); per 16-element block b = max|v|,
//   sf = E4M3_satfinite(b / (6 gs)), d = dec(sf) * gs,
//   nibble = E2M1_satfinite(|v| / d) | sign(v) << 3   (0 when d == 0),
//   element 2j -> low nibble, 2j+1 -> high nibble.
// Pass 1 (amax) writes per-CTA maxima; pass 2 reduces them in every CTA
// (no atomics, no memset) and streams the quantisation with 16-byte loads,
// one thread per 16-element block.
#include <cuda_bf16.h>

#include "internal.h"
#include "ptx.cuh"
#include "quant.cuh"

namespace nvmoe {

namespace {

constexpr int kAmaxThreads = 256;
constexpr int kPackThreads = 256;

template <typename T>
struct Vec;  // 16-byte vector of T

template <>
struct Vec<__nv_bfloat16> {
  static constexpr int kElems = 8;
  __device__ static void load(const __nv_bfloat16* p, float (&v)[8]) {
    uint4 u = __ldg(reinterpret_cast<const uint4*>(p));
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      v[2 * i] = __uint_as_float(w[i] << 16);
      v[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
  }
};

template <>
struct Vec<float> {
  static constexpr int kElems = 4;
  __device__ static void load(const float* p, float (&v)[4]) {
    float4 u = __ldg(reinterpret_cast<const float4*>(p));
    v[0] = u.x; v[1] = u.y; v[2] = u.z; v[3] = u.w;
  }
};

template <typename T>
__global__ void __launch_bounds__(kAmaxThreads) quant_amax_kernel(const T* __restrict__ x,
                                                                   int64_t n_vec,
                                                                   float* __restrict__ partial) {
  pdl_trigger();
  pdl_wait();
  constexpr int VE = Vec<T>::kElems;
  float m = 0.0f;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n_vec;
       i += (int64_t)gridDim.x * blockDim.x) {
    float v[VE];
    Vec<T>::load(x + i * VE, v);
#pragma unroll
    for (int j = 0; j < VE; ++j) m = fmaxf(m, fabsf(v[j]));
  }
  __shared__ float s[kAmaxThreads / 32];
  m = warp_max(m);
  if ((threadIdx.x & 31) == 0) s[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x < 32) {
    float r = threadIdx.x < kAmaxThreads / 32 ? s[threadIdx.x] : 0.0f;
    r = warp_max(r);
    if (threadIdx.x == 0) partial[blockIdx.x] = r;
  }
}

// Quantise rows of x given gs: one thread per 16-element block, a
// warp-uniform grid-stride loop so that the shuffles always see all 32 lanes.
template <typename T>
__device__ __forceinline__ void pack_rows(const T* __restrict__ x, int64_t rows, int cols,
                                          const int32_t* __restrict__ row_dst, int fanout,
                                          const int32_t* __restrict__ row_valid, float gs,
                                          uint8_t* __restrict__ q, uint8_t* __restrict__ sf_row,
                                          uint8_t* __restrict__ sf_mma, int k_atoms,
                                          int64_t out_rows, int* status) {
  constexpr int VE = Vec<T>::kElems;
  const float denom = __fmul_rn(6.0f, gs);
  const int bpr = cols >> 4;                       // blocks per row
  const int64_t total = rows * bpr;
  const int lane = threadIdx.x & 31;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t base = blockIdx.x * (int64_t)blockDim.x + (threadIdx.x & ~31); base < total;
       base += stride) {
    const int64_t i = base + lane;
    const bool active = i < total;
    const int64_t row = active ? i / bpr : 0;
    const int g = active ? static_cast<int>(i - row * bpr) : 0;
    bool valid = active && (row_valid == nullptr || row_valid[row] >= 0);
    float v[16];
    if (valid) {
      const T* src = x + row * cols + (int64_t)g * 16;
#pragma unroll
      for (int c = 0; c < 16 / VE; ++c) {
        float t[VE];
        Vec<T>::load(src + c * VE, t);
#pragma unroll
        for (int j = 0; j < VE; ++j) v[c * VE + j] = t[j];
      }
    } else {
#pragma unroll
      for (int j = 0; j < 16; ++j) v[j] = 0.0f;
    }
    uint32_t packed[2];
    const uint32_t sf = quant_block16(v, gs, denom, packed);
    // gather the 4 scale bytes of one staged 32-bit word (groups g..g+3)
    const uint32_t s1 = __shfl_down_sync(0xFFFFFFFFu, sf, 1);
    const uint32_t s2 = __shfl_down_sync(0xFFFFFFFFu, sf, 2);
    const uint32_t s3 = __shfl_down_sync(0xFFFFFFFFu, sf, 3);
    const uint32_t word = sf | (s1 << 8) | (s2 << 16) | (s3 << 24);
    if (!valid) continue;
    for (int j = 0; j < fanout; ++j) {
      const int64_t dst = row_dst != nullptr ? row_dst[row * fanout + j] : row;
      if (dst < 0 || !NVMOE_BOUNDS(dst < out_rows, status)) continue;
      *reinterpret_cast<uint2*>(q + dst * (cols >> 1) + (int64_t)g * 8) =
          make_uint2(packed[0], packed[1]);
      if (sf_row != nullptr) sf_row[dst * bpr + g] = static_cast<uint8_t>(sf);
      if (sf_mma != nullptr && (g & 3) == 0)
        *reinterpret_cast<uint32_t*>(sf_mma + staged_offset(dst, g, k_atoms)) = word;
    }
  }
}

template <typename T>
__global__ void __launch_bounds__(kPackThreads) quant_pack_kernel(
    const T* __restrict__ x, int64_t rows, int cols, const int32_t* __restrict__ row_dst,
    int fanout, const int32_t* __restrict__ row_valid, const float* __restrict__ partial,
    int n_partial, uint8_t* __restrict__ q, uint8_t* __restrict__ sf_row,
    uint8_t* __restrict__ sf_mma, float* __restrict__ gs_out, int k_atoms, int64_t out_rows,
    int* status) {
  pdl_trigger();
  pdl_wait();
  __shared__ float s_gs;
  if (threadIdx.x < 32) {
    const float amax = reduce_partials(partial, n_partial);
    if (threadIdx.x == 0) {
      const float gs = global_scale_from(amax);
      s_gs = gs;
      if (blockIdx.x == 0 && gs_out != nullptr) *gs_out = gs;
    }
  }
  __syncthreads();
  pack_rows<T>(x, rows, cols, row_dst, fanout, row_valid, s_gs, q, sf_row, sf_mma, k_atoms,
               out_rows, status);
}

// Small inputs: amax and quantisation in one CTA (one launch instead of two).
constexpr int kSmallThreads = 1024;

template <typename T>
__global__ void __launch_bounds__(kSmallThreads) quant_small_kernel(
    const T* __restrict__ x, int64_t rows, int cols, const int32_t* __restrict__ row_dst,
    int fanout, uint8_t* __restrict__ q, uint8_t* __restrict__ sf_row,
    uint8_t* __restrict__ sf_mma, float* __restrict__ gs_out, int k_atoms, int64_t out_rows,
    int* status) {
  pdl_trigger();
  pdl_wait();
  constexpr int VE = Vec<T>::kElems;
  __shared__ float s_red[kSmallThreads / 32];
  __shared__ float s_gs;
  const int64_t n_vec = rows * cols / VE;
  float m = 0.0f;
  for (int64_t i = threadIdx.x; i < n_vec; i += blockDim.x) {
    float v[VE];
    Vec<T>::load(x + i * VE, v);
#pragma unroll
    for (int j = 0; j < VE; ++j) m = fmaxf(m, fabsf(v[j]));
  }
  m = warp_max(m);
  if ((threadIdx.x & 31) == 0) s_red[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x < 32) {
    const float r = warp_max(s_red[threadIdx.x]);
    if (threadIdx.x == 0) {
      const float gs = global_scale_from(r);
      s_gs = gs;
      if (gs_out != nullptr) *gs_out = gs;
    }
  }
  __syncthreads();
  pack_rows<T>(x, rows, cols, row_dst, fanout, nullptr, s_gs, q, sf_row, sf_mma, k_atoms, out_rows,
               status);
}

// ------------------------------------------------------------- weights ----
// Per-expert amax: grid (parts, E).
__global__ void __launch_bounds__(kAmaxThreads) weight_amax_kernel(const float* __restrict__ w,
                                                                    int64_t per_expert_vec,
                                                                    float* __restrict__ partial) {
  const int e = blockIdx.y;
  const float* base = w + static_cast<int64_t>(e) * per_expert_vec * 4;
  float m = 0.0f;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < per_expert_vec;
       i += (int64_t)gridDim.x * blockDim.x) {
    float v[4];
    Vec<float>::load(base + i * 4, v);
#pragma unroll
    for (int j = 0; j < 4; ++j) m = fmaxf(m, fabsf(v[j]));
  }
  __shared__ float s[kAmaxThreads / 32];
  m = warp_max(m);
  if ((threadIdx.x & 31) == 0) s[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x < 32) {
    float r = threadIdx.x < kAmaxThreads / 32 ? s[threadIdx.x] : 0.0f;
    r = warp_max(r);
    if (threadIdx.x == 0) partial[e * gridDim.x + blockIdx.x] = r;
  }
}

// One thread per (expert, 16-row block of K, column n): reads 16 values
// down a column (coalesced across n), writes 8 packed bytes down the
// column of q (K/2, N) and one scale byte of sf (K/16, N).
__global__ void __launch_bounds__(kPackThreads) weight_quant_kernel(
    const float* __restrict__ w, int K, int N, const float* __restrict__ partial, int parts,
    uint8_t* __restrict__ q, uint8_t* __restrict__ sf, float* __restrict__ gs_out) {
  const int e = blockIdx.z;
  __shared__ float s_gs;
  if (threadIdx.x < 32) {
    const float amax = reduce_partials(partial + e * parts, parts);
    if (threadIdx.x == 0) {
      const float gs = global_scale_from(amax);
      s_gs = gs;
      if (blockIdx.x == 0 && blockIdx.y == 0) gs_out[e] = gs;
    }
  }
  __syncthreads();
  const float gs = s_gs;
  const float denom = __fmul_rn(6.0f, gs);
  const int n = blockIdx.x * blockDim.x + threadIdx.x;
  const int kb = blockIdx.y;
  if (n >= N) return;
  const float* src = w + (static_cast<int64_t>(e) * K + kb * 16) * N + n;
  float v[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __ldg(src + static_cast<int64_t>(i) * N);
  uint32_t packed[2];
  const uint32_t s = quant_block16(v, gs, denom, packed);
  uint8_t* qd = q + (static_cast<int64_t>(e) * (K / 2) + kb * 8) * N + n;
#pragma unroll
  for (int p = 0; p < 8; ++p)
    qd[static_cast<int64_t>(p) * N] = static_cast<uint8_t>(packed[p >> 2] >> (8 * (p & 3)));
  sf[(static_cast<int64_t>(e) * (K / 16) + kb) * N + n] = static_cast<uint8_t>(s);
}

// Checkpoint (K/2, N) bytes of expert e -> B-operand tiles: row n of the
// (E*N, K) matrix, K-stage kt (128 bytes) lives in the contiguous 16 KB tile
// ((n_global / 128) * KT + kt), at row n % 128.  Bytes past K/2 are zero.
// 32x32 byte tiles through shared memory.
__global__ void tile_weight_bytes_kernel(const uint8_t* __restrict__ src, int R, int C, int KT,
                                         uint8_t* __restrict__ dst) {
  // src: [E][R = K/2][C = N];  grid.y covers the padded R (KT * 128)
  __shared__ uint8_t tile[32][33];
  const int e = blockIdx.z;
  const int c0 = blockIdx.x * 32, r0 = blockIdx.y * 32;
  const uint8_t* s = src + static_cast<int64_t>(e) * R * C;
  for (int i = threadIdx.y; i < 32; i += blockDim.y) {
    const int r = r0 + i, c = c0 + threadIdx.x;
    if (c < C) tile[i][threadIdx.x] = r < R ? s[static_cast<int64_t>(r) * C + c] : 0;
  }
  __syncthreads();
  for (int i = threadIdx.y; i < 32; i += blockDim.y) {
    const int c = c0 + i, r = r0 + threadIdx.x;
    if (c >= C) continue;
    const int64_t n = static_cast<int64_t>(e) * C + c;
    const int64_t off = ((n / kTileRows) * KT + r / 128) * (kTileRows * 128) +
                        (n % kTileRows) * 128 + (r % 128);
    dst[off] = tile[threadIdx.x][i];
  }
}

// Checkpoint scales (K/16, N) of expert e -> staged layout of the (E*N, K)
// matrix (row = e*N + n, group g).
__global__ void stage_weight_sf_kernel(const uint8_t* __restrict__ sf_ckpt, int K, int N,
                                       int k_atoms, uint8_t* __restrict__ sf_out) {
  const int e = blockIdx.z;
  const int g = blockIdx.y;
  const int n = blockIdx.x * blockDim.x + threadIdx.x;
  if (n >= N) return;
  const uint8_t v = sf_ckpt[(static_cast<int64_t>(e) * (K / 16) + g) * N + n];
  sf_out[staged_offset(static_cast<int64_t>(e) * N + n, g, k_atoms)] = v;
}

}  // namespace

int quant_amax_blocks(int64_t n_elems) {
  const int64_t n_vec = n_elems / 4;  // conservative (fp32 vectors)
  int64_t b = ceil_div(n_vec, static_cast<int64_t>(kAmaxThreads) * 8);
  if (b < 1) b = 1;
  if (b > kQuantMaxPartials) b = kQuantMaxPartials;
  return static_cast<int>(b);
}

cudaError_t launch_quant_amax(const void* x, int x_dtype, int64_t n_elems, float* partial,
                              int n_partial, cudaStream_t stream) {
  if (x_dtype == 0) {
    (void)launch_pdl(quant_amax_kernel<__nv_bfloat16>, dim3(n_partial), dim3(kAmaxThreads), 0, stream, 
        static_cast<const __nv_bfloat16*>(x), n_elems / 8, partial);
  } else {
    (void)launch_pdl(quant_amax_kernel<float>, dim3(n_partial), dim3(kAmaxThreads), 0, stream, 
        static_cast<const float*>(x), n_elems / 4, partial);
  }
  return cudaGetLastError();
}

cudaError_t launch_quant_small(const void* x, int x_dtype, int64_t rows, int64_t cols,
                               const int32_t* row_dst, int fanout, uint8_t* q, uint8_t* sf_row,
                               uint8_t* sf_mma, float* gs_out, int64_t out_rows, int* status,
                               cudaStream_t stream) {
  const int k_atoms = static_cast<int>(round_up(cols, kStageK) / 64);
  if (x_dtype == 0)
    (void)launch_pdl(quant_small_kernel<__nv_bfloat16>, dim3(1), dim3(kSmallThreads), 0, stream, 
        static_cast<const __nv_bfloat16*>(x), rows, static_cast<int>(cols), row_dst, fanout, q,
        sf_row, sf_mma, gs_out, k_atoms, out_rows, status);
  else
    (void)launch_pdl(quant_small_kernel<float>, dim3(1), dim3(kSmallThreads), 0, stream, 
        static_cast<const float*>(x), rows, static_cast<int>(cols), row_dst, fanout, q, sf_row,
        sf_mma, gs_out, k_atoms, out_rows, status);
  return cudaGetLastError();
}

cudaError_t launch_quant_pack(const void* x, int x_dtype, int64_t rows, int64_t cols,
                              const int32_t* row_dst, int fanout, const int32_t* row_valid,
                              const float* partial, int n_partial, uint8_t* q, uint8_t* sf_row,
                              uint8_t* sf_mma, float* gs_out, int64_t out_rows, int* status,
                              cudaStream_t stream) {
  const int64_t total = rows * (cols / 16);
  int64_t blocks = ceil_div(total, kPackThreads);
  const int64_t cap = 152 * 16;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  const int k_atoms = static_cast<int>(round_up(cols, kStageK) / 64);
  if (x_dtype == 0) {
    (void)launch_pdl(quant_pack_kernel<__nv_bfloat16>, dim3(static_cast<int>(blocks)), dim3(kPackThreads), 0, stream, 
        static_cast<const __nv_bfloat16*>(x), rows, static_cast<int>(cols), row_dst, fanout,
        row_valid, partial, n_partial, q, sf_row, sf_mma, gs_out, k_atoms, out_rows, status);
  } else {
    (void)launch_pdl(quant_pack_kernel<float>, dim3(static_cast<int>(blocks)), dim3(kPackThreads), 0, stream, 
        static_cast<const float*>(x), rows, static_cast<int>(cols), row_dst, fanout, row_valid,
        partial, n_partial, q, sf_row, sf_mma, gs_out, k_atoms, out_rows, status);
  }
  return cudaGetLastError();
}

// Row-major activation scales [rows, cols/16] -> the staged layout, one CTA
// per 128-row tile.  Atom kb of tile mt holds in its 16-byte row i the four
// scale bytes of k-block kb of rows 32j + i (j = 0..3, word j); a lane reads
// the 16 bytes of four k-blocks of its four rows and writes one 16-byte atom
// row per k-block, so every load and store is a full 16 bytes and a warp's
// stores cover whole 512-byte atoms.  Rows at or past `rows` read as zero.
// (The quantiser's own staged writes are 4-byte words whose sectors are
// completed by other tokens' rows much later; this pass replaces them.)
__global__ void __launch_bounds__(kPackThreads) stage_act_sf_kernel(
    const uint8_t* __restrict__ sf_row, int64_t rows, int bpr, uint8_t* __restrict__ sf_mma,
    int k_atoms) {
  pdl_trigger();
  pdl_wait();
  const int64_t mt = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_quads = bpr / 16;
  for (int c = warp; c < n_quads; c += kPackThreads / 32) {
    uint32_t v[4][4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int64_t r = mt * kTileRows + 32 * j + lane;
      uint4 u = make_uint4(0u, 0u, 0u, 0u);
      if (r < rows) u = __ldg(reinterpret_cast<const uint4*>(sf_row + r * bpr) + c);
      v[j][0] = u.x; v[j][1] = u.y; v[j][2] = u.z; v[j][3] = u.w;
    }
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      uint4* dst = reinterpret_cast<uint4*>(
          sf_mma + (static_cast<size_t>(mt) * k_atoms + 4 * c + w) * kSfAtomBytes) + lane;
      *dst = make_uint4(v[0][w], v[1][w], v[2][w], v[3][w]);
    }
  }
}

cudaError_t launch_stage_act_sf(const uint8_t* sf_row, int64_t rows, int64_t cols,
                                uint8_t* sf_mma, cudaStream_t stream) {
  const int64_t tiles = ceil_div(rows, kTileRows);
  if (tiles == 0) return cudaSuccess;
  const int k_atoms = static_cast<int>(round_up(cols, kStageK) / 64);
  (void)launch_pdl(stage_act_sf_kernel, dim3(static_cast<unsigned>(tiles)), dim3(kPackThreads), 0,
                   stream, sf_row, rows, static_cast<int>(cols / 16), sf_mma, k_atoms);
  return cudaGetLastError();
}

cudaError_t launch_weight_amax(const float* w, int E, int64_t per_expert, float* partial,
                               int parts_per_expert, cudaStream_t stream) {
  dim3 grid(parts_per_expert, E);
  weight_amax_kernel<<<grid, kAmaxThreads, 0, stream>>>(w, per_expert / 4, partial);
  return cudaGetLastError();
}

cudaError_t launch_weight_quant(const float* w, int E, int K, int N, const float* partial,
                                int parts_per_expert, uint8_t* q, uint8_t* sf, float* gs,
                                cudaStream_t stream) {
  dim3 grid(static_cast<unsigned>(ceil_div(N, kPackThreads)), K / 16, E);
  weight_quant_kernel<<<grid, kPackThreads, 0, stream>>>(w, K, N, partial, parts_per_expert, q,
                                                         sf, gs);
  return cudaGetLastError();
}

cudaError_t launch_prepare_weights(const uint8_t* q_ckpt, const uint8_t* sf_ckpt, int E, int K,
                                   int N, uint8_t* q_out, uint8_t* sf_out, cudaStream_t stream) {
  const int KT = static_cast<int>(ceil_div(K, kStageK));
  dim3 tgrid(static_cast<unsigned>(ceil_div(N, 32)), static_cast<unsigned>(KT * 4), E);
  tile_weight_bytes_kernel<<<tgrid, dim3(32, 8), 0, stream>>>(q_ckpt, K / 2, N, KT, q_out);
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  const int k_atoms = static_cast<int>(round_up(K, kStageK) / 64);
  dim3 sgrid(static_cast<unsigned>(ceil_div(N, 256)), K / 16, E);
  stage_weight_sf_kernel<<<sgrid, 256, 0, stream>>>(sf_ckpt, K, N, k_atoms, sf_out);
  return cudaGetLastError();
}

}  // namespace nvmoe
