// Top-k weighted gather-reduce back to token order ("NVFP4 MegaMoE Debug
// Log", NVFP4 MoE Pipeline: the scatter of the L2 outputs with the routing
// weights):
//   y[t, :] = sum_{j ascending} w[t, j] * slot_out[slot_of[t*k + j], :]
// fp32 accumulation in a fixed order (deterministic), one store per element;
// slot_out in fp32, bf16 or fp16 (both widen exactly).
// Grid: (H/4 / threads, T); each thread owns 4 consecutive columns and reads
// k 16-byte vectors.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "internal.h"
#include "ptx.cuh"

namespace nvmoe {

namespace {

constexpr int kReduceThreads = 128;

// Four consecutive slot-output values as fp32 (bf16 widens exactly).
__device__ __forceinline__ float4 load4(const float* p) { return __ldcs(reinterpret_cast<const float4*>(p)); }
__device__ __forceinline__ float4 load4(const __nv_bfloat16* p) {
  const uint2 u = __ldcs(reinterpret_cast<const uint2*>(p));
  return make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xFFFF0000u),
                     __uint_as_float(u.y << 16), __uint_as_float(u.y & 0xFFFF0000u));
}

__device__ __forceinline__ float4 load4(const __half* p) {
  const uint2 u = __ldcs(reinterpret_cast<const uint2*>(p));
  const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&u.x));
  const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&u.y));
  return make_float4(a.x, a.y, b.x, b.y);
}

template <typename TIn, bool kBf16>
__global__ void __launch_bounds__(kReduceThreads) unpermute_reduce_kernel(
    const TIn* __restrict__ slot_out, const int32_t* __restrict__ slot_of,
    const float* __restrict__ topk_w, int64_t T, int k, int64_t H, void* __restrict__ y) {
  pdl_trigger();
  pdl_wait();
  __shared__ int s_slot[kMaxTopK];
  __shared__ float s_w[kMaxTopK];
  const int64_t c = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) * 4;
  for (int64_t t = blockIdx.y; t < T; t += gridDim.y) {
  __syncthreads();
  if (threadIdx.x < k) {
    s_slot[threadIdx.x] = slot_of[t * k + threadIdx.x];
    s_w[threadIdx.x] = topk_w[t * k + threadIdx.x];
  }
  __syncthreads();
  if (c >= H) continue;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int j = 0; j < k; ++j) {
    const int s = s_slot[j];
    if (s < 0) continue;
    const float w = s_w[j];
    const float4 v = load4(slot_out + s * H + c);
    acc.x = __fmaf_rn(w, v.x, acc.x);
    acc.y = __fmaf_rn(w, v.y, acc.y);
    acc.z = __fmaf_rn(w, v.z, acc.z);
    acc.w = __fmaf_rn(w, v.w, acc.w);
  }
  if (kBf16) {
    __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y);
    __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z, acc.w);
    uint2 out;
    out.x = *reinterpret_cast<uint32_t*>(&lo);
    out.y = *reinterpret_cast<uint32_t*>(&hi);
    *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(y) + t * H + c) = out;
  } else {
    *reinterpret_cast<float4*>(static_cast<float*>(y) + t * H + c) = acc;
  }
  }
}

}  // namespace

cudaError_t launch_reduce(const void* slot_out, int slot_dtype, const int32_t* slot_of,
                          const float* topk_w, int64_t T, int k, int64_t H, void* y, int y_dtype,
                          cudaStream_t stream) {
  if (T == 0) return cudaSuccess;
  dim3 grid(static_cast<unsigned>(ceil_div(H / 4, kReduceThreads)),
            static_cast<unsigned>(T < 65535 ? T : 65535));
  const float* f = static_cast<const float*>(slot_out);
  const __nv_bfloat16* b = static_cast<const __nv_bfloat16*>(slot_out);
  const __half* h = static_cast<const __half*>(slot_out);
  if (slot_dtype == 2 && y_dtype == 0)
    (void)launch_pdl(unpermute_reduce_kernel<__half, true>, dim3(grid), dim3(kReduceThreads), 0, stream, h, slot_of, topk_w, T, k, H, y);
  else if (slot_dtype == 2)
    (void)launch_pdl(unpermute_reduce_kernel<__half, false>, dim3(grid), dim3(kReduceThreads), 0, stream, h, slot_of, topk_w, T, k, H, y);
  else if (slot_dtype == 1 && y_dtype == 0)
    (void)launch_pdl(unpermute_reduce_kernel<float, true>, dim3(grid), dim3(kReduceThreads), 0, stream, f, slot_of, topk_w, T, k, H, y);
  else if (slot_dtype == 1)
    (void)launch_pdl(unpermute_reduce_kernel<float, false>, dim3(grid), dim3(kReduceThreads), 0, stream, f, slot_of, topk_w, T, k, H, y);
  else if (y_dtype == 0)
    (void)launch_pdl(unpermute_reduce_kernel<__nv_bfloat16, true>, dim3(grid), dim3(kReduceThreads), 0, stream, b, slot_of, topk_w, T, k, H, y);
  else
    (void)launch_pdl(unpermute_reduce_kernel<__nv_bfloat16, false>, dim3(grid), dim3(kReduceThreads), 0, stream, b, slot_of, topk_w, T, k, H, y);
  return cudaGetLastError();
}

}  // namespace nvmoe
