// NVFP4 block quantisation shared by the quantiser kernels and the fused
// decode kernel ("NVFP4 MegaMoE Debug Log", Hypotheses §6 steps 1-5; commit
// message "Three bugs fixed" on src).  IEEE fp32, round-to-nearest-even.
#pragma once

#include <cstdint>

#include "internal.h"
#include "ptx.cuh"

namespace nvmoe {

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
  return v;
}

// Quantise one 16-element block given gs and denom = 6*gs:
//   sf = E4M3_satfinite(b / denom), d = dec(sf) * gs,
//   nibble = E2M1_satfinite(|v| / d) | sign(v) << 3  (all 0 when d == 0).
// Returns the scale byte; `packed` receives 8 bytes (element 2j low nibble).
__device__ __forceinline__ uint32_t quant_block16(const float (&v)[16], float gs, float denom,
                                                  uint32_t (&packed)[2]) {
  float b = 0.0f;
#pragma unroll
  for (int i = 0; i < 16; ++i) b = fmaxf(b, fabsf(v[i]));
  const uint32_t sf = cvt_e4m3_satfinite(__fdiv_rn(b, denom));
  const float d = __fmul_rn(e4m3_to_float(sf), gs);
  packed[0] = packed[1] = 0u;
  if (d != 0.0f) {
    // |v| / d correctly rounded without 16 divisions: with rd = RN(1/d),
    // q0 = RN(|v|*rd) is within an ulp of the quotient, the residual
    // |v| - q0*d is exact in one fma, and RN(q0 + residual*rd) is the
    // correctly rounded quotient (Markstein's correction step, IBM J. Res.
    // Dev. 34(1), 1990).  It needs normal numbers, which holds wherever the
    // E2M1 decision can change (quotients >= 0.25); a divisor whose
    // reciprocal would not be normal takes true divisions.
    const float rd = __frcp_rn(d);
    const bool normal = d > 1.0e-36f && d < 1.0e36f;
    auto quot = [&](float a) {
      if (!normal) return __fdiv_rn(a, d);
      const float q0 = __fmul_rn(a, rd);
      return __fmaf_rn(__fmaf_rn(-q0, d, a), rd, q0);
    };
#pragma unroll
    for (int p = 0; p < 8; ++p) {
      const float lo = v[2 * p], hi = v[2 * p + 1];
      uint32_t byte = cvt_e2m1x2_satfinite(quot(fabsf(lo)), quot(fabsf(hi)));
      byte |= (__float_as_uint(lo) >> 31) << 3;
      byte |= (__float_as_uint(hi) >> 31) << 7;
      packed[p >> 2] |= byte << (8 * (p & 3));
    }
  }
  return sf;
}

// gs = amax / (6 * 448), 1 for an all-zero tensor.
__device__ __forceinline__ float global_scale_from(float amax) {
  return amax == 0.0f ? 1.0f : __fdiv_rn(amax, 2688.0f);
}

// Max of n partial maxima, by one warp (result in every lane).  Loads go
// through L2 so that values written earlier in the same kernel by other
// CTAs are seen.
__device__ __forceinline__ float reduce_partials(const float* __restrict__ partial, int n) {
  float m = 0.0f;
  for (int i = threadIdx.x & 31; i < n; i += 32) m = fmaxf(m, __ldcg(partial + i));
  return warp_max(m);
}

// Byte offset of scale (row, 16-element group g) in the staged layout.
__device__ __forceinline__ size_t staged_offset(int64_t row, int g, int k_atoms) {
  return (static_cast<size_t>(row / kTileRows) * k_atoms + (g >> 2)) * kSfAtomBytes +
         (row & 31) * 16 + ((row & 127) >> 5) * 4 + (g & 3);
}

}  // namespace nvmoe
