// Dense NVFP4 tensor-core throughput probe: back-to-back
// tcgen05.mma kind::mxf4nvf4 (E2M1 operands from shared memory, E4M3 block
// scales per 16 elements from TMEM, fp32 accumulator in TMEM) on every SM,
// with nothing else in the loop but the scale copies a GEMM would issue.
// It gives the denominator of the prefill roofline ("% of the dense FP4
// tensor peak") as a measured number, and the cost of each way of staging
// the block scales into TMEM.
//
// Variants (bit flags):
//   kProbePair    one MMA over a CTA pair (cta_group::2, M = 256; each CTA
//                 holds 128 rows of A and N/2 rows of B), else one CTA
//                 (M = 128)
//   kProbeN128    N = 128 instead of 256
//   kProbeCp32    per MMA (K = 64) the scale copies of a 32x128b.warpx4
//                 staging: 1 for A, N/128 for B
//   kProbeCp256   per four MMAs (K = 256) 128x256b copies: 1 for A,
//                 N/64 for B
//   kProbeAcc2    MMAs alternate between two accumulators (columns 0 and N)
//   kProbeAcc4    N = 128 only: four accumulators (columns 0, 128, 256, 384)
//   kProbeNoAcc   every MMA overwrites its accumulator (no dependence on
//                 the previous one)
//   kProbeNoMma   only the scale copies (with kProbeCp32 or kProbeCp256)
//   kProbeCpAOnly with kProbeCp256: only the A copy (one per four MMAs)
//   kProbeCpEarly with kProbeCp256: the next four MMAs' copies are issued
//                 after the second MMA of the current four
//   kProbeSt      the scales written by four warps with tcgen05.st (one CTA;
//                 see mma_probe_st_kernel)
// Without the copy flags the scale columns are never written: the MMAs read
// whatever TMEM holds, which changes no timing.
// Operand bytes are constant (E2M1 1.0, scales 1.0): the values do not
// change the tensor pipe's timing and cannot overflow.
#include "internal.h"
#include "ptx.cuh"

namespace nvmoe {

namespace {

constexpr int kProbeThreads = 128;
constexpr int kProbeABytes = 128 * 128;           // 128 rows x 128 B (K = 256)
constexpr int kProbeBBytes = 256 * 128;
constexpr int kProbeSfBytes = 5 * 4096;           // room for five 128x256b sources
constexpr int kProbeUsed = kProbeABytes + kProbeBBytes + kProbeSfBytes + 1024 + 64;
// more than half of an SM's shared memory, so that one CTA runs per SM (two
// would also contend for the 512 TMEM columns each allocates)
constexpr int kProbeSmem = 160 * 1024;
static_assert(kProbeUsed <= kProbeSmem, "probe shared memory");

template <bool kPair>
__global__ void __launch_bounds__(kProbeThreads, 1) mma_probe_kernel(int iters, int variant,
                                                                     long long* cycles,
                                                                     int* status) {
  extern __shared__ uint8_t raw[];
  uint8_t* smem = raw + ((1024u - (smem_u32(raw) & 1023u)) & 1023u);
  uint8_t* sA = smem;
  uint8_t* sB = sA + kProbeABytes;
  uint8_t* sSf = sB + kProbeBBytes;
  uint64_t* bar = reinterpret_cast<uint64_t*>(sSf + kProbeSfBytes);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar + 1);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int N = (variant & kProbeN128) ? 128 : 256;
  const uint32_t rank = kPair ? cluster_ctarank() : 0u;

  // operands: E2M1 code 2 (= 1.0) in both nibbles; scales 0x38 (= 1.0)
  for (int i = threadIdx.x; i < (kProbeABytes + kProbeBBytes) / 4; i += blockDim.x)
    reinterpret_cast<uint32_t*>(sA)[i] = 0x22222222u;
  for (int i = threadIdx.x; i < kProbeSfBytes / 4; i += blockDim.x)
    reinterpret_cast<uint32_t*>(sSf)[i] = 0x38383838u;
  fence_proxy_async_smem();
  if (threadIdx.x == 0) {
    mbar_init(bar, 1);
    fence_mbarrier_init();
  }
  if (warp == 1) {
    if (kPair) {
      tmem_alloc_pair(tmem_slot, 512);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(tmem_slot, 512);
      tmem_relinquish();
    }
  }
  tc_fence_before();
  if (kPair) cluster_sync(); else __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  const bool issuer = warp == 1 && lane == 0 && rank == 0;
  if (issuer) {
    const uint32_t idesc = idesc_mxf4nvf4(kPair ? 256 : 128, N);
    const uint32_t a0 = smem_u32(sA), b0 = smem_u32(sB), sf0 = smem_u32(sSf);
    const uint32_t sf_t0 = tmem + 256;
    const int n_acc = (variant & kProbeAcc4) ? 4 : (variant & kProbeAcc2) ? 2 : 1;
    const long long t0 = static_cast<long long>(clock64_now());
    for (int i = 0; i < iters; ++i) {
      const int kb = i & 3;
      const uint32_t slot = sf_t0 + ((i >> 2) & 3) * 48;     // four stage slots
      uint32_t sfa = slot + kb * 4, sfb = slot + 16 + kb * 8;
      if (variant & kProbeCp32) {
        const uint64_t d = smem_desc(sf0 + kb * 512, 16, 128, 0);
        if (kPair) {
          tmem_cp_32x128b_warpx4_pair(sfa, d);
          for (int h = 0; h < N / 128; ++h) tmem_cp_32x128b_warpx4_pair(sfb + 4 * h, d);
        } else {
          tmem_cp_32x128b_warpx4(sfa, d);
          for (int h = 0; h < N / 128; ++h) tmem_cp_32x128b_warpx4(sfb + 4 * h, d);
        }
      } else if ((variant & kProbeCp256) &&
                 kb == ((variant & kProbeCpEarly) ? 2 : 0)) {
        // early: the next stage's copies go out between this stage's MMAs
        const uint32_t cslot = (variant & kProbeCpEarly)
                                   ? sf_t0 + (((i >> 2) + 1) & 3) * 48 : slot;
        const int n_cp = (variant & kProbeCpAOnly) ? 1 : 1 + N / 64;
        for (int c = 0; c < n_cp; ++c) {
          // 128 rows x 32 B: 8-row groups 256 B apart, each two 128-byte
          // core matrices (16 B columns) 128 B apart; 4 KB per copy
          const uint64_t d = smem_desc(sf0 + c * 4096, 128, 256, 0);
          if (kPair) tmem_cp_128x256b_pair(cslot + c * 8, d);
          else tmem_cp_128x256b(cslot + c * 8, d);
        }
      }
      if (variant & kProbeNoMma) continue;
      const uint64_t ad = smem_desc(a0 + kb * 32, 16, 1024, 2);
      const uint64_t bd = smem_desc(b0 + kb * 32, 16, 1024, 2);
      uint32_t d = tmem;
      if (variant & kProbeAcc2) d += (i & 1) * N;
      if (variant & kProbeAcc4) d += (i & 3) * 128;
      const uint32_t acc = (variant & kProbeNoAcc) ? 0u : (i >= n_acc ? 1u : 0u);
      if (kPair) mma_mxf4nvf4_pair(d, ad, bd, idesc, sfa, sfb, acc);
      else mma_mxf4nvf4(d, ad, bd, idesc, sfa, sfb, acc);
    }
    if (kPair) tc_commit_pair(bar, 3); else tc_commit(bar);
    mbar_wait(bar, 0, status, nullptr);
    cycles[blockIdx.x] = static_cast<long long>(clock64_now()) - t0;
  } else if (kPair && rank == 1 && warp == 1 && lane == 0) {
    // the pair's MMAs write this CTA's TMEM and read its shared memory:
    // stay until they are done
    mbar_wait(bar, 0, status, nullptr);
    cycles[blockIdx.x] = -1;
  }
  tc_fence_before();
  if (kPair) cluster_sync(); else __syncthreads();
  tc_fence_after();
  if (warp == 1) {
    if (kPair) tmem_dealloc_pair(tmem, 512);
    else tmem_dealloc(tmem, 512);
  }
}

// kProbeSt: the block scales reach TMEM through tcgen05.st, written by four
// warps (warp w = TMEM lanes 32w..32w+31) from shared memory, one 256-K stage
// (four MMAs) at a time into four rotating slots; a fifth warp issues the
// MMAs.  Per stage and warp: the A scales of its 32 rows for the four
// k-blocks (one x16 store: k-block kb in column 4 kb + w, the column the
// MMA reads for this quarter) and the B scales of all N rows (one x32 store:
// N/32 columns per k-block), the same in every quarter.  Slot s: B at
// 256 + 64 s (32 columns), A at 256 + 64 s + 32 (16 columns); every store
// starts at a multiple of its column count, and the MMA's scale addresses
// are multiples of 4 (A) and 8 (B).
constexpr int kProbeStThreads = 160;

__global__ void __launch_bounds__(kProbeStThreads, 1) mma_probe_st_kernel(int iters, int variant,
                                                                         long long* cycles,
                                                                         int* status) {
  extern __shared__ uint8_t raw[];
  uint8_t* smem = raw + ((1024u - (smem_u32(raw) & 1023u)) & 1023u);
  uint8_t* sA = smem;
  uint8_t* sB = sA + kProbeABytes;
  uint8_t* sSf = sB + kProbeBBytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sSf + kProbeSfBytes);
  uint64_t* sf_full = bars;          // [4], 4 arrivals (one per writer warp)
  uint64_t* sf_empty = bars + 4;     // [4], MMA commit
  uint64_t* done = bars + 8;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 9);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int N = (variant & kProbeN128) ? 128 : 256;
  const int stages = iters / 4;

  for (int i = threadIdx.x; i < (kProbeABytes + kProbeBBytes) / 4; i += blockDim.x)
    reinterpret_cast<uint32_t*>(sA)[i] = 0x22222222u;
  for (int i = threadIdx.x; i < kProbeSfBytes / 4; i += blockDim.x)
    reinterpret_cast<uint32_t*>(sSf)[i] = 0x38383838u;
  fence_proxy_async_smem();
  if (threadIdx.x == 0) {
    for (int s = 0; s < 4; ++s) {
      mbar_init(&sf_full[s], 4);
      mbar_init(&sf_empty[s], 1);
    }
    mbar_init(done, 1);
    tmem_slot[1] = 0;                // abort word
    fence_mbarrier_init();
  }
  if (warp == 4) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  volatile int* abort = reinterpret_cast<volatile int*>(tmem_slot + 1);

  if (warp < 4) {
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(warp * 32) << 16);
    const uint32_t* src = reinterpret_cast<const uint32_t*>(sSf);
    for (int st = 0; st < stages; ++st) {
      const int slot = st & 3, use = st >> 2;
      if (use > 0 && !mbar_wait(&sf_empty[slot], (use - 1) & 1, status, abort)) break;
      tc_fence_after();
      uint32_t b[32], a[16];
#pragma unroll
      for (int j = 0; j < 32; ++j) b[j] = src[(j * 32 + lane) & 1023];
#pragma unroll
      for (int j = 0; j < 16; ++j) a[j] = (j & 3) == warp ? src[(1024 + j * 32 + lane) & 2047] : 0u;
      const uint32_t col = 256 + slot * 64;
      // 32 columns: N/32 per k-block (with N = 128 the upper half is unused)
      tmem_st_32x32b_x32(lane_base + col, b);
      tmem_st_32x32b_x16(lane_base + col + 32, a);
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sf_full[slot]);
    }
  } else if (lane == 0) {
    const uint32_t idesc = idesc_mxf4nvf4(128, N);
    const uint32_t a0 = smem_u32(sA), b0 = smem_u32(sB);
    const long long t0 = static_cast<long long>(clock64_now());
    bool ok = true;
    for (int st = 0; st < stages && ok; ++st) {
      const int slot = st & 3, use = st >> 2;
      if (!mbar_wait(&sf_full[slot], use & 1, status, abort)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t col = tmem + 256 + slot * 64;
      for (int kb = 0; kb < 4; ++kb) {
        const uint64_t ad = smem_desc(a0 + kb * 32, 16, 1024, 2);
        const uint64_t bd = smem_desc(b0 + kb * 32, 16, 1024, 2);
        mma_mxf4nvf4(tmem, ad, bd, idesc, col + 32 + 4 * kb, col + 8 * kb,
                     (st | kb) ? 1u : 0u);
      }
      tc_commit(&sf_empty[slot]);
    }
    tc_commit(done);
    mbar_wait(done, 0, status, nullptr);
    cycles[blockIdx.x] = static_cast<long long>(clock64_now()) - t0;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 4) tmem_dealloc(tmem, 512);
}

PerDeviceOnce g_probe_attr[2];
PerDeviceOnce g_probe_st_attr;

}  // namespace

cudaError_t launch_mma_probe(int variant, int iters, int grid, long long* cycles, int* status,
                             cudaStream_t stream) {
  if (variant & kProbeSt) {
    cudaError_t e = set_smem_attr_once(
        g_probe_st_attr, reinterpret_cast<const void*>(mma_probe_st_kernel), kProbeSmem);
    if (e != cudaSuccess) return e;
    mma_probe_st_kernel<<<grid, kProbeStThreads, kProbeSmem, stream>>>(iters, variant, cycles,
                                                                       status);
    return cudaGetLastError();
  }
  const bool pair = (variant & kProbePair) != 0;
  const void* fn = pair ? reinterpret_cast<const void*>(mma_probe_kernel<true>)
                        : reinterpret_cast<const void*>(mma_probe_kernel<false>);
  cudaError_t e = set_smem_attr_once(g_probe_attr[pair], fn, kProbeSmem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kProbeThreads);
  cfg.dynamicSmemBytes = kProbeSmem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = pair ? 2 : 1;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (pair) return cudaLaunchKernelEx(&cfg, mma_probe_kernel<true>, iters, variant, cycles, status);
  return cudaLaunchKernelEx(&cfg, mma_probe_kernel<false>, iters, variant, cycles, status);
}

}  // namespace nvmoe
