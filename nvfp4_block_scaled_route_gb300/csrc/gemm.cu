// Grouped NVFP4 block-scaled GEMM on the 5th-generation tensor cores
// (tcgen05.mma kind::mxf4nvf4, E4M3 scales per 16 elements, fp32
// accumulators in TMEM), fed by TMA, persistent over (expert, n-tile,
// m-tile) tiles.
//
//   L1 (mode 1): acc = A_e x [W1_gate tile | W1_up tile]^T, 128 x (128+128);
//                epilogue alpha1 = gs_x * gs_w1[e], h = silu(alpha1 g) *
//                (alpha1 u), per-CTA amax(|h|), optional alpha-scaled tap.
//   L2 (mode 2): acc = A_e x W2 tile^T, 128 x 256; epilogue alpha2 =
//                gs_h * gs_w2[e] times acc -> slot_out.
// ("NVFP4 MegaMoE Debug Log", NVFP4 MoE Pipeline: the L1/L2 GEMMs with
// per-expert alpha, SiLU(gate)*up on the plain [gate; up] halves.)
//
// Warp roles (192 threads, one CTA per SM):
//   warp 0      TMA producer (A tile, two 128-row B tiles, staged scales)
//   warp 1      TMEM allocator; lane 0 issues tcgen05.cp (scales -> TMEM)
//               and tcgen05.mma
//   warps 2..5  epilogue: tcgen05.ld of the accumulator, one row per thread
//
// Shared memory per stage (K = 256 elements = 128 bytes per row):
//   A 128 rows x 128 B (16 KB), B 256 rows x 128 B (32 KB), both in the
//   128-byte-swizzled K-major layout the TMA writes and the MMA reads;
//   SFA 4 atoms (2 KB), SFB 2 x 4 atoms (4 KB) of 512-byte scale atoms.
// TMEM (512 columns): accumulator in columns [0, 256); scale slots of
// stage s at 256 + 48 s: SFA 4 columns per 64-element k-block, SFB 8.
#include "internal.h"
#include "ptx.cuh"

namespace nvmoe {

namespace {

constexpr int kStages = 4;
constexpr int kBM = 128;
constexpr int kBN = 256;
constexpr int kRowBytes = kStageK / 2;                  // 128
constexpr int kABytes = kBM * kRowBytes;                // 16384
constexpr int kBBytes = kBN * kRowBytes;                // 32768
constexpr int kSfaBytes = 4 * kSfAtomBytes;             // 2048
constexpr int kSfbBytes = 2 * 4 * kSfAtomBytes;         // 4096
constexpr uint32_t kStageTx = kABytes + kBBytes + kSfaBytes + kSfbBytes;
constexpr int kOffA = 0;
constexpr int kOffB = kOffA + kStages * kABytes;
constexpr int kOffSfa = kOffB + kStages * kBBytes;
constexpr int kOffSfb = kOffSfa + kStages * kSfaBytes;
constexpr int kOffBar = kOffSfb + kStages * kSfbBytes;
constexpr int kSmemUsed = kOffBar + 256;
constexpr int kSmemBytes = kSmemUsed + 1024;            // alignment slack
constexpr int kThreads = 192;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemSf = 256;
constexpr uint32_t kTmemSfStage = 48;

struct __align__(8) Barriers {
  uint64_t full[kStages];
  uint64_t empty[kStages];
  uint64_t acc_full;
  uint64_t acc_empty;
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
};
static_assert(sizeof(Barriers) <= 256, "barrier block");

struct TileInfo {
  int e, nt, mt;
};

// Tile t -> (expert, n-tile, m-tile); m-tiles vary fastest so that CTAs
// running at the same time share the expert's B tile in L2.
__device__ __forceinline__ TileInfo decode_tile(int t, const int* prefix, const int* mtiles,
                                                int E) {
  int e = 0;
  while (e + 1 < E && prefix[e + 1] <= t) ++e;
  const int local = t - prefix[e];
  TileInfo ti;
  ti.e = e;
  ti.nt = local / mtiles[e];
  ti.mt = local - ti.nt * mtiles[e];
  return ti;
}

// Work partition.  With many tiles (>= kStreamKFactor per CTA) CTAs take
// whole tiles round-robin.  With few tiles (decode) the tiles x K-stages
// sequence is cut into gridDim.x equal contiguous ranges ("stream-K"): a
// tile split between CTAs is summed by the CTA that finishes it last, in
// ascending K order (deterministic), from fp32 partials in the workspace.
constexpr int kStreamKFactor = 4;

struct WorkIter {
  bool stream_k;
  int total, ks, G;
  int64_t cur, end;   // stream-K: linear stage units
  int t;              // round-robin: next tile

  __device__ void init(int total_tiles, int k_stages, int grid, int cta) {
    total = total_tiles;
    ks = k_stages;
    G = grid;
    stream_k = total_tiles < kStreamKFactor * grid;
    const int64_t W = static_cast<int64_t>(total_tiles) * k_stages;
    cur = end = 0;
    t = cta;
    if (stream_k) {
      // never more ranges than stage units, so that every range is non-empty
      // and the CTAs c_first..c_last of a tile all hold a piece of it
      if (W < G) G = static_cast<int>(W);
      if (cta < G) {
        cur = W * cta / G;
        end = W * (cta + 1) / G;
      }
    }
  }
  __device__ bool next(int& tile, int& s0, int& s1) {
    if (!stream_k) {
      if (t >= total) return false;
      tile = t;
      s0 = 0;
      s1 = ks;
      t += G;
      return true;
    }
    if (cur >= end) return false;
    tile = static_cast<int>(cur / ks);
    s0 = static_cast<int>(cur - static_cast<int64_t>(tile) * ks);
    const int64_t lim = end - static_cast<int64_t>(tile) * ks;
    s1 = lim < ks ? static_cast<int>(lim) : ks;
    cur = static_cast<int64_t>(tile) * ks + s1;
    return true;
  }
  // CTA whose range holds stage unit u
  __device__ int owner(int64_t u) const {
    const int64_t W = static_cast<int64_t>(total) * ks;
    return static_cast<int>(((u + 1) * G + W - 1) / W - 1);
  }
  __device__ int first_tile(int cta) const {
    const int64_t W = static_cast<int64_t>(total) * ks;
    return static_cast<int>(W * cta / G / ks);
  }
  // partial slot of CTA c's piece of tile t (a CTA holds at most two pieces)
  __device__ int slot(int c, int tile) const { return 2 * c + (tile == first_tile(c) ? 0 : 1); }
};

__device__ __forceinline__ float silu_f(float g) { return g / (1.0f + expf(-g)); }

// L1 epilogue on 32 columns: gate g[] and up u[] (raw accumulators).
__device__ __forceinline__ void epi_l1(const float (&g)[32], const float (&u)[32], float alpha,
                                       int64_t row, int col, const GemmArgs& args, float& amax) {
  const int I = args.I;
  float* hp = args.out + row * I + col;
#pragma unroll
  for (int i = 0; i < 32; i += 4) {
    float gv[4], uv[4], hv[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      gv[j] = __fmul_rn(alpha, g[i + j]);
      uv[j] = __fmul_rn(alpha, u[i + j]);
      hv[j] = __fmul_rn(silu_f(gv[j]), uv[j]);
      amax = fmaxf(amax, fabsf(hv[j]));
    }
    *reinterpret_cast<float4*>(hp + i) = make_float4(hv[0], hv[1], hv[2], hv[3]);
    if (args.tap != nullptr) {
      float* tp = args.tap + row * (2 * I) + col + i;
      *reinterpret_cast<float4*>(tp) = make_float4(gv[0], gv[1], gv[2], gv[3]);
      *reinterpret_cast<float4*>(tp + I) = make_float4(uv[0], uv[1], uv[2], uv[3]);
    }
  }
}

// L2 epilogue on 32 columns.
__device__ __forceinline__ void epi_l2(const float (&a)[32], float alpha, int64_t row, int col,
                                       const GemmArgs& args) {
  float* op = args.out + row * args.N + col;
#pragma unroll
  for (int i = 0; i < 32; i += 4)
    *reinterpret_cast<float4*>(op + i) =
        make_float4(__fmul_rn(alpha, a[i]), __fmul_rn(alpha, a[i + 1]),
                    __fmul_rn(alpha, a[i + 2]), __fmul_rn(alpha, a[i + 3]));
}

__device__ __forceinline__ void tmem_ld_f32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  tmem_ld_32x32b_x32(taddr, r);
  tmem_ld_wait();
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void epi_bar() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

__global__ void __launch_bounds__(kThreads, 1) grouped_gemm_kernel(
    const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b,
    const GemmArgs args) {
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte alignment for the 128-byte-swizzled tiles
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
  Barriers* bars = reinterpret_cast<Barriers*>(smem + kOffBar);

  __shared__ int s_prefix[kMaxExperts + 1];
  __shared__ int s_mtiles[kMaxExperts];
  __shared__ int s_off[kMaxExperts];
  __shared__ int s_cnt[kMaxExperts];
  __shared__ float s_amax[4];
  __shared__ int s_last;
  __shared__ int s_ok;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int E = args.E;

  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    const int c = args.expert_counts[e];
    s_cnt[e] = c;
    s_off[e] = args.expert_offsets[e];
    s_mtiles[e] = (c + kBM - 1) / kBM;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int acc = 0;
    for (int e = 0; e < E; ++e) {
      s_prefix[e] = acc;
      acc += s_mtiles[e] * args.n_tiles;
    }
    s_prefix[E] = acc;
  }
  if (warp == 0 && lane == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&bars->full[s], 1);
      mbar_init(&bars->empty[s], 1);
    }
    mbar_init(&bars->acc_full, 1);
    mbar_init(&bars->acc_empty, 4);
    mbar_init(&bars->drain, 1);
    bars->abort = 0;
    fence_mbarrier_init();
    prefetch_tensormap(&map_a);
    prefetch_tensormap(&map_b);
  }
  if (warp == 1) {
    tmem_alloc(&bars->tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  const int total_tiles = s_prefix[E];
  volatile int* abort = &bars->abort;
  const int k_blocks = args.K / 64;
  const int k_stages = (args.K + kStageK - 1) / kStageK;
  const int k_atoms = k_stages * 4;
  WorkIter it;
  it.init(total_tiles, k_stages, gridDim.x, blockIdx.x);
  int tile, s0, s1;

  if (warp == 0) {
    // ------------------------------------------------------- producer --
    if (lane == 0) {
      const uint64_t pol_a = policy_evict_last();
      const uint64_t pol_b = policy_evict_first();
      int stage = 0;
      uint32_t phase = 0;
      int issued = 0;
      bool ok = true;
      while (ok && it.next(tile, s0, s1)) {
        const TileInfo ti = decode_tile(tile, s_prefix, s_mtiles, E);
        const int a_row = s_off[ti.e] + ti.mt * kBM;
        int b_row0, b_row1;
        if (args.mode == 1) {
          b_row0 = ti.e * args.N + ti.nt * 128;
          b_row1 = b_row0 + args.I;
        } else {
          b_row0 = ti.e * args.N + ti.nt * kBN;
          b_row1 = b_row0 + 128;
        }
        // B is stored as contiguous 16 KB tiles (128 rows x one K-stage)
        const int b_tile0 = (b_row0 / 128) * k_stages;
        const int b_tile1 = (b_row1 / 128) * k_stages;
        const uint8_t* sfa = args.a_sf + (static_cast<size_t>(a_row / 128) * k_atoms) * kSfAtomBytes;
        const uint8_t* sfb0 = args.b_sf + (static_cast<size_t>(b_row0 / 128) * k_atoms) * kSfAtomBytes;
        const uint8_t* sfb1 = args.b_sf + (static_cast<size_t>(b_row1 / 128) * k_atoms) * kSfAtomBytes;
        for (int ks = s0; ks < s1; ++ks) {
          if (!mbar_wait(&bars->empty[stage], phase ^ 1u, args.status, abort)) {
            ok = false;
            break;
          }
          uint64_t* full = &bars->full[stage];
          mbar_arrive_expect_tx(full, kStageTx);
          const int32_t x = ks * kRowBytes;
          tma_load_2d(smem + kOffA + stage * kABytes, &map_a, x, a_row, full, pol_a);
          tma_load_3d(smem + kOffB + stage * kBBytes, &map_b, 0, 0, b_tile0 + ks, full, pol_b);
          tma_load_3d(smem + kOffB + stage * kBBytes + kBBytes / 2, &map_b, 0, 0, b_tile1 + ks,
                      full, pol_b);
          const size_t koff = static_cast<size_t>(ks) * 4 * kSfAtomBytes;
          bulk_load(smem + kOffSfa + stage * kSfaBytes, sfa + koff, kSfaBytes, full, pol_a);
          bulk_load(smem + kOffSfb + stage * kSfbBytes, sfb0 + koff, kSfaBytes, full, pol_b);
          bulk_load(smem + kOffSfb + stage * kSfbBytes + kSfaBytes, sfb1 + koff, kSfaBytes, full,
                    pol_b);
          ++issued;
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      // Wait (bounded) for the last loads issued so that no copy into this
      // CTA's shared memory is in flight when it exits.
      const int tail = issued < kStages ? issued : kStages;
      for (int i = 0; i < tail; ++i) {
        if (--stage < 0) {
          stage = kStages - 1;
          phase ^= 1u;
        }
        mbar_wait(&bars->full[stage], phase, args.status, nullptr);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA --
    if (lane == 0) {
      const uint32_t idesc = idesc_mxf4nvf4(kBM, kBN);
      int stage = 0;
      uint32_t phase = 0, acc_phase = 0;
      bool ok = true;
      while (ok && it.next(tile, s0, s1)) {
        if (!mbar_wait(&bars->acc_empty, acc_phase ^ 1u, args.status, abort)) break;
        tc_fence_after();
        for (int ks = s0; ks < s1; ++ks) {
          if (!mbar_wait(&bars->full[stage], phase, args.status, abort)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sfa_t = tmem + kTmemSf + stage * kTmemSfStage;
          const uint32_t sfb_t = sfa_t + 16;
          const uint32_t a_base = smem_u32(smem + kOffA + stage * kABytes);
          const uint32_t b_base = smem_u32(smem + kOffB + stage * kBBytes);
          const uint32_t sfa_s = smem_u32(smem + kOffSfa + stage * kSfaBytes);
          const uint32_t sfb_s = smem_u32(smem + kOffSfb + stage * kSfbBytes);
          const int nkb = min(4, k_blocks - ks * 4);
          for (int kb = 0; kb < nkb; ++kb) {
            tmem_cp_32x128b_warpx4(sfa_t + kb * 4, smem_desc(sfa_s + kb * kSfAtomBytes, 16, 128, 0));
            tmem_cp_32x128b_warpx4(sfb_t + kb * 8, smem_desc(sfb_s + kb * kSfAtomBytes, 16, 128, 0));
            tmem_cp_32x128b_warpx4(sfb_t + kb * 8 + 4,
                                   smem_desc(sfb_s + kSfaBytes + kb * kSfAtomBytes, 16, 128, 0));
          }
          for (int kb = 0; kb < nkb; ++kb) {
            const uint64_t adesc = smem_desc(a_base + kb * 32, 16, 1024, 2);
            const uint64_t bdesc = smem_desc(b_base + kb * 32, 16, 1024, 2);
            mma_mxf4nvf4(tmem, adesc, bdesc, idesc, sfa_t + kb * 4, sfb_t + kb * 8,
                         (ks != s0 || kb != 0) ? 1u : 0u);
          }
          tc_commit(&bars->empty[stage]);
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        tc_commit(&bars->acc_full);
        acc_phase ^= 1u;
      }
      // make sure every MMA issued by this thread has finished before TMEM
      // is released
      tc_commit(&bars->drain);
      mbar_wait(&bars->drain, 0, args.status, nullptr);
    }
  } else {
    // ------------------------------------------------------- epilogue --
    const int q = warp & 3;                      // TMEM lane quarter
    const int row_in_tile = q * 32 + lane;
    const uint32_t t_row = tmem + (static_cast<uint32_t>(q * 32) << 16);
    const bool lead = warp == 2 && lane == 0;
    float amax = 0.0f;
    uint32_t acc_phase = 0;
    const float gs_a = *args.gs_a;
    while (it.next(tile, s0, s1)) {
      const TileInfo ti = decode_tile(tile, s_prefix, s_mtiles, E);
      const float alpha = __fmul_rn(gs_a, args.gs_b[ti.e]);
      // one thread waits (bounded) and the decision is shared, so the four
      // epilogue warps always take the same path through the named barriers
      if (lead) s_ok = mbar_wait(&bars->acc_full, acc_phase, args.status, abort) ? 1 : 0;
      epi_bar();
      if (!s_ok) break;
      tc_fence_after();
      const bool valid = ti.mt * kBM + row_in_tile < s_cnt[ti.e];
      const int64_t row = s_off[ti.e] + ti.mt * kBM + row_in_tile;
      const int col0 = ti.nt * (args.mode == 1 ? 128 : kBN);
      if (s0 == 0 && s1 == k_stages) {
        // whole tile in this CTA: epilogue straight from TMEM
        if (args.mode == 1) {
          for (int c = 0; c < 4; ++c) {
            float g[32], u[32];
            tmem_ld_f32(t_row + c * 32, g);
            tmem_ld_f32(t_row + 128 + c * 32, u);
            if (valid) epi_l1(g, u, alpha, row, col0 + c * 32, args, amax);
          }
        } else {
          for (int c = 0; c < 8; ++c) {
            float a[32];
            tmem_ld_f32(t_row + c * 32, a);
            if (valid) epi_l2(a, alpha, row, col0 + c * 32, args);
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->acc_empty);
      } else {
        // a piece of a split tile: park the raw accumulator in the workspace
        float* mine = args.partials +
                      (static_cast<size_t>(it.slot(blockIdx.x, tile)) * kBM + row_in_tile) * kBN;
        for (int c = 0; c < 8; ++c) {
          float a[32];
          tmem_ld_f32(t_row + c * 32, a);
          if (valid) {
#pragma unroll
            for (int i = 0; i < 32; i += 4)
              __stcg(reinterpret_cast<float4*>(mine + c * 32 + i),
                     make_float4(a[i], a[i + 1], a[i + 2], a[i + 3]));
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->acc_empty);
        __threadfence();
        epi_bar();
        const int64_t u_first = static_cast<int64_t>(tile) * k_stages;
        const int c_first = it.owner(u_first);
        const int c_last = it.owner(u_first + k_stages - 1);
        if (lead) s_last = atomicAdd(&args.counters[tile], 1) == c_last - c_first;
        epi_bar();
        if (s_last) {
          // every piece has landed: sum them in ascending K order
          __threadfence();
          if (lead) args.counters[tile] = 0;
          if (valid) {
            const int nch = args.mode == 1 ? 4 : 8;
            for (int c = 0; c < nch; ++c) {
              float a[32], b[32];
#pragma unroll
              for (int i = 0; i < 32; ++i) a[i] = b[i] = 0.0f;
              for (int cc = c_first; cc <= c_last; ++cc) {
                const float* p = args.partials +
                                 (static_cast<size_t>(it.slot(cc, tile)) * kBM + row_in_tile) * kBN;
#pragma unroll
                for (int i = 0; i < 32; i += 4) {
                  const float4 v = __ldcg(reinterpret_cast<const float4*>(p + c * 32 + i));
                  a[i] += v.x; a[i + 1] += v.y; a[i + 2] += v.z; a[i + 3] += v.w;
                  if (args.mode == 1) {
                    const float4 w = __ldcg(reinterpret_cast<const float4*>(p + 128 + c * 32 + i));
                    b[i] += w.x; b[i + 1] += w.y; b[i + 2] += w.z; b[i + 3] += w.w;
                  }
                }
              }
              if (args.mode == 1)
                epi_l1(a, b, alpha, row, col0 + c * 32, args, amax);
              else
                epi_l2(a, alpha, row, col0 + c * 32, args);
            }
          }
        }
      }
      acc_phase ^= 1u;
    }
    if (args.mode == 1) {
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
      if (lane == 0) s_amax[q] = amax;
      epi_bar();
      if (lead)
        args.amax_partial[blockIdx.x] =
            fmaxf(fmaxf(s_amax[0], s_amax[1]), fmaxf(s_amax[2], s_amax[3]));
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

int gemm_smem_bytes() { return kSmemBytes; }

cudaError_t launch_gemm(const GemmArgs& args, const CUtensorMap& map_a, const CUtensorMap& map_b,
                        int grid, cudaStream_t stream) {
  static bool attr_set = false;  // per-process; the attribute is per function
  if (!attr_set) {
    cudaError_t err = cudaFuncSetAttribute(grouped_gemm_kernel,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           kSmemBytes);
    if (err != cudaSuccess) return err;
    attr_set = true;
  }
  grouped_gemm_kernel<<<grid, kThreads, kSmemBytes, stream>>>(map_a, map_b, args);
  return cudaGetLastError();
}

}  // namespace nvmoe
