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
// Two kernels share the role code below:
//   grouped_gemm_kernel   one GEMM (L1 or L2) per launch
//   fused_ffn_kernel      cooperative launch for the few-tile (decode) case:
//                         L1 -> grid barrier -> requantise h -> grid barrier
//                         -> L2 in one persistent kernel; the producer starts
//                         loading L2 weights while the L1 tail and the
//                         requantisation are still running.
//
// Warp roles (one CTA per SM; the layer kernel's differ, see there):
//   warp 0      TMA producer (A tile, two 128-row B tiles, staged scales)
//   warp 1      TMEM allocator; lane 0 issues tcgen05.mma (and, in the
//               cooperative kernels, the tcgen05.cp scale copies)
//   warps 2..5  epilogue: tcgen05.ld of the accumulator, one row per thread
//               (and the requantisation in the fused kernel)
//   warps 6..9  grouped_gemm_kernel only: scale writers, each stage's block
//               scales from shared memory into TMEM with tcgen05.st, one
//               warp per TMEM lane quarter.  tcgen05.cp copies of the scales
//               run in the tensor pipe in series with the MMAs: at N = 256
//               the 12 copies of a 256-K stage take 1.6x the time of its 4
//               MMAs, and 5 wide (128x256b) copies 0.5x; stores from warps
//               overlap the MMAs (98 % of the MMA-only rate, measured with
//               the library's probe).  The cooperative decode kernels cannot
//               take four more warps (that would cap their registers below
//               what their epilogue and quantisation code use):
//               fused_ffn_kernel keeps the copies; layer_kernel has one
//               writer warp for lane quarter 0, used when every valid row
//               lies there (one-token batches), else the copies.
//
// Shared memory per stage (K = 256 elements = 128 bytes per row):
//   A 128 rows x 128 B (16 KB), B 256 rows x 128 B (32 KB), both in the
//   128-byte-swizzled K-major layout the TMA writes and the MMA reads;
//   SFA 4 atoms (2 KB), SFB 2 x 4 atoms (4 KB) of 512-byte scale atoms.
// TMEM (512 columns): accumulator in columns [0, 256); scale slot of
// stage s at 256 + 64 s.  With scale writers: SFB in its first 32 columns
// (8 per 64-element k-block), SFA in the next 16 (4 per k-block), every
// tcgen05.st at a multiple of its column count.  With copies: SFA in the
// first 16, SFB in the next 32.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "internal.h"
#include "ptx.cuh"
#include "quant.cuh"

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
constexpr int kThreads = 224;                           // cooperative kernels (7 warps)
constexpr int kThreadsSt = 320;                         // grouped_gemm_kernel<false>
constexpr int kThreadsHalf = 448;                       // grouped_gemm_kernel<true>
constexpr int kSfWarp0 = 6;                             // first scale-writer warp
constexpr int kEpi2Warp0 = 10;                          // second epilogue set
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemSf = 256;
constexpr uint32_t kTmemSfStage = 64;

struct __align__(8) Barriers {
  uint64_t full[kStages];
  uint64_t empty[kStages];
  uint64_t sf_full[kStages];       // the stage's scales are in TMEM (4 writer warps)
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

// Per-expert tables shared by every role (in shared memory).
struct Tables {
  int prefix1[kMaxExperts + 1];   // tile prefix of the first (or only) GEMM
  int prefix2[kMaxExperts + 1];   // tile prefix of L2 in the fused kernel
  int dense[kMaxExperts + 1];     // prefix of slot counts (dense slot ids)
  int mtiles[kMaxExperts];
  int off[kMaxExperts];
  int cnt[kMaxExperts];
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

// The valid rows of a tile (rows row0 + [0, n_valid) of the slot buffers),
// or none when the debug-bounds build finds them past args.rows.
__device__ __forceinline__ int checked_rows(const GemmArgs& a, int64_t row0, int n_valid) {
  if (n_valid > 0 && a.rows > 0 && !NVMOE_BOUNDS(row0 + n_valid <= a.rows, a.status)) return 0;
  return n_valid;
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

  __device__ void init(int total_tiles, int k_stages, int grid, int cta, bool whole = false) {
    total = total_tiles;
    ks = k_stages;
    G = grid;
    stream_k = !whole && total_tiles < kStreamKFactor * grid;
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

// One grouped GEMM as the roles see it.
struct Phase {
  const GemmArgs* a;
  const AMaps* map_a;
  const CUtensorMap* map_b;
  const int* prefix;
  int total_tiles, k_blocks, k_stages, k_atoms;
  bool whole_tiles;     // round-robin whole tiles whatever their number
};

__device__ __forceinline__ Phase make_phase(const GemmArgs& a, const AMaps* ma,
                                            const CUtensorMap* mb, const int* prefix, int E) {
  Phase p;
  p.a = &a;
  p.map_a = ma;
  p.map_b = mb;
  p.prefix = prefix;
  p.total_tiles = prefix[E];
  p.k_blocks = a.K / 64;
  p.k_stages = (a.K + kStageK - 1) / kStageK;
  p.k_atoms = p.k_stages * 4;
  p.whole_tiles = false;
  return p;
}

// Pipeline position of one role (carried across the phases of the fused kernel).
struct Pipe {
  int stage = 0;
  uint32_t phase = 0;
  uint32_t acc_phase = 0;
  int issued = 0;
};

// silu(g) = g / (1 + e^-g) with the hardware exp2 approximation and fast
// division: a few ulp (relative error below 4e-6 for |g| < 30), far inside
// the L1 output tolerance; identical in every kernel that uses it.
__device__ __forceinline__ float silu_f(float g) { return __fdividef(g, 1.0f + __expf(-g)); }

// L1 epilogue on 32 columns: gate g[] and up u[] (raw accumulators).
__device__ __forceinline__ void epi_l1(const float (&g)[32], const float (&u)[32], float alpha,
                                       float alpha_u, int64_t row, int col, const GemmArgs& args,
                                       float& amax) {
  const int I = args.I;
  float* hp = args.out + row * I + col;
#pragma unroll
  for (int i = 0; i < 32; i += 8) {
    float gv[8], uv[8], hv[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      gv[j] = __fmul_rn(alpha, g[i + j]);
      uv[j] = __fmul_rn(alpha_u, u[i + j]);
      hv[j] = __fmul_rn(silu_f(gv[j]), uv[j]);
      amax = fmaxf(amax, fabsf(hv[j]));
    }
    st_global_v8(hp + i, hv);
    if (args.tap != nullptr) {
      float* tp = args.tap + row * (2 * I) + col + i;
      st_global_v8(tp, gv);
      st_global_v8(tp + I, uv);
    }
  }
}

// Two values as one bf16x2 word (round to nearest even), first in the low half.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

// Two values as one fp16x2 word (round to nearest even), first in the low half.
__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  const __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

// fp16 holds magnitudes up to 65504: a larger slot value is reported on the
// device (NVMOE_ERR_RANGE), never silently clamped.
constexpr float kF16Max = 65504.0f;

// L2 epilogue on 32 columns: slot_out = alpha * acc, stored as fp32, bf16 or
// fp16 (args.out_dtype 1, 0, 2).
__device__ __forceinline__ void epi_l2(const float (&a)[32], float alpha, int64_t row, int col,
                                       const GemmArgs& args) {
  if (args.out_dtype != 1) {
    const bool half = args.out_dtype == 2;
    uint16_t* op = reinterpret_cast<uint16_t*>(args.out) + row * args.N + col;
    float big = 0.0f;
#pragma unroll
    for (int i = 0; i < 32; i += 16) {
      float w[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float lo = __fmul_rn(alpha, a[i + 2 * j]), hi = __fmul_rn(alpha, a[i + 2 * j + 1]);
        big = fmaxf(big, fmaxf(fabsf(lo), fabsf(hi)));
        w[j] = __uint_as_float(half ? pack_f16x2(lo, hi) : pack_bf16x2(lo, hi));
      }
      st_global_v8(reinterpret_cast<float*>(op + i), w);
    }
    if (half && !(big <= kF16Max)) record_status(args.status, kErrRange);
    return;
  }
  float* op = args.out + row * args.N + col;
#pragma unroll
  for (int i = 0; i < 32; i += 8) {
    float v[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) v[j] = __fmul_rn(alpha, a[i + j]);
    st_global_v8(op + i, v);
  }
}

// The same epilogues on 4 columns (used by the split-tile fixup, where the
// 128 epilogue threads share the valid rows' columns).
__device__ __forceinline__ void epi_l1_4(float4 g, float4 u, float alpha, float alpha_u,
                                         int64_t row, int col, const GemmArgs& args,
                                         float& amax) {
  const int I = args.I;
  const float gv[4] = {__fmul_rn(alpha, g.x), __fmul_rn(alpha, g.y), __fmul_rn(alpha, g.z),
                       __fmul_rn(alpha, g.w)};
  const float uv[4] = {__fmul_rn(alpha_u, u.x), __fmul_rn(alpha_u, u.y), __fmul_rn(alpha_u, u.z),
                       __fmul_rn(alpha_u, u.w)};
  float hv[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    hv[j] = __fmul_rn(silu_f(gv[j]), uv[j]);
    amax = fmaxf(amax, fabsf(hv[j]));
  }
  *reinterpret_cast<float4*>(args.out + row * I + col) = make_float4(hv[0], hv[1], hv[2], hv[3]);
  if (args.tap != nullptr) {
    float* tp = args.tap + row * (2 * I) + col;
    *reinterpret_cast<float4*>(tp) = make_float4(gv[0], gv[1], gv[2], gv[3]);
    *reinterpret_cast<float4*>(tp + I) = make_float4(uv[0], uv[1], uv[2], uv[3]);
  }
}

__device__ __forceinline__ void epi_l2_4(float4 a, float alpha, int64_t row, int col,
                                         const GemmArgs& args) {
  if (args.out_dtype != 1) {
    uint16_t* op = reinterpret_cast<uint16_t*>(args.out) + row * args.N + col;
    const float v[4] = {__fmul_rn(alpha, a.x), __fmul_rn(alpha, a.y), __fmul_rn(alpha, a.z),
                        __fmul_rn(alpha, a.w)};
    if (args.out_dtype == 2) {
      *reinterpret_cast<uint2*>(op) = make_uint2(pack_f16x2(v[0], v[1]), pack_f16x2(v[2], v[3]));
      const float big = fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3])));
      if (!(big <= kF16Max)) record_status(args.status, kErrRange);
    } else {
      *reinterpret_cast<uint2*>(op) = make_uint2(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]));
    }
    return;
  }
  *reinterpret_cast<float4*>(args.out + row * args.N + col) =
      make_float4(__fmul_rn(alpha, a.x), __fmul_rn(alpha, a.y), __fmul_rn(alpha, a.z),
                  __fmul_rn(alpha, a.w));
}

// The same epilogues on one column (used where a warp's few valid rows are
// spread over its 32 lanes, one column per lane).
__device__ __forceinline__ void epi_l1_1(float g, float u, float alpha, float alpha_u,
                                         int64_t row, int col, const GemmArgs& args,
                                         float& amax) {
  const int I = args.I;
  const float gv = __fmul_rn(alpha, g), uv = __fmul_rn(alpha_u, u);
  const float hv = __fmul_rn(silu_f(gv), uv);
  amax = fmaxf(amax, fabsf(hv));
  args.out[row * I + col] = hv;
  if (args.tap != nullptr) {
    args.tap[row * (2 * I) + col] = gv;
    args.tap[row * (2 * I) + col + I] = uv;
  }
}

// Value v[j] of lane `src`, delivered to lane j (32 shuffles; the register
// index is a compile-time constant in every step).
__device__ __forceinline__ float from_lane_column(const float (&v)[32], int src) {
  const int lane = threadIdx.x & 31;
  float out = 0.0f;
#pragma unroll
  for (int j = 0; j < 32; ++j) {
    const float t = __shfl_sync(0xFFFFFFFFu, v[j], src);
    if (lane == j) out = t;
  }
  return out;
}

// At most this many valid rows in a warp's 32-row quarter: the full-tile L1
// epilogue (SiLU of 128 columns per row) turns each row over to the 32 lanes,
// one column each, instead of leaving one thread to work through the row
// alone.  Each row costs 64 shuffles per 32 columns, so this pays only for
// a few rows; the L2 epilogue (one multiply per column) never does.
constexpr int kNarrowRows = 4;

__device__ __forceinline__ void add4(float4& a, float4 b) {
  a.x += b.x;
  a.y += b.y;
  a.z += b.z;
  a.w += b.w;
}

__device__ __forceinline__ void tmem_ld_f32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  tmem_ld_32x32b_x32(taddr, r);
  tmem_ld_wait();
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void epi_bar() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

__device__ __forceinline__ int ld_acquire(const int* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

// Bounded wait until *flag >= target.  Returns false on timeout (status set)
// or when another role of the CTA has given up.
__device__ bool wait_flag(const int* flag, int target, int* status, volatile int* abort,
                          uint64_t limit_ns = kWaitLimitNs) {
  const uint64_t t0 = globaltimer_ns();
  while (ld_acquire(flag) < target) {
    if (abort != nullptr && *abort) return false;
    if (globaltimer_ns() - t0 > limit_ns) {
      record_status(status, kErrTimeout);
      if (abort != nullptr) *abort = 1;
      return false;
    }
    __nanosleep(64);
  }
  fence_proxy_async_global();
  return true;
}

// Grid-wide barrier of a cooperative launch, called by one thread per CTA.
// bar[0] counts arrivals, bar[1] is the generation; both start at zero
// (the host clears them before the launch).  Everything this CTA wrote
// before the call is visible to every CTA after it, to the generic and the
// async (TMA) proxy.
__device__ bool grid_barrier(int* bar, int generation, int* status, volatile int* abort) {
  fence_proxy_async_global();
  __threadfence();
  if (atomicAdd(&bar[0], 1) == static_cast<int>(gridDim.x) - 1) {
    atomicExch(&bar[0], 0);
    __threadfence();
    atomicExch(&bar[1], generation);
    return true;
  }
  return wait_flag(&bar[1], generation, status, abort);
}

// Grid-wide barrier of one use per launch, called by one thread per CTA:
// arrive on the counter, then wait for it to reach the grid size (no flag
// to publish, so the last arriver adds no round trip).  Everything this
// CTA wrote before the call is visible to every CTA after it, to the
// generic and the async (TMA) proxy.
__device__ bool count_barrier(int* count, int* status, volatile int* abort) {
  fence_proxy_async_global();
  __threadfence();
  atomicAdd(count, 1);
  return wait_flag(count, static_cast<int>(gridDim.x), status, abort);
}

// What the activation (A) loads of a phase wait for: a global word reaching
// `target` (a grid barrier's generation, or a count of CTAs whose share of
// the quantised activations is written).
struct Gate {
  const int* flag;
  int target;
};

// ------------------------------------------------------------ producer --
// Issues the loads of every stage of this CTA's items.  When `gate` is
// given, the A-operand (activation) loads wait until the gate opens: the
// weight (B) loads of the first stages go out first and the activation
// loads follow.
__device__ bool run_producer(const Phase& P, int E, const Tables& tb, Barriers* bars,
                             uint8_t* smem, Pipe& pp, volatile int* abort, const Gate* gate) {
  const GemmArgs& args = *P.a;
  WorkIter it;
  it.init(P.total_tiles, P.k_stages, gridDim.x, blockIdx.x, P.whole_tiles);
  const uint64_t pol_a = policy_evict_last();
  const uint64_t pol_b = policy_evict_first();
  // the caller's activation-ready flag: waited for before anything is
  // loaded, so that a wait that runs out leaves no copy in flight
  if (args.ready_flag != nullptr &&
      !wait_flag(args.ready_flag, args.ready_value, args.status, abort, args.ready_limit_ns))
    return false;
  bool gate_open = gate == nullptr;
  // activation loads waiting for the gate: (stage, a_row, ks, small box)
  int def_stage[kStages], def_row[kStages], def_ks[kStages];
  bool def_small[kStages];
  int n_def = 0;
  // An m-tile with at most kSmallABoxRows valid rows loads only those rows of
  // A; the MMA still runs 128 rows, and the stale rows only produce
  // accumulator rows that are never stored.
  auto issue_a = [&](int stage, int a_row, int ks, bool small) {
    uint64_t* full = &bars->full[stage];
    tma_load_2d(smem + kOffA + stage * kABytes, small ? &P.map_a->small : &P.map_a->full,
                ks * kRowBytes, a_row, full, pol_a);
    const uint8_t* sfa = args.a_sf +
                         (static_cast<size_t>(a_row / 128) * P.k_atoms + ks * 4) * kSfAtomBytes;
    bulk_load(smem + kOffSfa + stage * kSfaBytes, sfa, kSfaBytes, full, pol_a);
  };
  auto open_gate = [&]() -> bool {
    if (!wait_flag(gate->flag, gate->target, args.status, abort)) return false;
    gate_open = true;
    for (int i = 0; i < n_def; ++i) issue_a(def_stage[i], def_row[i], def_ks[i], def_small[i]);
    n_def = 0;
    return true;
  };
  bool ok = true;
  int tile, s0, s1;
  while (ok && it.next(tile, s0, s1)) {
    const TileInfo ti = decode_tile(tile, P.prefix, tb.mtiles, E);
    const int a_row = tb.off[ti.e] + ti.mt * kBM;
    const bool small_a = tb.cnt[ti.e] - ti.mt * kBM <= kSmallABoxRows;
    const uint32_t tx = small_a ? kStageTx - (kBM - kSmallABoxRows) * kRowBytes : kStageTx;
    int b_row0, b_row1;
    if (args.mode == 1) {
      b_row0 = ti.e * args.N + ti.nt * 128;
      b_row1 = b_row0 + args.I;
    } else {
      b_row0 = ti.e * args.N + ti.nt * kBN;
      b_row1 = b_row0 + 128;
    }
    // B is stored as contiguous 16 KB tiles (128 rows x one K-stage)
    const int b_tile0 = (b_row0 / 128) * P.k_stages;
    const int b_tile1 = (b_row1 / 128) * P.k_stages;
    const uint8_t* sfb0 = args.b_sf + (static_cast<size_t>(b_row0 / 128) * P.k_atoms) * kSfAtomBytes;
    const uint8_t* sfb1 = args.b_sf + (static_cast<size_t>(b_row1 / 128) * P.k_atoms) * kSfAtomBytes;
    for (int ks = s0; ks < s1; ++ks) {
      if (!gate_open && n_def == kStages && !open_gate()) {
        ok = false;
        break;
      }
      if (!mbar_wait(&bars->empty[pp.stage], pp.phase ^ 1u, args.status, abort)) {
        ok = false;
        break;
      }
      const int stage = pp.stage;
      uint64_t* full = &bars->full[stage];
      mbar_arrive_expect_tx(full, tx);
      tma_load_3d(smem + kOffB + stage * kBBytes, P.map_b, 0, 0, b_tile0 + ks, full, pol_b);
      tma_load_3d(smem + kOffB + stage * kBBytes + kBBytes / 2, P.map_b, 0, 0, b_tile1 + ks,
                  full, pol_b);
      const size_t koff = static_cast<size_t>(ks) * 4 * kSfAtomBytes;
      bulk_load(smem + kOffSfb + stage * kSfbBytes, sfb0 + koff, kSfaBytes, full, pol_b);
      bulk_load(smem + kOffSfb + stage * kSfbBytes + kSfaBytes, sfb1 + koff, kSfaBytes, full,
                pol_b);
      if (gate_open) {
        issue_a(stage, a_row, ks, small_a);
      } else {
        def_stage[n_def] = stage;
        def_row[n_def] = a_row;
        def_ks[n_def] = ks;
        def_small[n_def] = small_a;
        ++n_def;
      }
      ++pp.issued;
      if (++pp.stage == kStages) {
        pp.stage = 0;
        pp.phase ^= 1u;
      }
    }
  }
  if (ok && !gate_open && n_def > 0) ok = open_gate();
  return ok;
}

// Wait (bounded) for the last loads issued so that no copy into this CTA's
// shared memory is in flight when it exits.
__device__ void drain_producer(Barriers* bars, Pipe& pp, int* status) {
  const int tail = pp.issued < kStages ? pp.issued : kStages;
  int stage = pp.stage;
  uint32_t phase = pp.phase;
  for (int i = 0; i < tail; ++i) {
    if (--stage < 0) {
      stage = kStages - 1;
      phase ^= 1u;
    }
    mbar_wait(&bars->full[stage], phase, status, nullptr);
  }
}

// ----------------------------------------------------------------- MMA --
// kStSf: the stage's scales are written into TMEM by the writer warps
// (wait for sf_full); else this thread copies them with tcgen05.cp.
template <bool kStSf>
__device__ bool run_mma(const Phase& P, Barriers* bars, uint8_t* smem, uint32_t tmem, Pipe& pp,
                        volatile int* abort) {
  const GemmArgs& args = *P.a;
  WorkIter it;
  it.init(P.total_tiles, P.k_stages, gridDim.x, blockIdx.x, P.whole_tiles);
  const uint32_t idesc = idesc_mxf4nvf4(kBM, kBN);
  int tile, s0, s1;
  while (it.next(tile, s0, s1)) {
    if (!mbar_wait(&bars->acc_empty, pp.acc_phase ^ 1u, args.status, abort)) return false;
    tc_fence_after();
    for (int ks = s0; ks < s1; ++ks) {
      if (!mbar_wait(&bars->full[pp.stage], pp.phase, args.status, abort)) return false;
      if (kStSf && !mbar_wait(&bars->sf_full[pp.stage], pp.phase, args.status, abort))
        return false;
      tc_fence_after();
      const int stage = pp.stage;
      const uint32_t slot = tmem + kTmemSf + stage * kTmemSfStage;
      const uint32_t sfa_t = kStSf ? slot + 32 : slot;
      const uint32_t sfb_t = kStSf ? slot : slot + 16;
      const uint32_t a_base = smem_u32(smem + kOffA + stage * kABytes);
      const uint32_t b_base = smem_u32(smem + kOffB + stage * kBBytes);
      const int nkb = min(4, P.k_blocks - ks * 4);
      if (!kStSf) {
        const uint32_t sfa_s = smem_u32(smem + kOffSfa + stage * kSfaBytes);
        const uint32_t sfb_s = smem_u32(smem + kOffSfb + stage * kSfbBytes);
        for (int kb = 0; kb < nkb; ++kb) {
          tmem_cp_32x128b_warpx4(sfa_t + kb * 4,
                                 smem_desc(sfa_s + kb * kSfAtomBytes, 16, 128, 0));
          tmem_cp_32x128b_warpx4(sfb_t + kb * 8,
                                 smem_desc(sfb_s + kb * kSfAtomBytes, 16, 128, 0));
          tmem_cp_32x128b_warpx4(sfb_t + kb * 8 + 4,
                                 smem_desc(sfb_s + kSfaBytes + kb * kSfAtomBytes, 16, 128, 0));
        }
      }
      for (int kb = 0; kb < nkb; ++kb) {
        const uint64_t adesc = smem_desc(a_base + kb * 32, 16, 1024, 2);
        const uint64_t bdesc = smem_desc(b_base + kb * 32, 16, 1024, 2);
        mma_mxf4nvf4(tmem, adesc, bdesc, idesc, sfa_t + kb * 4, sfb_t + kb * 8,
                     (ks != s0 || kb != 0) ? 1u : 0u);
      }
      tc_commit(&bars->empty[stage]);
      if (++pp.stage == kStages) {
        pp.stage = 0;
        pp.phase ^= 1u;
      }
    }
    tc_commit(&bars->acc_full);
    pp.acc_phase ^= 1u;
  }
  return true;
}

// ------------------------------------------------------- scale writers --
// Warps 6..9, one per TMEM lane quarter q = warp % 4.  For every stage of
// this CTA's work (in the producer's order), once its loads have landed:
// lane l reads the 16-byte row l of each 512-byte scale atom of the stage
// (A: 4 atoms, one per k-block; B: 2 halves x 4 atoms) and writes them into
// its own TMEM lane 32q + l.  Every quarter gets the same columns, the
// layout the MMA reads: B k-block kb at slot + 8 kb + 4 h + j (half h,
// column j = B row 128 h + 32 j + l), A k-block kb at slot + 32 + 4 kb + j
// (column j = A row 32 j + l).  The slot is free once the stage's loads
// have landed: the producer refills a stage only after the MMAs that read
// its previous scales have completed.
// One stage's scales into this warp's TMEM lanes (the stage's loads have
// landed), then the warp's arrival on the stage's sf_full barrier.
__device__ __forceinline__ void write_stage_sf(int stage, Barriers* bars, const uint8_t* smem,
                                               uint32_t lane_base) {
  const int lane = threadIdx.x & 31;
  const uint4* sa = reinterpret_cast<const uint4*>(smem + kOffSfa + stage * kSfaBytes) + lane;
  const uint4* sb = reinterpret_cast<const uint4*>(smem + kOffSfb + stage * kSfbBytes) + lane;
  uint32_t a[16], b[32];
#pragma unroll
  for (int kb = 0; kb < 4; ++kb) {
    const uint4 v = sa[kb * 32];                       // atom kb, row l
    a[4 * kb] = v.x; a[4 * kb + 1] = v.y; a[4 * kb + 2] = v.z; a[4 * kb + 3] = v.w;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const uint4 u = sb[h * 128 + kb * 32];           // half h, atom kb, row l
      b[8 * kb + 4 * h] = u.x; b[8 * kb + 4 * h + 1] = u.y;
      b[8 * kb + 4 * h + 2] = u.z; b[8 * kb + 4 * h + 3] = u.w;
    }
  }
  const uint32_t col = kTmemSf + stage * kTmemSfStage;
  tmem_st_32x32b_x32(lane_base + col, b);
  tmem_st_32x32b_x16(lane_base + col + 32, a);
  tmem_st_wait();
  tc_fence_before();
  __syncwarp();
  if (lane == 0) mbar_arrive(&bars->sf_full[stage]);
}

__device__ bool run_sf_writer(const Phase& P, Barriers* bars, uint8_t* smem, uint32_t tmem,
                              Pipe& pp, volatile int* abort) {
  const GemmArgs& args = *P.a;
  const uint32_t q = (threadIdx.x >> 5) & 3;
  const uint32_t lane_base = tmem + ((q * 32u) << 16);
  WorkIter it;
  it.init(P.total_tiles, P.k_stages, gridDim.x, blockIdx.x, P.whole_tiles);
  int tile, s0, s1;
  while (it.next(tile, s0, s1)) {
    for (int ks = s0; ks < s1; ++ks) {
      if (!mbar_wait(&bars->full[pp.stage], pp.phase, args.status, abort)) return false;
      write_stage_sf(pp.stage, bars, smem, lane_base);
      if (++pp.stage == kStages) {
        pp.stage = 0;
        pp.phase ^= 1u;
      }
    }
  }
  return true;
}

// ------------------------------------------------------------ epilogue --
// Top-k weighted reduce done inside the layer kernel: when the last of a
// token's k slot rows of one 256-column tile of slot_out is written, the
// CTA that wrote it sums the k rows (ascending j, fp32, the same arithmetic
// as unpermute_reduce_kernel) into y.  A slot with no row (an expert id
// outside [0, E)) is counted in advance by CTA 0 and not summed, as in
// unpermute_reduce_kernel.
struct YReduce {
  int* counts;              // [T][n_tiles], zero between calls
  const float* topk_w;      // [T, k]
  const int* slot_row;      // [T*k] (shared memory)
  const int* dense_token;   // dense slot -> token (shared memory)
  void* y;
  int y_dtype;              // 0 bf16, 1 fp32
  int k;
  int n_tiles;
  int* s_list;              // [kBM] shared memory
  int* s_n;                 // shared memory
};

__device__ void y_after_tile(const YReduce& yr, const TileInfo& ti, const Tables& tb,
                             const GemmArgs& args) {
  const int etid = threadIdx.x - 64;
  const int n_valid = min(kBM, tb.cnt[ti.e] - ti.mt * kBM);
  const int d0 = tb.dense[ti.e] + ti.mt * kBM;
  const int H = args.N;
  __threadfence();                       // this tile's slot_out rows, device-wide
  if (etid == 0) *yr.s_n = 0;
  epi_bar();
  for (int r = etid; r < n_valid; r += 128) {
    const int t = yr.dense_token[d0 + r];
    int* c = &yr.counts[t * yr.n_tiles + ti.nt];
    if (atomicAdd(c, 1) == yr.k - 1) {
      *c = 0;
      yr.s_list[atomicAdd(yr.s_n, 1)] = t;
    }
  }
  epi_bar();
  const int n = *yr.s_n;
  if (n > 0) __threadfence();
  for (int wi = etid; wi < n * (kBN / 4); wi += 128) {
    const int t = yr.s_list[wi / (kBN / 4)];
    const int col = ti.nt * kBN + (wi % (kBN / 4)) * 4;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int j0 = 0; j0 < yr.k; j0 += 8) {
      float4 v[8];
      float wj[8];
      uint32_t live = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int s = j0 + j < yr.k ? yr.slot_row[t * yr.k + j0 + j] : -1;
        if (s >= 0) {
          v[j] = __ldcg(reinterpret_cast<const float4*>(args.out + static_cast<int64_t>(s) * H + col));
          wj[j] = __ldg(yr.topk_w + t * yr.k + j0 + j);
          live |= 1u << j;
        }
      }
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        if ((live >> j) & 1u) {
          acc.x = __fmaf_rn(wj[j], v[j].x, acc.x);
          acc.y = __fmaf_rn(wj[j], v[j].y, acc.y);
          acc.z = __fmaf_rn(wj[j], v[j].z, acc.z);
          acc.w = __fmaf_rn(wj[j], v[j].w, acc.w);
        }
      }
    }
    if (yr.y_dtype == 0) {
      __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y);
      __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z, acc.w);
      uint2 o;
      o.x = *reinterpret_cast<uint32_t*>(&lo);
      o.y = *reinterpret_cast<uint32_t*>(&hi);
      *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(yr.y) + static_cast<int64_t>(t) * H + col) = o;
    } else {
      *reinterpret_cast<float4*>(static_cast<float*>(yr.y) + static_cast<int64_t>(t) * H + col) = acc;
    }
  }
  epi_bar();
}

// With a static intermediate scale: requantise the 128 h columns of a
// finished L1 tile (its valid rows) with gs_mid[e], by the CTA that wrote
// them (epilogue warps; the h stores are visible to the CTA after the
// barrier).  One thread per 4-block quad, so a staged 32-bit scale word is
// written whole; the same block arithmetic as every other quantisation.
__device__ void requant_own_tile(const GemmArgs& args, const TileInfo& ti, const Tables& tb) {
  epi_bar();
  const float gs = __ldg(args.gs_mid + ti.e);
  const float denom = __fmul_rn(6.0f, gs);
  const int I = args.I;
  const int k_atoms = (I + kStageK - 1) / kStageK * 4;
  const int64_t row0 = tb.off[ti.e] + ti.mt * kBM;
  const int n_valid = checked_rows(args, row0, min(kBM, tb.cnt[ti.e] - ti.mt * kBM));
  const int g_base = ti.nt * 8;                       // 128 columns = 8 blocks
  for (int u = threadIdx.x - 64; u < n_valid * 2; u += 128) {
    const int64_t row = row0 + (u >> 1);
    const int g0 = g_base + (u & 1) * 4;
    uint32_t word = 0;
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      const float4* p = reinterpret_cast<const float4*>(args.out + row * I + (g0 + b) * 16);
      float v[16];
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const float4 f = __ldcg(p + c);
        v[4 * c] = f.x; v[4 * c + 1] = f.y; v[4 * c + 2] = f.z; v[4 * c + 3] = f.w;
      }
      uint32_t packed[2];
      word |= quant_block16(v, gs, denom, packed) << (8 * b);
      *reinterpret_cast<uint2*>(args.mid_q + row * (I / 2) + (g0 + b) * 8) =
          make_uint2(packed[0], packed[1]);
    }
    *reinterpret_cast<uint32_t*>(args.mid_sf + staged_offset(row, g0, k_atoms)) = word;
  }
  // the L2 activation loads (async proxy) come after a grid-wide sync
  fence_proxy_async_global();
}

// Four warps (128 threads, one accumulator row each).  Returns false when
// a wait gave up; the decision is shared so all four warps leave together.
// gs_a is the activations' global scale, passed by value: the caller knows
// when it is final.
__device__ bool run_epilogue(const Phase& P, float gs_a, int E, const Tables& tb, Barriers* bars,
                             uint32_t tmem, Pipe& pp, volatile int* abort, float& amax,
                             int* s_ok, int* s_last, const YReduce* yr = nullptr) {
  const GemmArgs& args = *P.a;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int q = warp & 3;                      // TMEM lane quarter
  const int row_in_tile = q * 32 + lane;
  const uint32_t t_row = tmem + (static_cast<uint32_t>(q * 32) << 16);
  const bool lead = warp == 2 && lane == 0;
  WorkIter it;
  it.init(P.total_tiles, P.k_stages, gridDim.x, blockIdx.x, P.whole_tiles);
  int tile, s0, s1;
  bool have = it.next(tile, s0, s1);
  // the weight scales of the next tile are loaded one tile ahead; the up
  // half of L1 has its own scale when the checkpoint gives one
  const float* gs_b_up = args.gs_b_up != nullptr ? args.gs_b_up : args.gs_b;
  // L2 with a static intermediate scale: the activation scale is per expert
  const bool mid_alpha = args.mode == 2 && args.gs_mid != nullptr;
  int e0 = have ? decode_tile(tile, P.prefix, tb.mtiles, E).e : 0;
  float gs_b = have ? __ldg(args.gs_b + e0) : 0.0f;
  float gs_u = have ? __ldg(gs_b_up + e0) : 0.0f;
  float gs_m = have && mid_alpha ? __ldg(args.gs_mid + e0) : gs_a;
  while (have) {
    const TileInfo ti = decode_tile(tile, P.prefix, tb.mtiles, E);
    const float alpha = __fmul_rn(gs_m, gs_b);
    const float alpha_u = __fmul_rn(gs_m, gs_u);
    int n_tile, n_s0, n_s1;
    const bool n_have = it.next(n_tile, n_s0, n_s1);
    if (n_have) {
      const int ne = decode_tile(n_tile, P.prefix, tb.mtiles, E).e;
      gs_b = __ldg(args.gs_b + ne);
      gs_u = __ldg(gs_b_up + ne);
      if (mid_alpha) gs_m = __ldg(args.gs_mid + ne);
    }
    // one thread waits (bounded) and the decision is shared, so the four
    // epilogue warps always take the same path through the named barriers
    if (lead) *s_ok = mbar_wait(&bars->acc_full, pp.acc_phase, args.status, abort) ? 1 : 0;
    epi_bar();
    if (!*s_ok) return false;
    tc_fence_after();
    const int tile_valid =
        checked_rows(args, tb.off[ti.e] + ti.mt * kBM, tb.cnt[ti.e] - ti.mt * kBM);
    const bool valid = row_in_tile < tile_valid;
    const int64_t row = tb.off[ti.e] + ti.mt * kBM + row_in_tile;
    const int col0 = ti.nt * (args.mode == 1 ? 128 : kBN);
    if (s0 == 0 && s1 == P.k_stages) {
      // whole tile in this CTA: epilogue straight from TMEM.  Valid rows of
      // this warp's quarter (warp-uniform):
      const int nv_w = min(32, max(0, tile_valid - q * 32));
      const int64_t qrow0 = tb.off[ti.e] + ti.mt * kBM + q * 32;
      if (args.mode == 1 && nv_w > 0 && nv_w <= kNarrowRows) {
        // few rows (decode): each row's columns spread over the lanes
        for (int c = 0; c < 4; ++c) {
          float g[32], u[32];
          tmem_ld_f32(t_row + c * 32, g);
          tmem_ld_f32(t_row + 128 + c * 32, u);
          for (int r = 0; r < nv_w; ++r)
            epi_l1_1(from_lane_column(g, r), from_lane_column(u, r), alpha, alpha_u, qrow0 + r,
                     col0 + c * 32 + lane, args, amax);
        }
      } else if (nv_w > 0) {
        if (args.mode == 1) {
          for (int c = 0; c < 4; ++c) {
            float g[32], u[32];
            tmem_ld_f32(t_row + c * 32, g);
            tmem_ld_f32(t_row + 128 + c * 32, u);
            if (valid) epi_l1(g, u, alpha, alpha_u, row, col0 + c * 32, args, amax);
          }
        } else {
          for (int c = 0; c < 8; ++c) {
            float a[32];
            tmem_ld_f32(t_row + c * 32, a);
            if (valid) epi_l2(a, alpha, row, col0 + c * 32, args);
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->acc_empty);
      if (yr != nullptr) y_after_tile(*yr, ti, tb, args);
      if (args.mode == 1 && args.gs_mid != nullptr && args.mid_in_epilogue)
        requant_own_tile(args, ti, tb);
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
      const int64_t u_first = static_cast<int64_t>(tile) * P.k_stages;
      const int c_first = it.owner(u_first);
      const int c_last = it.owner(u_first + P.k_stages - 1);
      if (lead) *s_last = atomicAdd(&args.counters[tile], 1) == c_last - c_first;
      epi_bar();
      if (*s_last) {
        // every piece has landed: sum them in ascending K order.  The valid
        // rows' 4-column groups are spread over all 128 epilogue threads and
        // the pieces are loaded four at a time, so the fixup is not a chain
        // of dependent L2 round trips on the few threads that own rows.
        __threadfence();
        if (lead) args.counters[tile] = 0;
        const int n_valid = min(kBM, tile_valid);
        const int groups = args.mode == 1 ? 32 : 64;   // float4 groups per row
        const int etid = threadIdx.x - 64;
        const int64_t row0 = tb.off[ti.e] + ti.mt * kBM;
        for (int wi = etid; wi < n_valid * groups; wi += 128) {
          const int r = wi / groups, g4 = wi - r * groups;
          float4 a = make_float4(0.f, 0.f, 0.f, 0.f), b = a;
          for (int cc0 = c_first; cc0 <= c_last; cc0 += 4) {
            float4 va[4], vb[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              if (cc0 + j <= c_last) {
                const float* p = args.partials +
                                 (static_cast<size_t>(it.slot(cc0 + j, tile)) * kBM + r) * kBN +
                                 g4 * 4;
                va[j] = __ldcg(reinterpret_cast<const float4*>(p));
                if (args.mode == 1) vb[j] = __ldcg(reinterpret_cast<const float4*>(p + 128));
              }
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              if (cc0 + j <= c_last) {
                add4(a, va[j]);
                if (args.mode == 1) add4(b, vb[j]);
              }
            }
          }
          if (args.mode == 1)
            epi_l1_4(a, b, alpha, alpha_u, row0 + r, col0 + g4 * 4, args, amax);
          else
            epi_l2_4(a, alpha, row0 + r, col0 + g4 * 4, args);
        }
        if (yr != nullptr) y_after_tile(*yr, ti, tb, args);
        if (args.mode == 1 && args.gs_mid != nullptr && args.mid_in_epilogue)
          requant_own_tile(args, ti, tb);
      }
    }
    pp.acc_phase ^= 1u;
    tile = n_tile;
    s0 = n_s0;
    s1 = n_s1;
    have = n_have;
  }
  return true;
}

// Lane groups of four (lanes 4g..4g+3) exchange 8-word blocks so that rows
// leave in 128-byte pieces: before, lane 4g+p holds row 4g+p as blocks
// v[0..3]; after, lane 4g+p holds block p of rows 4g+0..3 in v[0..3].  Two
// xor-shuffle rounds (lane bit 1, then bit 0), each sending the half of the
// blocks the partner keeps; one shuffle per word.
__device__ __forceinline__ void quad_transpose(uint32_t (&v)[4][8]) {
  const int lane = threadIdx.x & 31;
  const bool hi = (lane & 2) != 0, lo = (lane & 1) != 0;
#pragma unroll
  for (int b = 0; b < 2; ++b)
#pragma unroll
    for (int w = 0; w < 8; ++w) {
      const uint32_t r = __shfl_xor_sync(0xffffffffu, hi ? v[b][w] : v[b + 2][w], 2);
      if (hi) v[b][w] = r;
      else v[b + 2][w] = r;
    }
#pragma unroll
  for (int rb = 0; rb < 2; ++rb)
#pragma unroll
    for (int w = 0; w < 8; ++w) {
      const uint32_t r = __shfl_xor_sync(0xffffffffu, lo ? v[2 * rb][w] : v[2 * rb + 1][w], 1);
      if (lo) v[2 * rb][w] = r;
      else v[2 * rb + 1][w] = r;
    }
}

// After quad_transpose: lane 4g+p stores its block p of rows 4g+r (r = 0..3)
// at base + (row0 + 4g + r) * stride + 32 p bytes, rows past n_valid skipped.
// One instruction writes 8 rows x 128 contiguous bytes.
__device__ __forceinline__ void quad_store(uint32_t (&v)[4][8], uint8_t* base, int64_t row0,
                                           int64_t stride, int q_row0, int n_valid) {
  const int lane = threadIdx.x & 31;
  const int g = lane >> 2, p = lane & 3;
#pragma unroll
  for (int r = 0; r < 4; ++r)
    if (q_row0 + 4 * g + r < n_valid)
      st_global_v8_b32(base + (row0 + 4 * g + r) * stride + 32 * p, v[r]);
}

// grouped_gemm_kernel<true>, where every CTA takes whole tiles: two epilogue sets,
// warps 2..5 (set 0) and 10..13 (set 1), each one warp per TMEM lane
// quarter, take half of every tile's output columns (L1: h columns
// [64 set, 64 set + 64), from gate columns 64 set + c and up columns
// 128 + 64 set + c; L2: columns [128 set, 128 set + 128)).  The arithmetic
// is epi_l1's and epi_l2's; without taps the rows are regrouped by
// quad_transpose and stored 128 bytes per row piece (the row-per-lane stores
// of the tapped path make 32 separate 32-byte requests per instruction).
// acc_empty counts the 8 warps.
// One tile's share of an epilogue set (see run_epilogue_half): rows
// row0 + [0, 128) of which n_valid are valid, output column tile nt; this
// warp's TMEM lanes at t_row.  release() hands the accumulator back: on the
// untapped paths as soon as this warp's share is in registers (h, or the
// 16-bit slot rows), so that the regrouping and the stores overlap the next
// tile's MMAs; elsewhere after the stores.
template <typename Release>
__device__ __forceinline__ void epi_tile_half(const GemmArgs& args, int nt, int n_valid,
                                              int64_t row0, float alpha, float alpha_u,
                                              uint32_t t_row, int set, float& amax,
                                              Release release) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int q = warp & 3;
  const int row_in_tile = q * 32 + lane;
  const bool grouped = args.tap == nullptr;
  n_valid = checked_rows(args, row0, n_valid);
  const bool valid = row_in_tile < n_valid;
  const int64_t row = row0 + row_in_tile;
  const int nv_w = min(32, max(0, n_valid - q * 32));
  if (nv_w == 0) {
    release();
  } else if (args.mode == 1 && nv_w <= kNarrowRows) {
    // few rows: each row's columns spread over the lanes, as in epi_l1_1
    for (int c = 0; c < 2; ++c) {
      float g[32], u[32];
      tmem_ld_f32(t_row + set * 64 + c * 32, g);
      tmem_ld_f32(t_row + 128 + set * 64 + c * 32, u);
      for (int r = 0; r < nv_w; ++r)
        epi_l1_1(from_lane_column(g, r), from_lane_column(u, r), alpha, alpha_u,
                 row0 + q * 32 + r, nt * 128 + set * 64 + c * 32 + lane, args, amax);
    }
    release();
  } else if (args.mode == 1 && grouped) {
    uint8_t* base = reinterpret_cast<uint8_t*>(args.out) + (nt * 128 + set * 64) * sizeof(float);
    uint32_t v[2][4][8];
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      float g[32], u[32];
      tmem_ld_f32(t_row + set * 64 + c * 32, g);
      tmem_ld_f32(t_row + 128 + set * 64 + c * 32, u);
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const float h = __fmul_rn(silu_f(__fmul_rn(alpha, g[j])), __fmul_rn(alpha_u, u[j]));
        if (valid) amax = fmaxf(amax, fabsf(h));
        v[c][j / 8][j % 8] = __float_as_uint(h);
      }
    }
    release();
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      quad_transpose(v[c]);
      quad_store(v[c], base + c * 32 * sizeof(float), row0 + q * 32,
                 static_cast<int64_t>(args.I) * sizeof(float), q * 32, n_valid);
    }
  } else if (args.mode == 1) {
    for (int c = 0; c < 2; ++c) {
      float g[32], u[32];
      tmem_ld_f32(t_row + set * 64 + c * 32, g);
      tmem_ld_f32(t_row + 128 + set * 64 + c * 32, u);
      if (valid) epi_l1(g, u, alpha, alpha_u, row, nt * 128 + set * 64 + c * 32, args, amax);
    }
    release();
  } else if (grouped && args.out_dtype != 1) {
    // 16-bit slot rows: 64 columns (128 bytes) per round
    const bool half = args.out_dtype == 2;
    uint8_t* base = reinterpret_cast<uint8_t*>(args.out) + (nt * kBN + set * 128) * 2;
    float big = 0.0f;
    uint32_t v[2][4][8];
#pragma unroll
    for (int c = 0; c < 2; ++c) {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        float a[32];
        tmem_ld_f32(t_row + set * 128 + c * 64 + h * 32, a);
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const float x0 = __fmul_rn(alpha, a[2 * j]), x1 = __fmul_rn(alpha, a[2 * j + 1]);
          big = fmaxf(big, fmaxf(fabsf(x0), fabsf(x1)));
          v[c][2 * h + j / 8][j % 8] = half ? pack_f16x2(x0, x1) : pack_bf16x2(x0, x1);
        }
      }
    }
    release();
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      quad_transpose(v[c]);
      quad_store(v[c], base + c * 64 * 2, row0 + q * 32, static_cast<int64_t>(args.N) * 2, q * 32,
                 n_valid);
    }
    if (half && valid && !(big <= kF16Max)) record_status(args.status, kErrRange);
  } else if (grouped) {
    uint8_t* base = reinterpret_cast<uint8_t*>(args.out) + (nt * kBN + set * 128) * 4;
    for (int c = 0; c < 4; ++c) {
      float a[32];
      tmem_ld_f32(t_row + set * 128 + c * 32, a);
      uint32_t v[4][8];
#pragma unroll
      for (int j = 0; j < 32; ++j) v[j / 8][j % 8] = __float_as_uint(__fmul_rn(alpha, a[j]));
      quad_transpose(v);
      quad_store(v, base + c * 32 * 4, row0 + q * 32, static_cast<int64_t>(args.N) * 4, q * 32,
                 n_valid);
    }
    release();
  } else {
    for (int c = 0; c < 4; ++c) {
      float a[32];
      tmem_ld_f32(t_row + set * 128 + c * 32, a);
      if (valid) epi_l2(a, alpha, row, nt * kBN + set * 128 + c * 32, args);
    }
    release();
  }
}

// With a static intermediate scale (two-set epilogues): this set requantises
// the 64 h columns of the tile it has just stored, for the tile's valid rows,
// with the expert's gs_mid: four 16-element blocks and one staged scale word
// per row, re-read from L2 once every store of the set has been made (one
// row per thread; the same block arithmetic as every other quantisation).
// The L1 epilogue has the slack for it: a tile's MMAs take far longer.
__device__ __noinline__ void requant_set_cols(const GemmArgs& args, int nt, int n_valid,
                                              int64_t row0, float gs, int set) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (set == 0)
    asm volatile("bar.sync 3, 128;" ::: "memory");
  else
    asm volatile("bar.sync 4, 128;" ::: "memory");
  n_valid = checked_rows(args, row0, n_valid);
  const int r = (warp & 3) * 32 + lane;
  if (r < n_valid) {
    const float denom = __fmul_rn(6.0f, gs);
    const int I = args.I;
    const int k_atoms = (I + kStageK - 1) / kStageK * 4;
    const int64_t row = row0 + r;
    const int g0 = nt * 8 + set * 4;
    uint32_t word = 0;
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      const float4* p = reinterpret_cast<const float4*>(args.out + row * I + (g0 + b) * 16);
      float v[16];
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const float4 f = __ldcg(p + c);
        v[4 * c] = f.x; v[4 * c + 1] = f.y; v[4 * c + 2] = f.z; v[4 * c + 3] = f.w;
      }
      uint32_t packed[2];
      word |= quant_block16(v, gs, denom, packed) << (8 * b);
      *reinterpret_cast<uint2*>(args.mid_q + row * (I / 2) + (g0 + b) * 8) =
          make_uint2(packed[0], packed[1]);
    }
    *reinterpret_cast<uint32_t*>(args.mid_sf + staged_offset(row, g0, k_atoms)) = word;
  }
}

__device__ bool run_epilogue_half(const Phase& P, float gs_a, int E, const Tables& tb,
                                  Barriers* bars, uint32_t tmem, volatile int* abort,
                                  float& amax) {
  const GemmArgs& args = *P.a;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int set = warp >= kEpi2Warp0 ? 1 : 0;
  const uint32_t t_row = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
  const float* gs_b_up = args.gs_b_up != nullptr ? args.gs_b_up : args.gs_b;
  const bool mid_alpha = args.mode == 2 && args.gs_mid != nullptr;
  WorkIter it;
  it.init(P.total_tiles, P.k_stages, gridDim.x, blockIdx.x, P.whole_tiles);
  uint32_t acc_phase = 0;
  int tile, s0, s1;
  while (it.next(tile, s0, s1)) {
    const TileInfo ti = decode_tile(tile, P.prefix, tb.mtiles, E);
    const float gs_m = mid_alpha ? __ldg(args.gs_mid + ti.e) : gs_a;
    const float alpha = __fmul_rn(gs_m, __ldg(args.gs_b + ti.e));
    const float alpha_u = __fmul_rn(gs_m, __ldg(gs_b_up + ti.e));
    if (!mbar_wait(&bars->acc_full, acc_phase, args.status, abort)) return false;
    tc_fence_after();
    epi_tile_half(args, ti.nt, tb.cnt[ti.e] - ti.mt * kBM, tb.off[ti.e] + ti.mt * kBM, alpha,
                  alpha_u, t_row, set, amax, [&]() {
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&bars->acc_empty);
                  });
    acc_phase ^= 1u;
  }
  return true;
}

// The two epilogue sets' per-CTA amax of h -> amax_partial[blockIdx.x].
__device__ void publish_amax_half(float amax, float* s_amax, float* out) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  amax = warp_max(amax);
  if (lane == 0) s_amax[(warp >= kEpi2Warp0 ? 4 : 0) + (warp & 3)] = amax;
  asm volatile("bar.sync 2, 256;" ::: "memory");
  if (warp == 2 && lane == 0) {
    float m = 0.0f;
    for (int i = 0; i < 8; ++i) m = fmaxf(m, s_amax[i]);
    out[blockIdx.x] = m;
  }
}

// Per-CTA amax of the L1 epilogue -> amax_partial[blockIdx.x] (epilogue warps).
__device__ void publish_amax(float amax, float* s_amax, float* out) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  amax = warp_max(amax);
  if (lane == 0) s_amax[warp & 3] = amax;
  epi_bar();
  if (warp == 2 && lane == 0)
    out[blockIdx.x] = fmaxf(fmaxf(s_amax[0], s_amax[1]), fmaxf(s_amax[2], s_amax[3]));
}

// ---------------------------------------------------------- kernel set-up --
__device__ void load_tables(Tables& tb, const GemmArgs& a1, int n_tiles2) {
  const int E = a1.E;
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    const int c = a1.expert_counts[e];
    tb.cnt[e] = c;
    tb.off[e] = a1.expert_offsets[e];
    tb.mtiles[e] = (c + kBM - 1) / kBM;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int p1 = 0, p2 = 0, d = 0;
    for (int e = 0; e < E; ++e) {
      tb.prefix1[e] = p1;
      tb.prefix2[e] = p2;
      tb.dense[e] = d;
      p1 += tb.mtiles[e] * a1.n_tiles;
      p2 += tb.mtiles[e] * n_tiles2;
      d += tb.cnt[e];
    }
    tb.prefix1[E] = p1;
    tb.prefix2[E] = p2;
    tb.dense[E] = d;
  }
}

__device__ uint32_t setup_cta(Barriers* bars, const CUtensorMap* m0, const CUtensorMap* m1,
                              const CUtensorMap* m2, const CUtensorMap* m3,
                              uint32_t acc_empty_arrivals = 4, uint32_t sf_arrivals = 4) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (warp == 0 && lane == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&bars->full[s], 1);
      mbar_init(&bars->empty[s], 1);
      mbar_init(&bars->sf_full[s], sf_arrivals);
    }
    mbar_init(&bars->acc_full, 1);
    mbar_init(&bars->acc_empty, acc_empty_arrivals);
    mbar_init(&bars->drain, 1);
    bars->abort = 0;
    fence_mbarrier_init();
    prefetch_tensormap(m0);
    prefetch_tensormap(m1);
    if (m2 != nullptr) prefetch_tensormap(m2);
    if (m3 != nullptr) prefetch_tensormap(m3);
  }
  if (warp == 1) {
    tmem_alloc(&bars->tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  return bars->tmem_base;
}

// The MMA thread makes sure every MMA it issued has finished; then the
// allocating warp releases TMEM.
__device__ void teardown_cta(Barriers* bars, uint32_t tmem) {
  tc_fence_before();
  __syncthreads();
  if ((threadIdx.x >> 5) == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

__device__ void mma_drain(Barriers* bars, int* status) {
  tc_commit(&bars->drain);
  mbar_wait(&bars->drain, 0, status, nullptr);
}

__device__ __forceinline__ uint8_t* aligned_smem(uint8_t* raw) {
  const uint32_t a = smem_u32(raw);
  return raw + ((1024u - (a & 1023u)) & 1023u);
}

// ------------------------------------------------------------- kernels --
template <bool kHalf>
__global__ void __launch_bounds__(kHalf ? kThreadsHalf : kThreadsSt, 1) grouped_gemm_kernel(
    const __grid_constant__ AMaps map_a, const __grid_constant__ CUtensorMap map_b,
    const GemmArgs args) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = aligned_smem(smem_raw);
  Barriers* bars = reinterpret_cast<Barriers*>(smem + kOffBar);
  __shared__ Tables tb;
  __shared__ float s_amax[8];
  __shared__ int s_last, s_ok;

  // the next kernel may be scheduled; this one's prologue (barriers, TMEM,
  // tensor maps) touches no memory of the kernels before it
  pdl_trigger();
  const uint32_t tmem = setup_cta(bars, &map_a.full, &map_b, &map_a.small, nullptr, kHalf ? 8u : 4u);
  pdl_wait();
  load_tables(tb, args, args.n_tiles);
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  volatile int* abort = &bars->abort;
  Phase P = make_phase(args, &map_a, &map_b, tb.prefix1, args.E);
  P.whole_tiles = kHalf;
  Pipe pp;
  if (warp == 0) {
    if (lane == 0) {
      run_producer(P, args.E, tb, bars, smem, pp, abort, nullptr);
      drain_producer(bars, pp, args.status);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      run_mma<true>(P, bars, smem, tmem, pp, abort);
      mma_drain(bars, args.status);
    }
  } else if (warp >= kSfWarp0 && warp < kEpi2Warp0) {
    run_sf_writer(P, bars, smem, tmem, pp, abort);
  } else if constexpr (kHalf) {
    float amax = 0.0f;
    run_epilogue_half(P, __ldcg(args.gs_a), args.E, tb, bars, tmem, abort, amax);
    if (args.mode == 1) publish_amax_half(amax, s_amax, args.amax_partial);
  } else {
    float amax = 0.0f;
    run_epilogue(P, __ldcg(args.gs_a), args.E, tb, bars, tmem, pp, abort, amax, &s_ok, &s_last);
    if (args.mode == 1) publish_amax(amax, s_amax, args.amax_partial);
  }
  teardown_cta(bars, tmem);
}

// ----------------------------------------------------------- CTA pairs --
// grouped_gemm_pair_kernel: the whole-tile GEMM over clusters of two CTAs.
// One MMA (tcgen05.mma.cta_group::2, M = 256, N = 256, K = 64), issued by
// the even CTA, computes two m-tiles of one expert against one 256-row B
// tile: CTA r holds its own m-tile of A (128 rows) and B rows
// [128 r, 128 r + 128) of the tile in its shared memory, and its 128 x 256
// accumulator in its TMEM.  Halving B per CTA halves the B traffic into
// each SM and makes a stage 38 KB, so five stages fit where a one-CTA tile
// holds four.  Each CTA loads its own operands, its own A scales and all
// 256 rows of B scales (its TMEM gets the scale layout of the one-CTA
// kernel); its four scale writers arrive on the even CTA's sf_full, which
// therefore means "both CTAs' loads have landed and both CTAs' scales are in
// TMEM" and is the one barrier the MMA thread waits for.  The MMA thread's
// commits arrive on the stage's empty barrier and on acc_full in both CTAs;
// both CTAs' epilogue warps (8 each) arrive on the even CTA's acc_empty.
// Pair tiles are (expert, n-tile, m-tile pair); an expert with an odd
// number of m-tiles leaves the odd CTA of its last pair without rows: it
// loads the even CTA's m-tile again (always in bounds) and stores nothing.
constexpr int kStagesP = 5;
constexpr int kBHalfBytes = 128 * kRowBytes;                             // 16384
constexpr uint32_t kStageTxP = kABytes + kBHalfBytes + kSfaBytes + kSfbBytes;
constexpr int kOffAP = 0;
constexpr int kOffBP = kOffAP + kStagesP * kABytes;
constexpr int kOffSfaP = kOffBP + kStagesP * kBHalfBytes;
constexpr int kOffSfbP = kOffSfaP + kStagesP * kSfaBytes;
constexpr int kOffBarP = kOffSfbP + kStagesP * kSfbBytes;
constexpr int kSmemBytesP = kOffBarP + 256 + 1024;
// TMEM: accumulator columns [0, 256); B scales 32 columns per stage from
// 256, A scales 16 per stage from 416 (every tcgen05.st at a multiple of its
// width; MMA scale addresses at multiples of 8 and 4)
constexpr uint32_t kTmemSfbP = 256;
constexpr uint32_t kTmemSfaP = kTmemSfbP + kStagesP * 32;
static_assert(kTmemSfaP + kStagesP * 16 <= kTmemCols, "pair TMEM columns");

struct BarriersP {
  uint64_t full[kStagesP];      // this CTA's loads of the stage
  uint64_t empty[kStagesP];     // the pair's MMAs on the stage are done
  uint64_t sf_full[kStagesP];   // even CTA: both CTAs' scales written (8 warps)
  uint64_t acc_full;            // the tile's MMAs are done
  uint64_t acc_empty;           // even CTA: both CTAs' epilogues released (16 warps)
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
};
static_assert(sizeof(BarriersP) <= 256, "pair barriers");

struct PairTables {
  int prefix[kMaxExperts + 1];  // pair-tile prefix
  int pmt[kMaxExperts];         // m-tile pairs per expert
  int mtiles[kMaxExperts];
  int off[kMaxExperts];
  int cnt[kMaxExperts];
};

__device__ void load_pair_tables(PairTables& tb, const GemmArgs& a) {
  const int E = a.E;
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    const int c = a.expert_counts[e];
    tb.cnt[e] = c;
    tb.off[e] = a.expert_offsets[e];
    tb.mtiles[e] = (c + kBM - 1) / kBM;
    tb.pmt[e] = (tb.mtiles[e] + 1) / 2;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int p = 0;
    for (int e = 0; e < E; ++e) {
      tb.prefix[e] = p;
      p += tb.pmt[e] * a.n_tiles;
    }
    tb.prefix[E] = p;
  }
  __syncthreads();
}

// This CTA's m-tile of pair tile t and whether it holds rows.
struct PairTile {
  int e, nt, m;
  bool has_rows;
};

__device__ __forceinline__ PairTile pair_tile(int t, const PairTables& tb, int E, uint32_t rank) {
  const TileInfo ti = decode_tile(t, tb.prefix, tb.pmt, E);
  PairTile p;
  p.e = ti.e;
  p.nt = ti.nt;
  p.m = 2 * ti.mt + static_cast<int>(rank);
  p.has_rows = p.m < tb.mtiles[ti.e];
  return p;
}

__device__ bool run_producer_pair(const GemmArgs& args, const PairTables& tb, const AMaps* map_a,
                                  const CUtensorMap* map_b, BarriersP* bars, uint8_t* smem,
                                  uint32_t rank, volatile int* abort, int& issued, int& stage,
                                  uint32_t& phase) {
  const int E = args.E;
  const int k_stages = (args.K + kStageK - 1) / kStageK;
  const int k_atoms = k_stages * 4;
  // Normal L2 priority for both operands.  An expert's A tile is reused by
  // its n-tiles over several waves and its B tile by the m-tile pairs of one
  // wave; with A marked evict_last, the A lines of experts already done (the
  // slot activations of a 16k-token batch are 4x the L2) crowded out the
  // lines in use, and the L1 GEMM read 2.3x its operand bytes from DRAM
  // (4.52 GB against 1.93 GB at T = 16384).
  const uint64_t pol_a = policy_evict_normal();
  const uint64_t pol_b = pol_a;
  if (args.ready_flag != nullptr &&
      !wait_flag(args.ready_flag, args.ready_value, args.status, abort, args.ready_limit_ns))
    return false;
  const int n_clusters = gridDim.x >> 1;
  for (int t = blockIdx.x >> 1; t < tb.prefix[E]; t += n_clusters) {
    const PairTile pt = pair_tile(t, tb, E, rank);
    const int m = pt.has_rows ? pt.m : pt.m - 1;            // the even CTA's m-tile
    const int a_row = tb.off[pt.e] + m * kBM;
    int b_row0, b_row1;
    if (args.mode == 1) {
      b_row0 = pt.e * args.N + pt.nt * 128;
      b_row1 = b_row0 + args.I;
    } else {
      b_row0 = pt.e * args.N + pt.nt * kBN;
      b_row1 = b_row0 + 128;
    }
    const int b_tile = ((rank == 0 ? b_row0 : b_row1) / 128) * k_stages;
    const uint8_t* sfb0 = args.b_sf + (static_cast<size_t>(b_row0 / 128) * k_atoms) * kSfAtomBytes;
    const uint8_t* sfb1 = args.b_sf + (static_cast<size_t>(b_row1 / 128) * k_atoms) * kSfAtomBytes;
    const uint8_t* sfa = args.a_sf + (static_cast<size_t>(a_row / 128) * k_atoms) * kSfAtomBytes;
    for (int ks = 0; ks < k_stages; ++ks) {
      if (!mbar_wait(&bars->empty[stage], phase ^ 1u, args.status, abort)) return false;
      uint64_t* full = &bars->full[stage];
      mbar_arrive_expect_tx(full, kStageTxP);
      const size_t koff = static_cast<size_t>(ks) * 4 * kSfAtomBytes;
      tma_load_3d(smem + kOffBP + stage * kBHalfBytes, map_b, 0, 0, b_tile + ks, full, pol_b);
      bulk_load(smem + kOffSfbP + stage * kSfbBytes, sfb0 + koff, kSfaBytes, full, pol_b);
      bulk_load(smem + kOffSfbP + stage * kSfbBytes + kSfaBytes, sfb1 + koff, kSfaBytes, full,
                pol_b);
      tma_load_2d(smem + kOffAP + stage * kABytes, &map_a->full, ks * kRowBytes, a_row, full,
                  pol_a);
      bulk_load(smem + kOffSfaP + stage * kSfaBytes, sfa + koff, kSfaBytes, full, pol_a);
      ++issued;
      if (++stage == kStagesP) {
        stage = 0;
        phase ^= 1u;
      }
    }
  }
  return true;
}

__device__ bool run_mma_pair(const GemmArgs& args, const PairTables& tb, BarriersP* bars,
                             uint8_t* smem, uint32_t tmem, volatile int* abort) {
  const int E = args.E;
  const int k_stages = (args.K + kStageK - 1) / kStageK;
  const int k_blocks = args.K / 64;
  const uint32_t idesc = idesc_mxf4nvf4(2 * kBM, kBN);
  const int n_clusters = gridDim.x >> 1;
  int stage = 0;
  uint32_t phase = 0, acc_phase = 0;
  for (int t = blockIdx.x >> 1; t < tb.prefix[E]; t += n_clusters) {
    if (!mbar_wait(&bars->acc_empty, acc_phase ^ 1u, args.status, abort)) return false;
    tc_fence_after();
    for (int ks = 0; ks < k_stages; ++ks) {
      if (!mbar_wait(&bars->sf_full[stage], phase, args.status, abort)) return false;
      tc_fence_after();
      const uint32_t sfa_t = tmem + kTmemSfaP + stage * 16;
      const uint32_t sfb_t = tmem + kTmemSfbP + stage * 32;
      const uint32_t a_base = smem_u32(smem + kOffAP + stage * kABytes);
      const uint32_t b_base = smem_u32(smem + kOffBP + stage * kBHalfBytes);
      const int nkb = min(4, k_blocks - ks * 4);
      for (int kb = 0; kb < nkb; ++kb) {
        const uint64_t adesc = smem_desc(a_base + kb * 32, 16, 1024, 2);
        const uint64_t bdesc = smem_desc(b_base + kb * 32, 16, 1024, 2);
        mma_mxf4nvf4_pair(tmem, adesc, bdesc, idesc, sfa_t + kb * 4, sfb_t + kb * 8,
                          (ks != 0 || kb != 0) ? 1u : 0u);
      }
      tc_commit_pair(&bars->empty[stage], 3);
      if (++stage == kStagesP) {
        stage = 0;
        phase ^= 1u;
      }
    }
    tc_commit_pair(&bars->acc_full, 3);
    acc_phase ^= 1u;
  }
  return true;
}

// Scale writers of a pair CTA: as run_sf_writer, into this CTA's TMEM, then
// an arrival on the even CTA's sf_full.
__device__ bool run_sf_writer_pair(const GemmArgs& args, const PairTables& tb, BarriersP* bars,
                                   const uint8_t* smem, uint32_t tmem, volatile int* abort) {
  const int E = args.E;
  const int lane = threadIdx.x & 31;
  const uint32_t q = (threadIdx.x >> 5) & 3;
  const uint32_t lane_base = tmem + ((q * 32u) << 16);
  const int k_stages = (args.K + kStageK - 1) / kStageK;
  const int n_clusters = gridDim.x >> 1;
  int stage = 0;
  uint32_t phase = 0;
  for (int t = blockIdx.x >> 1; t < tb.prefix[E]; t += n_clusters) {
    for (int ks = 0; ks < k_stages; ++ks) {
      if (!mbar_wait(&bars->full[stage], phase, args.status, abort)) return false;
      const uint4* sa = reinterpret_cast<const uint4*>(smem + kOffSfaP + stage * kSfaBytes) + lane;
      const uint4* sb = reinterpret_cast<const uint4*>(smem + kOffSfbP + stage * kSfbBytes) + lane;
      uint32_t a[16], b[32];
#pragma unroll
      for (int kb = 0; kb < 4; ++kb) {
        const uint4 v = sa[kb * 32];
        a[4 * kb] = v.x; a[4 * kb + 1] = v.y; a[4 * kb + 2] = v.z; a[4 * kb + 3] = v.w;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const uint4 u = sb[h * 128 + kb * 32];
          b[8 * kb + 4 * h] = u.x; b[8 * kb + 4 * h + 1] = u.y;
          b[8 * kb + 4 * h + 2] = u.z; b[8 * kb + 4 * h + 3] = u.w;
        }
      }
      tmem_st_32x32b_x32(lane_base + kTmemSfbP + stage * 32, b);
      tmem_st_32x32b_x16(lane_base + kTmemSfaP + stage * 16, a);
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(map_shared_rank(smem_u32(&bars->sf_full[stage]), 0));
      if (++stage == kStagesP) {
        stage = 0;
        phase ^= 1u;
      }
    }
  }
  return true;
}

// kMidOwn: L1 with a static intermediate scale requantised by the epilogue
// sets (a separate instantiation, so that the common path keeps its
// register allocation).
template <bool kMidOwn>
__device__ bool run_epilogue_pair(const GemmArgs& args, const PairTables& tb, BarriersP* bars,
                                  uint32_t tmem, uint32_t rank, volatile int* abort,
                                  float& amax) {
  const int E = args.E;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int set = warp >= kEpi2Warp0 ? 1 : 0;
  const uint32_t t_row = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
  const float gs_a = __ldcg(args.gs_a);
  const float* gs_b_up = args.gs_b_up != nullptr ? args.gs_b_up : args.gs_b;
  const bool mid_alpha = args.mode == 2 && args.gs_mid != nullptr;
  const uint32_t acc_empty0 = map_shared_rank(smem_u32(&bars->acc_empty), 0);
  const int n_clusters = gridDim.x >> 1;
  uint32_t acc_phase = 0;
  for (int t = blockIdx.x >> 1; t < tb.prefix[E]; t += n_clusters) {
    const PairTile pt = pair_tile(t, tb, E, rank);
    const float gs_m = mid_alpha ? __ldg(args.gs_mid + pt.e) : gs_a;
    const float alpha = __fmul_rn(gs_m, __ldg(args.gs_b + pt.e));
    const float alpha_u = __fmul_rn(gs_m, __ldg(gs_b_up + pt.e));
    if (!mbar_wait(&bars->acc_full, acc_phase, args.status, abort)) return false;
    tc_fence_after();
    const int n_valid = pt.has_rows ? tb.cnt[pt.e] - pt.m * kBM : 0;
    epi_tile_half(args, pt.nt, n_valid, tb.off[pt.e] + pt.m * kBM, alpha, alpha_u, t_row, set,
                  amax, [&]() {
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive_cluster(acc_empty0);
                  });
    if (kMidOwn)
      requant_set_cols(args, pt.nt, n_valid, tb.off[pt.e] + pt.m * kBM,
                       __ldg(args.gs_mid + pt.e), set);
    acc_phase ^= 1u;
  }
  return true;
}

template <bool kMidOwn>
__global__ void __launch_bounds__(kThreadsHalf, 1) grouped_gemm_pair_kernel(
    const __grid_constant__ AMaps map_a, const __grid_constant__ CUtensorMap map_b,
    const GemmArgs args) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = aligned_smem(smem_raw);
  BarriersP* bars = reinterpret_cast<BarriersP*>(smem + kOffBarP);
  __shared__ PairTables tb;
  __shared__ float s_amax[8];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();

  pdl_trigger();
  if (warp == 0 && lane == 0) {
    for (int s = 0; s < kStagesP; ++s) {
      mbar_init(&bars->full[s], 1);
      mbar_init(&bars->empty[s], 1);
      mbar_init(&bars->sf_full[s], 8);
    }
    mbar_init(&bars->acc_full, 1);
    mbar_init(&bars->acc_empty, 16);
    mbar_init(&bars->drain, 1);
    bars->abort = 0;
    fence_mbarrier_init();
    prefetch_tensormap(&map_a.full);
    prefetch_tensormap(&map_b);
  }
  if (warp == 1) {
    tmem_alloc_pair(&bars->tmem_base, kTmemCols);
    tmem_relinquish_pair();
  }
  // both CTAs' barriers are initialised before any remote arrival
  tc_fence_before();
  cluster_sync();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  volatile int* abort = &bars->abort;
  pdl_wait();
  load_pair_tables(tb, args);

  if (warp == 0) {
    if (lane == 0) {
      int issued = 0, stage = 0;
      uint32_t phase = 0;
      run_producer_pair(args, tb, &map_a, &map_b, bars, smem, rank, abort, issued, stage, phase);
      // no copy into this CTA's shared memory is in flight at exit
      const int tail = issued < kStagesP ? issued : kStagesP;
      for (int i = 0; i < tail; ++i) {
        if (--stage < 0) {
          stage = kStagesP - 1;
          phase ^= 1u;
        }
        mbar_wait(&bars->full[stage], phase, args.status, nullptr);
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && rank == 0) {
      run_mma_pair(args, tb, bars, smem, tmem, abort);
      tc_commit_pair(&bars->drain, 1);
      mbar_wait(&bars->drain, 0, args.status, nullptr);
    }
  } else if (warp >= kSfWarp0 && warp < kEpi2Warp0) {
    run_sf_writer_pair(args, tb, bars, smem, tmem, abort);
  } else {
    float amax = 0.0f;
    run_epilogue_pair<kMidOwn>(args, tb, bars, tmem, rank, abort, amax);
    if (args.mode == 1) publish_amax_half(amax, s_amax, args.amax_partial);
  }
  // the pair's MMAs read both CTAs' shared memory and TMEM: neither leaves
  // before both are done
  tc_fence_before();
  cluster_sync();
  tc_fence_after();
  if (warp == 1) tmem_dealloc_pair(tmem, kTmemCols);
}

struct FusedArgs {
  int* grid_bar;          // [2] arrival count, generation; zero at launch
  const int32_t* row_token;
  uint8_t* hq;            // [rows, I/2]
  uint8_t* hsf;           // staged scales of hq
  float* gs_h;            // [1]
};

// Requantise h over the valid rows (epilogue warps of every CTA).  The
// 16-element blocks of all valid rows are spread over the grid, 32 per warp
// per step; each warp gathers 4 scale bytes into one staged 32-bit word.
__device__ void requantise(const GemmArgs& a1, const FusedArgs& f, const Tables& tb, int E,
                           float gs) {
  const int I = a1.I;
  const int bpr = I >> 4;
  const int k_atoms = static_cast<int>((I + kStageK - 1) / kStageK) * 4;
  const float denom = __fmul_rn(6.0f, gs);
  const int64_t total = static_cast<int64_t>(tb.dense[E]) * bpr;
  const int lane = threadIdx.x & 31;
  const int ew = (threadIdx.x >> 5) - 2;                     // 0..3
  const int64_t stride = static_cast<int64_t>(gridDim.x) * 128;
  for (int64_t base = static_cast<int64_t>(blockIdx.x) * 128 + ew * 32; base < total;
       base += stride) {
    const int64_t i = base + lane;
    const bool active = i < total;
    const int s = active ? static_cast<int>(i / bpr) : 0;
    const int g = active ? static_cast<int>(i - static_cast<int64_t>(s) * bpr) : 0;
    int e = 0;
    while (e + 1 < E && tb.dense[e + 1] <= s) ++e;
    const int64_t row = tb.off[e] + (s - tb.dense[e]);
    float v[16];
    if (active) {
      const float* src = a1.out + row * I + g * 16;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const float4 t = __ldcg(reinterpret_cast<const float4*>(src) + c);
        v[4 * c] = t.x; v[4 * c + 1] = t.y; v[4 * c + 2] = t.z; v[4 * c + 3] = t.w;
      }
    } else {
#pragma unroll
      for (int j = 0; j < 16; ++j) v[j] = 0.0f;
    }
    uint32_t packed[2];
    const uint32_t sf = quant_block16(v, gs, denom, packed);
    const uint32_t s1 = __shfl_down_sync(0xFFFFFFFFu, sf, 1);
    const uint32_t s2 = __shfl_down_sync(0xFFFFFFFFu, sf, 2);
    const uint32_t s3 = __shfl_down_sync(0xFFFFFFFFu, sf, 3);
    if (!active) continue;
    *reinterpret_cast<uint2*>(f.hq + row * (I >> 1) + g * 8) = make_uint2(packed[0], packed[1]);
    if ((g & 3) == 0)
      *reinterpret_cast<uint32_t*>(f.hsf + staged_offset(row, g, k_atoms)) =
          sf | (s1 << 8) | (s2 << 16) | (s3 << 24);
  }
}

// Like the layer kernel: 7 warps (warp 0 scale writer for one-token
// batches, warp 1 MMA, warps 2-5 epilogue, warp 6 TMA producer).
__global__ void __launch_bounds__(kThreads, 1) fused_ffn_kernel(
    const __grid_constant__ AMaps map_x, const __grid_constant__ CUtensorMap map_w1,
    const __grid_constant__ AMaps map_h, const __grid_constant__ CUtensorMap map_w2,
    const GemmArgs a1, const GemmArgs a2, const FusedArgs f) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = aligned_smem(smem_raw);
  Barriers* bars = reinterpret_cast<Barriers*>(smem + kOffBar);
  __shared__ Tables tb;
  __shared__ float s_amax[4];
  __shared__ int s_last, s_ok;

  load_tables(tb, a1, a2.n_tiles);
  const uint32_t tmem = setup_cta(bars, &map_x.full, &map_w1, &map_h.full, &map_w2, 4, 1);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  volatile int* abort = &bars->abort;
  const int E = a1.E;
  const Phase P1 = make_phase(a1, &map_x, &map_w1, tb.prefix1, E);
  const Phase P2 = make_phase(a2, &map_h, &map_w2, tb.prefix2, E);
  // every valid row in lane quarter 0: one scale-writer warp instead of copies
  bool one_quarter = true;
  for (int e = 0; e < E; ++e) one_quarter = one_quarter && tb.cnt[e] <= 32;
  Pipe pp;
  if (warp == 6) {
    if (lane == 0) {
      const Gate g2{&f.grid_bar[1], 2};
      // both phases through one copy of the role's code (the loop is not
      // unrolled), so that L2 runs instructions L1 has already fetched
#pragma unroll 1
      for (int ph = 0; ph < 2; ++ph) {
        const Phase P = ph ? P2 : P1;
        if (!run_producer(P, E, tb, bars, smem, pp, abort, ph ? &g2 : nullptr)) break;
      }
      drain_producer(bars, pp, a1.status);
    }
  } else if (warp == 1) {
    if (lane == 0) {
#pragma unroll 1
      for (int ph = 0; ph < 2; ++ph) {
        const Phase P = ph ? P2 : P1;
        if (one_quarter ? !run_mma<true>(P, bars, smem, tmem, pp, abort)
                        : !run_mma<false>(P, bars, smem, tmem, pp, abort))
          break;
      }
      mma_drain(bars, a1.status);
    }
  } else if (warp == 0) {
    if (one_quarter) {
#pragma unroll 1
      for (int ph = 0; ph < 2; ++ph) {
        const Phase P = ph ? P2 : P1;
        if (!run_sf_writer(P, bars, smem, tmem, pp, abort)) break;
      }
    }
  } else {
    float amax = 0.0f;
#pragma unroll 1
    for (int ph = 0; ph < 2; ++ph) {
      const Phase P = ph ? P2 : P1;
      // L2: gs_h is final (the requantisation before the second barrier wrote it)
      bool ok = run_epilogue(P, __ldcg(ph ? a2.gs_a : a1.gs_a), E, tb, bars, tmem, pp, abort,
                             amax, &s_ok, &s_last);
      if (ph == 1) break;
      publish_amax(amax, s_amax, a1.amax_partial);
      if (a1.gs_mid != nullptr) {
        // static intermediate scale: every tile was requantised by its own
        // CTA; one barrier (generation 2 opens the producer's L2 activation
        // loads)
        if (warp == 2 && lane == 0)
          s_ok = ok && grid_barrier(f.grid_bar, 2, a1.status, abort) ? 1 : 0;
        epi_bar();
        ok = s_ok != 0;
      } else {
        // barrier 1: every h row and every per-CTA amax is written
        if (warp == 2 && lane == 0)
          s_ok = ok && grid_barrier(f.grid_bar, 1, a1.status, abort) ? 1 : 0;
        epi_bar();
        ok = s_ok != 0;
        if (ok) {
          const float gs = global_scale_from(reduce_partials(a1.amax_partial, gridDim.x));
          if (blockIdx.x == 0 && warp == 2 && lane == 0) *f.gs_h = gs;
          requantise(a1, f, tb, E, gs);
          epi_bar();
          // barrier 2: hq, its scales and gs_h are written (opens the
          // producer's activation loads of L2)
          if (warp == 2 && lane == 0)
            s_ok = grid_barrier(f.grid_bar, 2, a1.status, abort) ? 1 : 0;
          epi_bar();
          ok = s_ok != 0;
        }
      }
      if (!ok) break;
    }
  }
  teardown_cta(bars, tmem);
}

// ------------------------------------------------------- layer kernel ----
// The whole forward of a small batch in one cooperative launch: routing,
// activation quantisation, L1, requantisation, L2 and the weighted reduce.
//  * every CTA builds the routing tables itself from topk_ids and computes
//    gs_x over all of x (no barrier), and its weight loads start at once;
//  * the activation blocks are quantised once, spread over the grid (each
//    CTA a 1/G share, written to every slot row of the token); a CTA's
//    activation loads wait for a grid-wide count of finished shares;
//  * one grid barrier after L1 (the intermediate global scale needs every
//    h); then h is requantised the same way, a 1/G share per CTA, and the
//    L2 activation loads wait for the second count;
//  * the top-k reduce of a (token, 256-column tile) is done by the CTA that
//    writes the last of the token's k slot rows of that tile (slots with no
//    row counted in advance by CTA 0).
// Work per CTA before each wait is one or two rounds of 16-element blocks
// per thread: on a small batch the critical path is a handful of memory
// round trips, not a loop over whole rows.
// Warp roles of the layer kernel (7 warps): warp 0 scale writer (see
// below), warp 1 MMA issuer and TMEM owner, warps 2-5 epilogue, warp 6 TMA
// producer.  When no tile has a valid row outside TMEM lane quarter 0 (at
// most 32 rows per expert, e.g. one token), the stage's block scales reach
// the MMA through warp 0 alone (tcgen05.st into lanes 0-31; the other
// quarters keep stale scales and produce only accumulator rows that are
// never stored) instead of tcgen05.cp copies in the tensor pipe, where they
// paced the weight stream at 0.79 us per stage.  7 warps keep two per SMSP,
// so the kernel keeps its register budget.
constexpr int kLayerProducerWarp = 6;

struct LayerArgs {
  const __nv_bfloat16* x;     // [T, H]
  const int32_t* topk_ids;    // [T, k]
  const float* topk_w;        // [T, k]
  int T, k;
  int64_t rows;               // slot rows (moe_route_rows_bound)
  uint8_t* xq;                // [rows, H/2]
  uint8_t* xsf;               // staged scales of xq
  float* gs_x;                // [1]
  int32_t* expert_offsets;    // [E+1]   (written by CTA 0)
  int32_t* expert_counts;     // [E]
  int32_t* row_token;         // [rows]
  int32_t* slot_of;           // [T*k]
  int* grid_bar;              // [kLayerBarWords]: barrier arrivals, (unused), exits,
                              // x shares done, h shares done, max |h| bits;
                              // zero between calls
  int* ycnt;                  // [T * H/256], zero between calls
  uint8_t* hq;
  uint8_t* hsf;
  float* gs_h;
  void* y;
  int y_dtype;
};


// Quantise this CTA's share of the 16-element blocks of `n_rows` source
// rows of `cols` columns (epilogue warps, one block per thread per round),
// with scale gs.  kFromTokens: source row t is token t of the bf16 x and its
// blocks go to the k slot rows of the token (slot_row[t*k + j], -1 = none);
// else source row i is flat slot i, read (fp32) from and written to slot
// row slot_row[i].  Shares are whole groups of 4 blocks, so the 4 scale
// bytes of a staged 32-bit word come from 4 neighbouring lanes.
// dry: one pass by a whole warp through the same arithmetic and stores on
// dummy values (no loads; slot_row all 0, q and sf a shared-memory scratch),
// to bring the code into the SM's instruction cache before the share itself
// is on the critical path (not inlined, so both calls run the same code).
template <bool kFromTokens>
__device__ __noinline__ void quantise_share(const void* src, int n_rows, int cols, int k,
                                            const int* slot_row, uint8_t* q, uint8_t* sf,
                                            float gs_all, const float* gs_expert = nullptr,
                                            const int32_t* ids = nullptr, bool dry = false) {
  const int bpr = cols >> 4;
  const int k_atoms = (cols + kStageK - 1) / kStageK * 4;
  const int etid = threadIdx.x - 64;
  const int n_quads = n_rows * (bpr >> 2);
  const int q0 = static_cast<int>(static_cast<int64_t>(n_quads) * blockIdx.x / gridDim.x);
  const int q1 = static_cast<int>(static_cast<int64_t>(n_quads) * (blockIdx.x + 1) / gridDim.x);
  const int b_end = 4 * q1;
  for (int b0 = 4 * q0 + (etid & ~31); dry || b0 < b_end; b0 += 128) {      // warp-uniform
    const int b = b0 + (etid & 31);
    const bool active = dry || b < b_end;
    const int r = active && !dry ? b / bpr : 0;
    const int g = active && !dry ? b - r * bpr : 0;
    float v[16];
    int row = -1;
    float gs = gs_all;
    if (kFromTokens) {
      uint4 u0 = make_uint4(0u, 0u, 0u, 0u), u1 = u0;
      if (active && !dry) {
        const uint4* p = reinterpret_cast<const uint4*>(
            static_cast<const __nv_bfloat16*>(src) + static_cast<int64_t>(r) * cols + g * 16);
        u0 = __ldg(p);
        u1 = __ldg(p + 1);
      }
      const uint32_t w8[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
#pragma unroll
      for (int m = 0; m < 8; ++m) {
        v[2 * m] = __uint_as_float(w8[m] << 16);
        v[2 * m + 1] = __uint_as_float(w8[m] & 0xFFFF0000u);
      }
    } else {
      if (active) row = slot_row[r];
      // h rows (flat slot r) under a static per-expert intermediate scale
      // (a slot with no row, i.e. an invalid expert id, is skipped)
      if (gs_expert != nullptr && row >= 0) gs = __ldg(gs_expert + ids[r]);
      float4 f[4];
#pragma unroll
      for (int c = 0; c < 4; ++c) f[c] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (row >= 0 && !dry) {
        const float4* p = reinterpret_cast<const float4*>(
            static_cast<const float*>(src) + static_cast<int64_t>(row) * cols + g * 16);
#pragma unroll
        for (int c = 0; c < 4; ++c) f[c] = __ldcg(p + c);
      }
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        v[4 * c] = f[c].x;
        v[4 * c + 1] = f[c].y;
        v[4 * c + 2] = f[c].z;
        v[4 * c + 3] = f[c].w;
      }
    }
    if (dry) {
#pragma unroll
      for (int j = 0; j < 16; ++j) v[j] = 1.0f + 0.25f * j;
    }
    uint32_t packed[2];
    const uint32_t s = quant_block16(v, gs, __fmul_rn(6.0f, gs), packed);
    const uint32_t word = s | (__shfl_down_sync(0xFFFFFFFFu, s, 1) << 8) |
                          (__shfl_down_sync(0xFFFFFFFFu, s, 2) << 16) |
                          (__shfl_down_sync(0xFFFFFFFFu, s, 3) << 24);
    if (!active) continue;
    auto put = [&](int dst) {
      *reinterpret_cast<uint2*>(q + static_cast<int64_t>(dst) * (cols >> 1) + g * 8) =
          make_uint2(packed[0], packed[1]);
      if ((g & 3) == 0)
        *reinterpret_cast<uint32_t*>(sf + staged_offset(dst, g, k_atoms)) = word;
    };
    if (kFromTokens) {
      for (int j = 0; j < k; ++j) {
        const int dst = slot_row[r * k + j];
        if (dst >= 0) put(dst);
      }
    } else if (row >= 0) {
      put(row);
    }
    if (dry) break;
  }
}

// Publish this CTA's finished share: its writes are made visible to every
// CTA, to the generic and the async (TMA) proxy, then counted.
__device__ void share_done(int* count) {
  fence_proxy_async_global();
  __threadfence();
  epi_bar();
  if (threadIdx.x == 64) atomicAdd(count, 1);
}

__global__ void __launch_bounds__(kThreads, 1) layer_kernel(
    const __grid_constant__ AMaps map_x, const __grid_constant__ CUtensorMap map_w1,
    const __grid_constant__ AMaps map_h, const __grid_constant__ CUtensorMap map_w2,
    const GemmArgs a1, const GemmArgs a2, const LayerArgs L) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = aligned_smem(smem_raw);
  Barriers* bars = reinterpret_cast<Barriers*>(smem + kOffBar);
  __shared__ Tables tb;
  __shared__ float s_amax[4];
  __shared__ int s_last, s_ok, s_n;
  __shared__ int s_row[kLayerMaxSlots];       // slot row of flat index t*k+j
  __shared__ int s_tok[kLayerMaxSlots];       // token of dense slot
  __shared__ int s_scratch[kMaxExperts];      // running counts, then the reduce list
  __shared__ float s_gs;
  // dry passes of the share quantisers: slot rows (all 0), then q and sf bytes
  __shared__ __align__(16) int s_dry[kMaxTopK + 8];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int E = a1.E, k = L.k, S = L.T * L.k;
  const int H = a1.K, I = a1.I;

  // ---- routing tables, in every CTA ----
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    tb.cnt[e] = 0;
    s_scratch[e] = 0;
  }
  if (threadIdx.x == 0) s_amax[0] = 0.0f;
  if (threadIdx.x < kMaxTopK + 8) s_dry[threadIdx.x] = 0;
  __syncthreads();
  for (int i = threadIdx.x; i < S; i += blockDim.x) {
    const int e = L.topk_ids[i];
    if (e >= 0 && e < E)
      atomicAdd(&tb.cnt[e], 1);
    else if (blockIdx.x == 0)
      record_status(a1.status, kErrBadIndex);
  }
  __syncthreads();
  if (warp == 0) {
    // exclusive prefix sums over the experts: each lane a run of experts,
    // then a warp scan of the run totals (slots, m-tiles)
    const int per = (E + 31) / 32;
    const int e0 = min(E, lane * per), e1 = min(E, e0 + per);
    int c_sum = 0, m_sum = 0;
    for (int e = e0; e < e1; ++e) {
      c_sum += tb.cnt[e];
      m_sum += (tb.cnt[e] + kBM - 1) / kBM;
    }
    int c_inc = c_sum, m_inc = m_sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int c_up = __shfl_up_sync(0xFFFFFFFFu, c_inc, o);
      const int m_up = __shfl_up_sync(0xFFFFFFFFu, m_inc, o);
      if (lane >= o) {
        c_inc += c_up;
        m_inc += m_up;
      }
    }
    int d = c_inc - c_sum, mt = m_inc - m_sum;
    for (int e = e0; e < e1; ++e) {
      const int c = tb.cnt[e];
      const int m = (c + kBM - 1) / kBM;
      tb.mtiles[e] = m;
      tb.off[e] = mt * kBM;
      tb.prefix1[e] = mt * a1.n_tiles;
      tb.prefix2[e] = mt * a2.n_tiles;
      tb.dense[e] = d;
      d += c;
      mt += m;
    }
    if (lane == 31) {
      tb.prefix1[E] = m_inc * a1.n_tiles;
      tb.prefix2[E] = m_inc * a2.n_tiles;
      tb.dense[E] = c_inc;
      if (blockIdx.x == 0) L.expert_offsets[E] = m_inc * kBM;
    }
  }
  __syncthreads();
  // every valid row in lane quarter 0: one scale-writer warp instead of copies
  bool one_quarter = true;
  for (int e = 0; e < E; ++e) one_quarter = one_quarter && tb.cnt[e] <= 32;
  const uint32_t tmem = setup_cta(bars, &map_x.full, &map_w1, &map_h.full, &map_w2, 4, 1);
  volatile int* abort = &bars->abort;
  const Phase P1 = make_phase(a1, &map_x, &map_w1, tb.prefix1, E);
  const Phase P2 = make_phase(a2, &map_h, &map_w2, tb.prefix2, E);
  Pipe pp;
  // Warm the instruction cache with the two share quantisers while their
  // code is off the critical path: warp 1 (its MMAs wait for the activation
  // gate anyway) runs the activation one, warp 0 the intermediate one (needed
  // after the grid barrier; its first weight loads go out a little later).
  {
    uint8_t* dq = reinterpret_cast<uint8_t*>(s_dry + kMaxTopK);
    uint8_t* dsf = reinterpret_cast<uint8_t*>(s_dry + kMaxTopK + 4);
    if (warp == 1)
      quantise_share<true>(L.x, L.T, H, k, s_dry, dq, dsf, 1.0f, nullptr, nullptr, true);
    else if (warp == 0)
      quantise_share<false>(a1.out, S, I, k, s_dry, dq, dsf, 1.0f, nullptr, nullptr, true);
  }
  if (warp == kLayerProducerWarp) {
    if (lane == 0) {
      const int G = static_cast<int>(gridDim.x);
      const Gate g1{&L.grid_bar[3], G};
      const Gate g2{&L.grid_bar[4], G};
      // both phases through one copy of the role's code (the loop is not
      // unrolled), so that L2 runs instructions L1 has already fetched
#pragma unroll 1
      for (int ph = 0; ph < 2; ++ph) {
        const Phase P = ph ? P2 : P1;
        const Gate g = ph ? g2 : g1;
        if (!run_producer(P, E, tb, bars, smem, pp, abort, &g)) break;
      }
      drain_producer(bars, pp, a1.status);
    }
  } else if (warp == 1) {
    if (lane == 0) {
#pragma unroll 1
      for (int ph = 0; ph < 2; ++ph) {
        const Phase P = ph ? P2 : P1;
        if (one_quarter ? !run_mma<true>(P, bars, smem, tmem, pp, abort)
                        : !run_mma<false>(P, bars, smem, tmem, pp, abort))
          break;
      }
      mma_drain(bars, a1.status);
    }
  } else if (warp == 0) {
    if (one_quarter) {
#pragma unroll 1
      for (int ph = 0; ph < 2; ++ph) {
        const Phase P = ph ? P2 : P1;
        if (!run_sf_writer(P, bars, smem, tmem, pp, abort)) break;
      }
    }
  } else {
    // The weight loads are already going out; meanwhile the epilogue warps
    // rank the slots, take the activations' global scale and quantise this
    // CTA's share of the activation blocks.
    const bool lead = warp == 2 && lane == 0;
    const int etid = threadIdx.x - 64;
    if (warp == 2) {
      // stable rank inside each expert: one warp, 32 flat indices per round
      const unsigned lt = (1u << lane) - 1u;
      for (int base = 0; base < S; base += 32) {
        const int i = base + lane;
        int e = i < S ? L.topk_ids[i] : -1;
        if (e < 0 || e >= E) e = -1;
        const unsigned peers = __match_any_sync(0xFFFFFFFFu, e);
        const int rank = __popc(peers & lt);
        const int before = e >= 0 ? s_scratch[e] : 0;
        __syncwarp();
        if (e >= 0 && (peers >> lane) == 1u) s_scratch[e] = before + rank + 1;
        __syncwarp();
        if (i < S) {
          s_row[i] = e >= 0 ? tb.off[e] + before + rank : -1;
          if (e >= 0) s_tok[tb.dense[e] + before + rank] = i / k;
        }
      }
    }
    {
      // gs_x = amax(x) / 2688; the loads of a thread are issued in batches
      const int n_vec = L.T * H / 8;
      float m = 0.0f;
      for (int i0 = etid; i0 < n_vec; i0 += 128 * 8) {
        uint4 u[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int i = i0 + j * 128;
          u[j] = i < n_vec ? __ldg(reinterpret_cast<const uint4*>(L.x) + i)
                           : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const uint32_t w4[4] = {u[j].x, u[j].y, u[j].z, u[j].w};
#pragma unroll
          for (int c = 0; c < 4; ++c)
            m = fmaxf(m, fmaxf(fabsf(__uint_as_float(w4[c] << 16)),
                               fabsf(__uint_as_float(w4[c] & 0xFFFF0000u))));
        }
      }
      m = warp_max(m);
      // |x| >= 0, so the float bits order like the values
      if (lane == 0) atomicMax(reinterpret_cast<int*>(&s_amax[0]), __float_as_int(m));
    }
    epi_bar();
    if (lead) {
      s_gs = global_scale_from(s_amax[0]);
      if (blockIdx.x == 0) *L.gs_x = s_gs;
    }
    if (blockIdx.x == 0) {
      // routing outputs for the caller
      for (int e = etid; e < E; e += 128) {
        L.expert_offsets[e] = tb.off[e];
        L.expert_counts[e] = tb.cnt[e];
      }
      for (int64_t r = etid; r < L.rows; r += 128) L.row_token[r] = -1;
    }
    epi_bar();
    if (blockIdx.x == 0) {
      for (int i = etid; i < S; i += 128) {
        L.slot_of[i] = s_row[i];
        if (s_row[i] >= 0) {
          L.row_token[s_row[i]] = i / k;
        } else {
          // an expert id outside [0, E): no L2 tile will count this slot, so
          // it is counted now (the grid barrier orders this before every L2
          // epilogue); a token without any valid slot gets y = 0
          const int t = i / k;
          bool any = false;
          for (int j = 0; j < k; ++j) any |= s_row[t * k + j] >= 0;
          if (any) {
            for (int nt = 0; nt < a2.n_tiles; ++nt) atomicAdd(&L.ycnt[t * a2.n_tiles + nt], 1);
          } else if (i == t * k) {
            for (int c = 0; c < H; ++c) {
              if (L.y_dtype == 0)
                static_cast<__nv_bfloat16*>(L.y)[static_cast<int64_t>(t) * H + c] = __float2bfloat16(0.0f);
              else
                static_cast<float*>(L.y)[static_cast<int64_t>(t) * H + c] = 0.0f;
            }
          }
        }
      }
    }
    quantise_share<true>(L.x, L.T, H, k, s_row, L.xq, L.xsf, s_gs);
    share_done(&L.grid_bar[3]);
    float amax = 0.0f;
    // every CTA computed the same gs_x itself (CTA 0's copy in memory is for
    // the caller, with no ordering against this read)
    // L1 and L2 run through one copy of the epilogue code (see the producer)
    const YReduce yr{L.ycnt, L.topk_w, s_row, s_tok, L.y, L.y_dtype, k, a2.n_tiles,
                     s_scratch, &s_n};
    float gs_phase = s_gs;
#pragma unroll 1
    for (int ph = 0; ph < 2; ++ph) {
      const Phase P = ph ? P2 : P1;
      bool ok = run_epilogue(P, gs_phase, E, tb, bars, tmem, pp, abort, amax, &s_ok, &s_last,
                             ph ? &yr : nullptr);
      if (ph == 1) break;
      publish_amax(amax, s_amax, a1.amax_partial);
      // the one grid barrier: every h row is written and every CTA's max of
      // |h| is folded into one word (non-negative floats order like their bits)
      if (lead) {
        s_ok = 0;
        if (ok) {
          const float cta_max = fmaxf(fmaxf(s_amax[0], s_amax[1]), fmaxf(s_amax[2], s_amax[3]));
          atomicMax(&L.grid_bar[5], __float_as_int(cta_max));
          s_ok = count_barrier(&L.grid_bar[0], a1.status, abort) ? 1 : 0;
        }
      }
      epi_bar();
      if (s_ok == 0) {
        // the producer's wait for the h shares ends at once
        if (lead) *abort = 1;
        break;
      }
      if (a1.gs_mid != nullptr) {
        // static intermediate scale: no global max; the share of h is
        // requantised with the scale of each slot's expert
        quantise_share<false>(a1.out, S, I, k, s_row, L.hq, L.hsf, 0.0f, a1.gs_mid, L.topk_ids);
        gs_phase = 0.0f;
      } else {
        const float gs = global_scale_from(__int_as_float(ld_acquire(&L.grid_bar[5])));
        if (blockIdx.x == 0 && lead) *L.gs_h = gs;
        quantise_share<false>(a1.out, S, I, k, s_row, L.hq, L.hsf, gs);
        gs_phase = gs;
      }
      share_done(&L.grid_bar[4]);
    }
  }
  teardown_cta(bars, tmem);
  // last CTA out clears the barrier words for the next call
  if (threadIdx.x == 0) {
    __threadfence();
    if (atomicAdd(&L.grid_bar[2], 1) == static_cast<int>(gridDim.x) - 1) {
      for (int i = 0; i < kLayerBarWords; ++i) L.grid_bar[i] = 0;
      __threadfence();
    }
  }
}

PerDeviceOnce g_gemm_attr, g_gemm_half_attr, g_gemm_pair_attr, g_gemm_pair_mid_attr, g_fused_attr,
    g_layer_attr;

}  // namespace

cudaError_t launch_layer(const GemmArgs& a1, const GemmArgs& a2, const AMaps& map_x,
                         const CUtensorMap& map_w1, const AMaps& map_h,
                         const CUtensorMap& map_w2, const LayerLaunch& l, int grid,
                         cudaStream_t stream) {
  {
    const cudaError_t err =
        set_smem_attr_once(g_layer_attr, reinterpret_cast<const void*>(layer_kernel), kSmemBytes);
    if (err != cudaSuccess) return err;
  }
  LayerArgs L{static_cast<const __nv_bfloat16*>(l.x), l.topk_ids, l.topk_w, l.T, l.k, l.rows,
              l.xq, l.xsf, l.gs_x, l.expert_offsets, l.expert_counts, l.row_token, l.slot_of,
              l.grid_bar, l.ycnt, l.hq, l.hsf, l.gs_h, l.y, l.y_dtype};
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, layer_kernel, map_x, map_w1, map_h, map_w2, a1, a2, L);
}

int gemm_smem_bytes() { return kSmemBytes; }

cudaError_t launch_gemm(const GemmArgs& args, const AMaps& map_a, const CUtensorMap& map_b,
                        int grid, int64_t min_tiles, bool allow_pair, cudaStream_t stream) {
  // At least kStreamKFactor tiles per CTA whatever the routing: whole tiles
  // and two epilogue sets, over CTA pairs when the grid holds at least one
  // pair.  A static intermediate scale requantised in the L1 epilogue takes
  // the pair kernel's own instantiation (each set requantises the columns
  // it stored), else the one-CTA kernel.
  const bool mid_own = args.mode == 1 && args.gs_mid != nullptr && args.mid_in_epilogue;
  const bool pair = min_tiles >= int64_t{kStreamKFactor} * grid && allow_pair && grid >= 2;
  const bool half = min_tiles >= int64_t{kStreamKFactor} * grid && !mid_own;
  cudaLaunchConfig_t cfg = {};
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  cfg.attrs = attr;
  if (pair) {
    const void* kernel = mid_own ? reinterpret_cast<const void*>(grouped_gemm_pair_kernel<true>)
                                 : reinterpret_cast<const void*>(grouped_gemm_pair_kernel<false>);
    const cudaError_t err =
        set_smem_attr_once(mid_own ? g_gemm_pair_mid_attr : g_gemm_pair_attr, kernel, kSmemBytesP);
    if (err != cudaSuccess) return err;
    cfg.gridDim = dim3(grid & ~1);
    cfg.blockDim = dim3(kThreadsHalf);
    cfg.dynamicSmemBytes = kSmemBytesP;
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.numAttrs = 1 + pdl_attr(&attr[1]);
    if (mid_own) return cudaLaunchKernelEx(&cfg, grouped_gemm_pair_kernel<true>, map_a, map_b, args);
    return cudaLaunchKernelEx(&cfg, grouped_gemm_pair_kernel<false>, map_a, map_b, args);
  }
  cfg.gridDim = dim3(grid);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.numAttrs = pdl_attr(&attr[0]);
  if (half) {
    const cudaError_t err = set_smem_attr_once(
        g_gemm_half_attr, reinterpret_cast<const void*>(grouped_gemm_kernel<true>), kSmemBytes);
    if (err != cudaSuccess) return err;
    cfg.blockDim = dim3(kThreadsHalf);
    return cudaLaunchKernelEx(&cfg, grouped_gemm_kernel<true>, map_a, map_b, args);
  }
  const cudaError_t err = set_smem_attr_once(
      g_gemm_attr, reinterpret_cast<const void*>(grouped_gemm_kernel<false>), kSmemBytes);
  if (err != cudaSuccess) return err;
  cfg.blockDim = dim3(kThreadsSt);
  return cudaLaunchKernelEx(&cfg, grouped_gemm_kernel<false>, map_a, map_b, args);
}

cudaError_t launch_fused_ffn(const GemmArgs& a1, const GemmArgs& a2, const AMaps& map_x,
                             const CUtensorMap& map_w1, const AMaps& map_h,
                             const CUtensorMap& map_w2, int* grid_bar, const int32_t* row_token,
                             uint8_t* hq, uint8_t* hsf, float* gs_h, int grid,
                             cudaStream_t stream) {
  {
    const cudaError_t err =
        set_smem_attr_once(g_fused_attr, reinterpret_cast<const void*>(fused_ffn_kernel), kSmemBytes);
    if (err != cudaSuccess) return err;
  }
  cudaError_t err = cudaMemsetAsync(grid_bar, 0, 2 * sizeof(int), stream);
  if (err != cudaSuccess) return err;
  FusedArgs f{grid_bar, row_token, hq, hsf, gs_h};
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, fused_ffn_kernel, map_x, map_w1, map_h, map_w2, a1, a2, f);
}

}  // namespace nvmoe
