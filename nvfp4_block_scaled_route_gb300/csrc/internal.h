// Internal launchers shared between the kernel translation units and the
// C-ABI layer (api.cu).  Not part of the public interface.
#pragma once

#include <atomic>
#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>
#include <utility>

namespace nvmoe {

// Kernel attributes (the dynamic shared-memory size) are set once per device
// and kernel: one bit per device id (ids 0..63; larger ids set the attribute
// on every launch).
struct PerDeviceOnce {
  std::atomic<uint64_t> done{0};
};

inline cudaError_t set_smem_attr_once(PerDeviceOnce& once, const void* fn, int bytes) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = dev >= 0 && dev < 64 ? (uint64_t{1} << dev) : 0;
  if (bit != 0 && (once.done.load(std::memory_order_acquire) & bit)) return cudaSuccess;
  e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && bit != 0) once.done.fetch_or(bit, std::memory_order_acq_rel);
  return e;
}

constexpr int kTileRows = 128;        // rows per tensor-core tile / SF atom row block
constexpr int kSfAtomBytes = 512;     // 128 rows x 4 scale bytes
constexpr int kStageK = 256;          // K elements per pipeline stage
constexpr int kMaxExperts = 256;
constexpr int kMaxTopK = 32;
constexpr int kQuantMaxPartials = 1024;

// Adds to the count of kernels this library has enqueued
// (nvmoe_kernel_launch_count).
void note_launches(int kernels);

inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }
inline int64_t round_up(int64_t a, int64_t b) { return ceil_div(a, b) * b; }

// Byte size of a staged scale buffer for rows x cols.
inline size_t sf_mma_bytes(int64_t rows, int64_t cols) {
  return static_cast<size_t>(round_up(rows, kTileRows) * (round_up(cols, kStageK) / 16));
}

// ---- route ----
cudaError_t launch_route(const int32_t* topk_ids, int64_t T, int k, int E,
                         int32_t* expert_offsets, int32_t* expert_counts,
                         int32_t* row_token, int64_t rows_bound, int32_t* slot_of,
                         int32_t* chunk_counts, int n_chunks, int* status,
                         cudaStream_t stream);
int route_chunk_elems();

// ---- quantiser ----
// Pass 1: per-block maxima of |x| into partial[0..n_partial).
cudaError_t launch_quant_amax(const void* x, int x_dtype, int64_t n_elems, float* partial,
                              int n_partial, cudaStream_t stream);
// Pass 2: reduce partial maxima -> gs; quantise rows.  row_valid (nullable)
// skips rows whose entry is < 0.
cudaError_t launch_quant_pack(const void* x, int x_dtype, int64_t rows, int64_t cols,
                              const int32_t* row_dst, int fanout, const int32_t* row_valid,
                              const float* partial, int n_partial, uint8_t* q,
                              uint8_t* sf_row, uint8_t* sf_mma, float* gs_out,
                              int64_t out_rows, int* status, cudaStream_t stream);
int quant_amax_blocks(int64_t n_elems);

// ---- programmatic dependent launch ----
// Whether the step kernels of the multi-launch path are launched with
// programmatic stream serialization (nvmoe_set_pdl; default off), and the
// launch attribute that does it (attr count 0 or 1 written into attr[]).
bool pdl_enabled();
int pdl_attr(cudaLaunchAttribute* attr);

// kernel<<<grid, block, smem, stream>>>(args...) with the PDL attribute when
// enabled; the kernel must call pdl_wait() before touching memory of earlier
// kernels.  Errors as for any launch (also left for cudaGetLastError).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  cfg.attrs = attr;
  cfg.numAttrs = pdl_attr(attr);
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// ---- expert-parallel dispatch / combine (ep.cu) ----
cudaError_t launch_ep_dest(const int32_t* ids, int64_t S, int E, int G, int32_t* dest, int* status,
                           cudaStream_t stream);
cudaError_t launch_ep_pack(const int32_t* ids, const int32_t* padded, const int32_t* dest,
                           const int32_t* offsets, const int32_t* counts, int64_t S, int k, int E,
                           int G, const uint8_t* q_tok, const uint8_t* sf_tok, int H,
                           int32_t* send_pos, uint8_t* send_rows, int32_t* send_expert,
                           cudaStream_t stream);
cudaError_t launch_ep_scatter(const uint8_t* rows, int64_t n, int H, const int32_t* slot_of,
                              int64_t out_rows, uint8_t* xq, uint8_t* xsf, int k_atoms,
                              int* status, cudaStream_t stream);
cudaError_t launch_ep_gather(const void* slot_out, int64_t row_bytes, int64_t slot_rows,
                             const int32_t* slot_of, int64_t n, void* out, int* status,
                             cudaStream_t stream);
cudaError_t launch_max_reduce(const float* partial, int n, float* out, cudaStream_t stream);
// Both passes in one CTA, for inputs of at most kQuantSmallElems elements.
constexpr int64_t kQuantSmallElems = 64 * 1024;
// Row-major activation scales (cols % 256 == 0, 16-byte aligned) into the
// staged layout, rows rounded up to whole 128-row tiles (rows past `rows`
// get zero scales).
cudaError_t launch_stage_act_sf(const uint8_t* sf_row, int64_t rows, int64_t cols,
                                uint8_t* sf_mma, cudaStream_t stream);
cudaError_t launch_quant_small(const void* x, int x_dtype, int64_t rows, int64_t cols,
                               const int32_t* row_dst, int fanout, uint8_t* q, uint8_t* sf_row,
                               uint8_t* sf_mma, float* gs_out, int64_t out_rows, int* status, cudaStream_t stream);

// ---- weights ----
cudaError_t launch_weight_amax(const float* w, int E, int64_t per_expert, float* partial,
                               int parts_per_expert, cudaStream_t stream);
cudaError_t launch_weight_quant(const float* w, int E, int K, int N, const float* partial,
                                int parts_per_expert, uint8_t* q, uint8_t* sf, float* gs,
                                cudaStream_t stream);
cudaError_t launch_prepare_weights(const uint8_t* q_ckpt, const uint8_t* sf_ckpt, int E, int K,
                                   int N, uint8_t* q_out, uint8_t* sf_out, cudaStream_t stream);

// ---- grouped GEMM ----
struct GemmArgs {
  int mode;               // 1: L1 (gate/up pairs, SiLU epilogue), 2: L2
  int E;
  int K;                  // reduction length (elements)
  int N;                  // rows of each expert's B matrix (L1: 2I, L2: H)
  int I;                  // L1 only: intermediate size
  int n_tiles;            // tiles along N per expert
  const int32_t* expert_offsets;
  const int32_t* expert_counts;
  const uint8_t* a_sf;    // staged, rows_bound x K
  const uint8_t* b_sf;    // staged, E*N x K
  const float* gs_a;      // [1]
  const float* gs_b;      // [E]
  const float* gs_b_up;   // L1: [E] scale of the up half, or null (= gs_b)
  const float* gs_mid;    // [E] static intermediate scale, or null (dynamic).  L1:
                          // each finished tile of h is requantised with
                          // gs_mid[e] into mid_q / mid_sf by its own CTA;
                          // L2: alpha = gs_mid[e] * gs_b[e] (gs_a unused)
  uint8_t* mid_q;         // L1 with gs_mid: hq [rows, I/2]
  uint8_t* mid_sf;        // L1 with gs_mid: staged scales of hq
  bool mid_in_epilogue;   // L1 with gs_mid: requantise in the epilogue (else the
                          // caller requantises after its grid barrier)
  float* out;             // L1: h [rows, I]; L2: slot_out [rows, N]
  int out_dtype;          // L2: slot_out element type, 0 bf16, 1 fp32, 2 fp16 (RNE)
  float* tap;             // L1: l1_out [rows, 2I] or null
  float* amax_partial;    // L1: [grid]
  float* partials;        // split-tile pieces: [2 * grid][128][256] fp32
  int* counters;          // split-tile arrival counts: [kMaxSplitTiles], zero between calls
  int* status;
  int64_t rows;           // rows of out / tap / mid_q (checked by the debug-bounds build)
  // Optional: the A operand (activation rows and their scales) is ready once
  // *ready_flag >= ready_value; the producer waits for it (at most
  // ready_limit_ns) before its first load.  nullptr = ready at launch.
  const int* ready_flag;
  int ready_value;
  uint64_t ready_limit_ns;
};
constexpr int kMaxGrid = 256;
constexpr int kMaxSplitTiles = 4 * kMaxGrid;
// Activation (A operand) maps of one matrix: 128-row boxes, and 32-row boxes
// used for m-tiles with at most 32 valid rows (decode), so that padding rows
// are not fetched.
struct AMaps {
  CUtensorMap full;
  CUtensorMap small;
};
constexpr int kSmallABoxRows = 32;
// min_tiles: tiles that exist whatever the routing (a lower bound); with at
// least 4 per CTA the kernel with whole tiles and two epilogue sets runs,
// over CTA pairs (cta_group::2) when allow_pair (grid rounded down to even).
cudaError_t launch_gemm(const GemmArgs& args, const AMaps& map_a, const CUtensorMap& map_b,
                        int grid, int64_t min_tiles, bool allow_pair, cudaStream_t stream);
int gemm_smem_bytes();
// L1 -> grid barrier -> requantise -> grid barrier -> L2 in one cooperative
// launch (grid <= SM count, one CTA per SM).
// The whole forward of a small batch (routing .. reduce) in one cooperative
// launch; limits: T*k <= kLayerMaxSlots, T*H <= kQuantSmallElems, bf16 x.
constexpr int kLayerMaxSlots = 128;
// Synchronisation words of the layer kernel (zero between calls).
constexpr int kLayerBarWords = 8;
struct LayerLaunch {
  const void* x;              // bf16 [T, H]
  const int32_t* topk_ids;
  const float* topk_w;
  int T, k;
  int64_t rows;
  uint8_t* xq;
  uint8_t* xsf;
  float* gs_x;
  int32_t* expert_offsets;
  int32_t* expert_counts;
  int32_t* row_token;
  int32_t* slot_of;
  int* grid_bar;              // [3], zero between calls
  int* ycnt;                  // [T * H/256], zero between calls
  uint8_t* hq;
  uint8_t* hsf;
  float* gs_h;
  void* y;
  int y_dtype;
};
cudaError_t launch_layer(const GemmArgs& a1, const GemmArgs& a2, const AMaps& map_x,
                         const CUtensorMap& map_w1, const AMaps& map_h,
                         const CUtensorMap& map_w2, const LayerLaunch& l, int grid,
                         cudaStream_t stream);
cudaError_t launch_fused_ffn(const GemmArgs& a1, const GemmArgs& a2, const AMaps& map_x,
                             const CUtensorMap& map_w1, const AMaps& map_h,
                             const CUtensorMap& map_w2, int* grid_bar, const int32_t* row_token,
                             uint8_t* hq, uint8_t* hsf, float* gs_h, int grid,
                             cudaStream_t stream);

// ---- dense FP4 tensor-core probe (peak.cu) ----
enum : int {
  kProbePair = 1, kProbeN128 = 2, kProbeCp32 = 4, kProbeCp256 = 8,
  kProbeAcc2 = 16, kProbeAcc4 = 32, kProbeNoAcc = 64, kProbeNoMma = 128,
  kProbeCpAOnly = 256, kProbeCpEarly = 512, kProbeSt = 1024
};
cudaError_t launch_mma_probe(int variant, int iters, int grid, long long* cycles, int* status,
                             cudaStream_t stream);

// ---- reduce ----
// Router front-end (router.cu): logits partials [splits][T][E] fp32 in the
// workspace, then top-k and softmax per token.
size_t router_workspace_bytes(int64_t T, int H, int E);
// map_x: x as bytes [T, 2H], box 128 B x 128 rows; map_w: the router weight
// as bytes [E, 2H], box 128 B x (E padded to 16) rows; both 128-byte swizzle.
cudaError_t launch_router(const CUtensorMap& map_x, const CUtensorMap& map_w, int64_t T, int H,
                          int E, int k, int mode, int32_t* ids, float* weights, float* partials,
                          int* status, cudaStream_t stream);

cudaError_t launch_reduce(const void* slot_out, int slot_dtype, const int32_t* slot_of,
                          const float* topk_w, int64_t T, int k, int64_t H, void* y, int y_dtype,
                          cudaStream_t stream);

}  // namespace nvmoe
