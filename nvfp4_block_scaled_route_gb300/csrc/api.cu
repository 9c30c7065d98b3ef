// C-ABI entry points of libnvfp4moe.so (declared in include/nvfp4moe.h):
// argument checks, workspace carving, TMA descriptor encoding and kernel
// launches.  No allocation, no host synchronisation on the compute calls.
#include <nvtx3/nvToolsExt.h>
#include <cstring>
#include <atomic>
#include <mutex>

#include "nvfp4moe.h"
#include "internal.h"

using namespace nvmoe;

namespace {

constexpr size_t kStatusBytes = 256;   // every workspace starts with the status word
constexpr size_t kAlign = 256;

size_t align_up(size_t v) { return (v + kAlign - 1) / kAlign * kAlign; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// ---- cuTensorMapEncodeTiled through the runtime's driver entry point ----
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn get_encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// 2-D uint8 tensor [rows, row_bytes], box 128 x 128 bytes, 128-byte swizzle.
bool make_map(CUtensorMap* map, const void* base, int64_t row_bytes, int64_t rows,
              uint32_t box_rows = 128) {
  EncodeTiledFn fn = get_encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(row_bytes), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(row_bytes)};
  cuuint32_t box[2] = {128, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// B-operand tiles: [n_tiles][128 rows][128 bytes] contiguous, as a 3-D map
// with a 128 x 128 x 1 box (one 16 KB tile per load).
bool make_tiled_map(CUtensorMap* map, const void* base, int64_t n_tiles) {
  EncodeTiledFn fn = get_encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t dims[3] = {128, 128, static_cast<cuuint64_t>(n_tiles)};
  cuuint64_t strides[2] = {128, 128 * 128};
  cuuint32_t box[3] = {128, 128, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// NVTX range around each call that enqueues GPU work: named for the entry
// point in a tool's timeline (nsys, ncu --nvtx); a few ns without a tool.
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};

int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return n;
}

// The CUDA error behind the last NVMOE_ERR_CUDA of this host thread.
thread_local cudaError_t g_last_cuda = cudaSuccess;

cudaError_t note(cudaError_t e) {
  if (e != cudaSuccess) g_last_cuda = e;
  return e;
}

int fail(cudaError_t e) {
  note(e);
  return NVMOE_ERR_CUDA;
}

int status_of(cudaError_t e) { return e == cudaSuccess ? NVMOE_OK : fail(e); }

// Kernels of this library enqueued so far (CUDA-graph replays are not
// launches and are not counted).
std::atomic<uint64_t> g_launches{0};

cudaError_t counted(cudaError_t e, int kernels) {
  if (e == cudaSuccess) g_launches += kernels;
  return note(e);
}

}  // namespace

void nvmoe::note_launches(int kernels) { g_launches += kernels; }

namespace {
std::atomic<int> g_pdl{0};
}  // namespace

bool nvmoe::pdl_enabled() { return g_pdl.load(std::memory_order_relaxed) != 0; }

int nvmoe::pdl_attr(cudaLaunchAttribute* attr) {
  if (!pdl_enabled()) return 0;
  attr->id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr->val.programmaticStreamSerializationAllowed = 1;
  return 1;
}

namespace {

// Workspace carving helper.
struct Carve {
  uint8_t* base;
  size_t off = 0;
  template <typename T>
  T* take(size_t bytes) {
    T* p = reinterpret_cast<T*>(base == nullptr ? nullptr : base + off);
    off += align_up(bytes);
    return p;
  }
};

// T*k < 2^31 (slot indices are int32), checked without forming the product,
// which could overflow int64 for a huge T.
bool slots_fit(int64_t T, int k) { return k >= 1 && T <= int64_t{INT32_MAX} / k; }

// rows * cols elements below 2^40, checked without forming the product.
bool elems_fit(int64_t rows, int64_t cols) {
  return cols <= 0 || rows <= (int64_t{1} << 40) / cols;
}

int64_t rows_bound(int64_t T, int k, int E) {
  const int64_t S = T * k;
  const int64_t pad = (S < E ? S : E) * (kTileRows - 1);
  return round_up(S + pad, kTileRows);
}

}  // namespace

extern "C" {

const char* nvmoe_last_cuda_error(void) {
  return g_last_cuda == cudaSuccess ? "" : cudaGetErrorName(g_last_cuda);
}

const char* nvmoe_status_str(int s) {
  switch (s) {
    case NVMOE_OK: return "ok";
    case NVMOE_ERR_INVALID_ARG: return "invalid argument";
    case NVMOE_ERR_UNSUPPORTED_SHAPE: return "unsupported shape";
    case NVMOE_ERR_MISALIGNED: return "pointer not 16-byte aligned";
    case NVMOE_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case NVMOE_ERR_CUDA: return "CUDA error";
    case NVMOE_ERR_TIMEOUT: return "device wait timed out";
    case NVMOE_ERR_DEVICE_BAD_INDEX: return "expert id out of range";
    case NVMOE_ERR_RANGE: return "value beyond the range of its storage type";
    case NVMOE_ERR_DEVICE_BOUNDS: return "index outside its buffer (debug-bounds build)";
    default: return "unknown status";
  }
}

int nvmoe_version(void) { return 200; }

int nvmoe_set_pdl(int enable) {
  const int old = g_pdl.exchange(enable != 0 ? 1 : 0);
  return old;
}

uint64_t nvmoe_kernel_launch_count(void) { return g_launches.load(); }

int nvmoe_read_status(const void* ws, cudaStream_t stream, int* out) {
  if (ws == nullptr || out == nullptr) return NVMOE_ERR_INVALID_ARG;
  int v = 0;
  cudaError_t e = cudaMemcpyAsync(&v, ws, sizeof(int), cudaMemcpyDeviceToHost, stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return fail(e);
  *out = v;
  return NVMOE_OK;
}

int nvmoe_clear_status(void* ws, cudaStream_t stream) {
  if (ws == nullptr) return NVMOE_ERR_INVALID_ARG;
  return status_of(cudaMemsetAsync(ws, 0, kStatusBytes, stream));
}

size_t nvfp4_sf_mma_bytes(int64_t rows, int64_t cols) {
  if (rows < 0 || cols < 0) return 0;
  return sf_mma_bytes(rows, cols);
}

// ------------------------------------------------------- FP4 probe ----
int nvmoe_fp4_mma_probe(int variant, int iters, int grid, long long* cycles, void* ws,
                        size_t ws_bytes, cudaStream_t stream) {
  const NvtxRange nvtx_range("nvmoe_fp4_mma_probe");
  if (variant < 0 || variant > 2047 || ((variant & kProbeCp32) && (variant & kProbeCp256)))
    return NVMOE_ERR_INVALID_ARG;
  // four accumulators of 128 columns fill the 512 TMEM columns: N = 128 only
  if ((variant & kProbeAcc4) && (!(variant & kProbeN128) || (variant & kProbeAcc2)))
    return NVMOE_ERR_INVALID_ARG;
  if ((variant & kProbeNoMma) && !(variant & (kProbeCp32 | kProbeCp256)))
    return NVMOE_ERR_INVALID_ARG;
  if ((variant & (kProbeCpAOnly | kProbeCpEarly)) && !(variant & kProbeCp256))
    return NVMOE_ERR_INVALID_ARG;
  // the tcgen05.st form: one CTA, whole stages of four MMAs, no other flags
  if ((variant & kProbeSt) && ((variant & ~(kProbeSt | kProbeN128)) || (iters % 4) != 0))
    return NVMOE_ERR_INVALID_ARG;
  if (iters < 1 || iters > (1 << 20) || grid < 1 || grid > 65535 || cycles == nullptr ||
      ws == nullptr)
    return NVMOE_ERR_INVALID_ARG;
  if ((variant & kProbePair) && (grid & 1)) return NVMOE_ERR_INVALID_ARG;
  if (ws_bytes < kStatusBytes) return NVMOE_ERR_WORKSPACE_TOO_SMALL;
  return status_of(counted(launch_mma_probe(variant, iters, grid, cycles, static_cast<int*>(ws),
                                            stream), 1));
}

// ------------------------------------------------------------- route ----
int64_t moe_route_rows_bound(int64_t T, int k, int E) {
  if (T < 0 || k < 1 || E < 1 || !slots_fit(T, k)) return 0;
  return rows_bound(T, k, E);
}

size_t moe_route_workspace_size(int64_t T, int k, int E) {
  if (T < 0 || k < 1 || E < 1 || !slots_fit(T, k)) return 0;
  const int64_t S = T * k;
  const int64_t chunks = S > 0 ? ceil_div(S, route_chunk_elems()) : 1;
  return kStatusBytes + align_up(static_cast<size_t>(chunks) * E * sizeof(int32_t));
}

int moe_route_permute(const int32_t* topk_ids, int64_t T, int k, int E, int32_t* expert_offsets,
                      int32_t* expert_counts, int32_t* row_token, int32_t* slot_of, void* ws,
                      size_t ws_bytes, cudaStream_t stream) {
  const NvtxRange nvtx_range("moe_route_permute");
  if (T < 0 || k < 1 || k > kMaxTopK || E < 1 || E > kMaxExperts) return NVMOE_ERR_INVALID_ARG;
  if (!slots_fit(T, k)) return NVMOE_ERR_UNSUPPORTED_SHAPE;
  if (expert_offsets == nullptr || expert_counts == nullptr || ws == nullptr)
    return NVMOE_ERR_INVALID_ARG;
  if (T > 0 && (topk_ids == nullptr || row_token == nullptr || slot_of == nullptr))
    return NVMOE_ERR_INVALID_ARG;
  if (ws_bytes < moe_route_workspace_size(T, k, E)) return NVMOE_ERR_WORKSPACE_TOO_SMALL;
  const int64_t S = T * k;
  const int n_chunks = static_cast<int>(S > 0 ? ceil_div(S, route_chunk_elems()) : 1);
  Carve c{static_cast<uint8_t*>(ws)};
  int* status = c.take<int>(kStatusBytes);
  int32_t* chunk_counts = c.take<int32_t>(static_cast<size_t>(n_chunks) * E * sizeof(int32_t));
  return status_of(counted(launch_route(topk_ids, T, k, E, expert_offsets, expert_counts, row_token,
                                rows_bound(T, k, E), slot_of, chunk_counts, n_chunks, status,
                                stream), n_chunks == 1 ? 1 : 2));
}

// --------------------------------------------------------- quantiser ----
size_t nvfp4_quantize_workspace_size(int64_t rows, int64_t cols) {
  (void)rows;
  (void)cols;
  return kStatusBytes + align_up(kQuantMaxPartials * sizeof(float));
}

int nvfp4_quantize_act(const void* x, int x_dtype, int64_t rows, int64_t cols,
                       const int32_t* row_dst, int fanout, int64_t out_rows, uint8_t* q,
                       uint8_t* sf_rowmajor, uint8_t* sf_mma, float* gs_out, void* ws,
                       size_t ws_bytes, cudaStream_t stream) {
  const NvtxRange nvtx_range("nvfp4_quantize_act");
  if (rows < 0 || cols <= 0 || out_rows < 0) return NVMOE_ERR_INVALID_ARG;
  if (x_dtype != NVMOE_BF16 && x_dtype != NVMOE_F32) return NVMOE_ERR_INVALID_ARG;
  if (cols % 64 != 0 || !elems_fit(rows, cols) || !elems_fit(out_rows, cols))
    return NVMOE_ERR_UNSUPPORTED_SHAPE;
  if (fanout < 1 || fanout > kMaxTopK) return NVMOE_ERR_INVALID_ARG;
  if (row_dst != nullptr && !slots_fit(rows, fanout)) return NVMOE_ERR_UNSUPPORTED_SHAPE;
  if (row_dst == nullptr && (fanout != 1 || out_rows < rows)) return NVMOE_ERR_INVALID_ARG;
  if (gs_out == nullptr || ws == nullptr) return NVMOE_ERR_INVALID_ARG;
  if (rows > 0 && (x == nullptr || q == nullptr)) return NVMOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(q) || !aligned16(sf_mma) || !aligned16(ws))
    return NVMOE_ERR_MISALIGNED;
  if (ws_bytes < nvfp4_quantize_workspace_size(rows, cols)) return NVMOE_ERR_WORKSPACE_TOO_SMALL;
  Carve c{static_cast<uint8_t*>(ws)};
  int* status = c.take<int>(kStatusBytes);
  float* partial = c.take<float>(kQuantMaxPartials * sizeof(float));
  const int64_t n = rows * cols;
  if (n <= kQuantSmallElems)
    return status_of(counted(launch_quant_small(x, x_dtype, rows, cols, row_dst, fanout, q,
                                                sf_rowmajor, sf_mma, gs_out, out_rows, status,
                                                stream), 1));
  const int parts = quant_amax_blocks(n);
  cudaError_t e = counted(launch_quant_amax(x, x_dtype, n, partial, parts, stream), 1);
  if (e != cudaSuccess) return fail(e);
  // both scale layouts asked for: the quantiser writes the row-major one
  // (whole sectors) and one pass over it writes the staged one (whole
  // atoms), which is faster than the quantiser's scattered 4-byte staged
  // words, at large sizes by about a third of the quantiser's time
  const bool staged_after = sf_mma != nullptr && sf_rowmajor != nullptr && cols % kStageK == 0 &&
                            aligned16(sf_rowmajor);
  e = counted(launch_quant_pack(x, x_dtype, rows, cols, row_dst, fanout, nullptr, partial, parts,
                                q, sf_rowmajor, staged_after ? nullptr : sf_mma, gs_out, out_rows,
                                status, stream), 1);
  if (e != cudaSuccess || !staged_after) return status_of(e);
  return status_of(counted(launch_stage_act_sf(sf_rowmajor, out_rows, cols, sf_mma, stream), 1));
}

int nvfp4_amax(const void* x, int x_dtype, int64_t rows, int64_t cols, float* amax_out, void* ws,
               size_t ws_bytes, cudaStream_t stream) {
  const NvtxRange nvtx_range("nvfp4_amax");
  if (rows < 0 || cols <= 0) return NVMOE_ERR_INVALID_ARG;
  if (x_dtype != NVMOE_BF16 && x_dtype != NVMOE_F32) return NVMOE_ERR_INVALID_ARG;
  if (cols % 64 != 0 || !elems_fit(rows, cols)) return NVMOE_ERR_UNSUPPORTED_SHAPE;
  if (amax_out == nullptr || ws == nullptr || (rows > 0 && x == nullptr))
    return NVMOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(ws)) return NVMOE_ERR_MISALIGNED;
  if (ws_bytes < nvfp4_quantize_workspace_size(rows, cols)) return NVMOE_ERR_WORKSPACE_TOO_SMALL;
  Carve c{static_cast<uint8_t*>(ws)};
  c.take<int>(kStatusBytes);
  float* partial = c.take<float>(kQuantMaxPartials * sizeof(float));
  const int64_t n = rows * cols;
  int parts = 0;
  if (n > 0) {
    parts = quant_amax_blocks(n);
    const cudaError_t e = counted(launch_quant_amax(x, x_dtype, n, partial, parts, stream), 1);
    if (e != cudaSuccess) return fail(e);
  }
  return status_of(counted(launch_max_reduce(partial, parts, amax_out, stream), 1));
}

int nvfp4_quantize_act_amax(const void* x, int x_dtype, int64_t rows, int64_t cols,
                            const int32_t* row_dst, int fanout, int64_t out_rows,
                            const float* amax_in, uint8_t* q, uint8_t* sf_rowmajor,
                            uint8_t* sf_mma, float* gs_out, cudaStream_t stream) {
  const NvtxRange nvtx_range("nvfp4_quantize_act_amax");
  if (rows < 0 || cols <= 0 || out_rows < 0) return NVMOE_ERR_INVALID_ARG;
  if (x_dtype != NVMOE_BF16 && x_dtype != NVMOE_F32) return NVMOE_ERR_INVALID_ARG;
  if (cols % 64 != 0 || !elems_fit(rows, cols) || !elems_fit(out_rows, cols))
    return NVMOE_ERR_UNSUPPORTED_SHAPE;
  if (fanout < 1 || fanout > kMaxTopK) return NVMOE_ERR_INVALID_ARG;
  if (row_dst != nullptr && !slots_fit(rows, fanout)) return NVMOE_ERR_UNSUPPORTED_SHAPE;
  if (row_dst == nullptr && (fanout != 1 || out_rows < rows)) return NVMOE_ERR_INVALID_ARG;
  if (gs_out == nullptr || amax_in == nullptr) return NVMOE_ERR_INVALID_ARG;
  if (rows > 0 && (x == nullptr || q == nullptr)) return NVMOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(q) || !aligned16(sf_mma)) return NVMOE_ERR_MISALIGNED;
  return status_of(counted(launch_quant_pack(x, x_dtype, rows, cols, row_dst, fanout, nullptr,
                                             amax_in, 1, q, sf_rowmajor, sf_mma, gs_out, out_rows,
                                             nullptr, stream), 1));
}

// ----------------------------------------------------------- weights ----
size_t nvfp4_quantize_weights_workspace_size(int E, int K, int N) {
  (void)K;
  (void)N;
  if (E < 1) return 0;
  return kStatusBytes + align_up(static_cast<size_t>(E) * 64 * sizeof(float));
}

int nvfp4_quantize_weights(const float* w, int E, int K, int N, uint8_t* q, uint8_t* sf,
                           float* gs, void* ws, size_t ws_bytes, cudaStream_t stream) {
  const NvtxRange nvtx_range("nvfp4_quantize_weights");
  if (E < 1 || K < 1 || N < 1 || w == nullptr || q == nullptr || sf == nullptr ||
      gs == nullptr || ws == nullptr)
    return NVMOE_ERR_INVALID_ARG;
  if (K % 64 != 0 || E > 65535) return NVMOE_ERR_UNSUPPORTED_SHAPE;
  if (!aligned16(w) || !aligned16(ws)) return NVMOE_ERR_MISALIGNED;
  if (ws_bytes < nvfp4_quantize_weights_workspace_size(E, K, N))
    return NVMOE_ERR_WORKSPACE_TOO_SMALL;
  Carve c{static_cast<uint8_t*>(ws)};
  c.take<int>(kStatusBytes);
  float* partial = c.take<float>(static_cast<size_t>(E) * 64 * sizeof(float));
  cudaError_t e = counted(launch_weight_amax(w, E, static_cast<int64_t>(K) * N, partial, 64, stream), 1);
  if (e != cudaSuccess) return fail(e);
  return status_of(counted(launch_weight_quant(w, E, K, N, partial, 64, q, sf, gs, stream), 1));
}

size_t moe_nvfp4_prepared_bytes(int E, int K, int N) {
  if (E < 1 || K < 1 || N < 1) return 0;
  return static_cast<size_t>(E) * N * ceil_div(K, kStageK) * 128;
}

int moe_nvfp4_prepare_weights(const uint8_t* q_ckpt, const uint8_t* sf_ckpt, int E, int K, int N,
                              uint8_t* q_out, uint8_t* sf_out, cudaStream_t stream) {
  const NvtxRange nvtx_range("moe_nvfp4_prepare_weights");
  if (E < 1 || K < 1 || N < 1 || q_ckpt == nullptr || sf_ckpt == nullptr ||
      q_out == nullptr || sf_out == nullptr)
    return NVMOE_ERR_INVALID_ARG;
  if (K % 64 != 0 || N % kTileRows != 0 || E > 65535) return NVMOE_ERR_UNSUPPORTED_SHAPE;
  return status_of(counted(launch_prepare_weights(q_ckpt, sf_ckpt, E, K, N, q_out, sf_out, stream), 2));
}

// ----------------------------------------------------------- forward ----
struct FwdBuffers {
  int* status;
  int* counters;      // [2][kMaxSplitTiles]: split-tile arrivals of L1 and of L2
  int* grid_bar;      // fused kernel's grid barrier words
  float* pieces;      // split-tile partial accumulators
  float* h;
  uint8_t* hq;
  uint8_t* hsf;
  float* gs_h;
  float* amax;        // per-CTA maxima of |h|
};

static size_t forward_layout(int64_t T, int k, int E, int I, uint8_t* base, FwdBuffers* b) {
  Carve c{base};
  const int64_t rows = rows_bound(T, k, E);
  b->status = c.take<int>(kStatusBytes);
  b->counters = c.take<int>(2 * kMaxSplitTiles * sizeof(int));
  b->grid_bar = c.take<int>(2 * sizeof(int));
  b->pieces = c.take<float>(static_cast<size_t>(2) * kMaxGrid * 128 * 256 * sizeof(float));
  b->h = c.take<float>(static_cast<size_t>(rows) * I * sizeof(float));
  b->hq = c.take<uint8_t>(static_cast<size_t>(rows) * (I / 2));
  b->hsf = c.take<uint8_t>(sf_mma_bytes(rows, I));
  b->gs_h = c.take<float>(sizeof(float));
  b->amax = c.take<float>(kQuantMaxPartials * sizeof(float));
  return c.off;
}

size_t moe_nvfp4_workspace_size(int64_t T, int k, int E, int H, int I) {
  if (T < 0 || k < 1 || E < 1 || H < 1 || I < 1 || !slots_fit(T, k)) return 0;
  FwdBuffers b;
  return forward_layout(T, k, E, I, nullptr, &b);
}

// Steps 3-6 (and, with `layer`, the whole layer in one launch).
static int forward_impl(const nvmoe_weights* w, const uint8_t* xq, const uint8_t* xsf_mma,
                        const float* gs_x, const int32_t* expert_offsets,
                        const int32_t* expert_counts, const int32_t* row_token, int64_t T, int k,
                        void* slot_out, int slot_out_dtype, const nvmoe_taps* taps, void* ws,
                        size_t ws_bytes, cudaStream_t stream, LayerLaunch* layer,
                        int phase = 0, float* amax_h = nullptr);

int moe_nvfp4_forward(const nvmoe_weights* w, const uint8_t* xq, const uint8_t* xsf_mma,
                      const float* gs_x, const int32_t* expert_offsets,
                      const int32_t* expert_counts, const int32_t* row_token, int64_t T, int k,
                      void* slot_out, int slot_out_dtype, const nvmoe_taps* taps, void* ws,
                      size_t ws_bytes, cudaStream_t stream) {
  const NvtxRange nvtx_range("moe_nvfp4_forward");
  if (taps != nullptr && taps->path == NVMOE_PATH_LAYER) return NVMOE_ERR_INVALID_ARG;
  return forward_impl(w, xq, xsf_mma, gs_x, expert_offsets, expert_counts, row_token, T, k,
                      slot_out, slot_out_dtype, taps, ws, ws_bytes, stream, nullptr);
}

int moe_nvfp4_forward_phase(const nvmoe_weights* w, const uint8_t* xq, const uint8_t* xsf_mma,
                            const float* gs_x, const int32_t* expert_offsets,
                            const int32_t* expert_counts, const int32_t* row_token, int64_t T,
                            int k, void* slot_out, int slot_out_dtype, int phase, float* amax_h,
                            const nvmoe_taps* taps, void* ws, size_t ws_bytes,
                            cudaStream_t stream) {
  const NvtxRange nvtx_range("moe_nvfp4_forward_phase");
  if (phase != 1 && phase != 2) return NVMOE_ERR_INVALID_ARG;
  if (taps != nullptr && taps->path == NVMOE_PATH_LAYER) return NVMOE_ERR_INVALID_ARG;
  return forward_impl(w, xq, xsf_mma, gs_x, expert_offsets, expert_counts, row_token, T, k,
                      slot_out, slot_out_dtype, taps, ws, ws_bytes, stream, nullptr, phase,
                      amax_h);
}

static int forward_impl(const nvmoe_weights* w, const uint8_t* xq, const uint8_t* xsf_mma,
                        const float* gs_x, const int32_t* expert_offsets,
                        const int32_t* expert_counts, const int32_t* row_token, int64_t T, int k,
                        void* slot_out, int slot_out_dtype, const nvmoe_taps* taps, void* ws,
                        size_t ws_bytes, cudaStream_t stream, LayerLaunch* layer, int phase,
                        float* amax_h) {
  if (w == nullptr || T < 0 || k < 1 || k > kMaxTopK) return NVMOE_ERR_INVALID_ARG;
  if (phase < 0 || phase > 2 || (phase != 0 && (layer != nullptr || amax_h == nullptr)))
    return NVMOE_ERR_INVALID_ARG;
  if (slot_out_dtype != NVMOE_BF16 && slot_out_dtype != NVMOE_F32 && slot_out_dtype != NVMOE_F16)
    return NVMOE_ERR_INVALID_ARG;
  // the single-kernel layer path reduces from fp32 slot rows inside the kernel
  if (layer != nullptr && slot_out_dtype != NVMOE_F32) return NVMOE_ERR_INVALID_ARG;
  const int E = w->E, H = w->H, I = w->I;
  if (E < 1 || E > kMaxExperts || H < 1 || I < 1) return NVMOE_ERR_INVALID_ARG;
  if (H % 256 != 0 || I % 128 != 0 || !slots_fit(T, k)) return NVMOE_ERR_UNSUPPORTED_SHAPE;
  if (w->w1 == nullptr || w->w1_sf == nullptr || w->gs_w1 == nullptr || w->w2 == nullptr ||
      w->w2_sf == nullptr || w->gs_w2 == nullptr || xq == nullptr || xsf_mma == nullptr ||
      gs_x == nullptr || expert_offsets == nullptr || expert_counts == nullptr ||
      row_token == nullptr || slot_out == nullptr || ws == nullptr)
    return NVMOE_ERR_INVALID_ARG;
  if (!aligned16(w->w1) || !aligned16(w->w2) || !aligned16(w->w1_sf) || !aligned16(w->w2_sf) ||
      !aligned16(xq) || !aligned16(xsf_mma) || !aligned16(slot_out) || !aligned16(ws))
    return NVMOE_ERR_MISALIGNED;
  if (ws_bytes < moe_nvfp4_workspace_size(T, k, E, H, I)) return NVMOE_ERR_WORKSPACE_TOO_SMALL;
  int path = NVMOE_PATH_AUTO;
  if (taps != nullptr) path = taps->path;
  if (path != NVMOE_PATH_AUTO && path != NVMOE_PATH_SEPARATE && path != NVMOE_PATH_FUSED &&
      path != NVMOE_PATH_LAYER && path != NVMOE_PATH_SEPARATE_SINGLE)
    return NVMOE_ERR_INVALID_ARG;
  const bool allow_pair = path != NVMOE_PATH_SEPARATE_SINGLE;
  if (path == NVMOE_PATH_SEPARATE_SINGLE) path = NVMOE_PATH_SEPARATE;
  if (phase != 0) path = NVMOE_PATH_SEPARATE;   // the phases are the three-launch path, split
  if (T == 0) {
    // an empty batch still reports max |h| = 0 (the caller reduces it over ranks)
    if (phase == 1) return status_of(counted(launch_max_reduce(nullptr, 0, amax_h, stream), 1));
    return NVMOE_OK;
  }
  FwdBuffers b;
  forward_layout(T, k, E, I, static_cast<uint8_t*>(ws), &b);
  float* tap_l1 = nullptr;
  cudaEvent_t ev[4] = {nullptr, nullptr, nullptr, nullptr};
  if (taps != nullptr) {
    for (int i = 0; i < 4; ++i) ev[i] = taps->stage_events[i];
    if (taps->h != nullptr) b.h = taps->h;
    if (taps->hq != nullptr) b.hq = taps->hq;
    if (taps->hsf_mma != nullptr) b.hsf = taps->hsf_mma;
    if (taps->gs_h != nullptr) b.gs_h = taps->gs_h;
    tap_l1 = taps->l1_out;
    if (!aligned16(b.h) || !aligned16(b.hq) || !aligned16(b.hsf) || !aligned16(tap_l1))
      return NVMOE_ERR_MISALIGNED;
  }
  const int64_t rows = rows_bound(T, k, E);
  int nsm = sm_count();
  if (nsm <= 0) return fail(cudaErrorNoDevice);
  if (nsm > kMaxGrid) nsm = kMaxGrid;

  AMaps map_x, map_h;
  CUtensorMap map_w1, map_w2;
  const int64_t kt1 = ceil_div(H, kStageK), kt2 = ceil_div(I, kStageK);
  if (!make_map(&map_x.full, xq, H / 2, rows) ||
      !make_map(&map_x.small, xq, H / 2, rows, kSmallABoxRows) ||
      !make_tiled_map(&map_w1, w->w1, int64_t(E) * 2 * I / kTileRows * kt1) ||
      !make_map(&map_h.full, b.hq, I / 2, rows) ||
      !make_map(&map_h.small, b.hq, I / 2, rows, kSmallABoxRows) ||
      !make_tiled_map(&map_w2, w->w2, int64_t(E) * H / kTileRows * kt2))
    return fail(cudaErrorInvalidValue);  // tensor-map encoding refused

  GemmArgs a1{};
  a1.mode = 1;
  a1.E = E;
  a1.K = H;
  a1.N = 2 * I;
  a1.I = I;
  a1.n_tiles = I / 128;
  a1.expert_offsets = expert_offsets;
  a1.expert_counts = expert_counts;
  a1.a_sf = xsf_mma;
  a1.b_sf = w->w1_sf;
  a1.gs_a = gs_x;
  a1.gs_b = w->gs_w1;
  a1.gs_b_up = w->gs_w1_up;
  a1.gs_mid = w->gs_mid;
  a1.mid_q = b.hq;
  a1.mid_sf = b.hsf;
  // the layer kernel requantises after its grid barrier, spread over the grid
  a1.mid_in_epilogue = layer == nullptr;
  a1.out = b.h;
  a1.out_dtype = NVMOE_F32;
  a1.tap = tap_l1;
  a1.amax_partial = b.amax;
  a1.partials = b.pieces;
  a1.counters = b.counters;
  a1.status = b.status;
  a1.rows = rows;
  if (taps != nullptr && taps->ready_flag != nullptr) {
    a1.ready_flag = taps->ready_flag;
    a1.ready_value = taps->ready_value;
    a1.ready_limit_ns = taps->ready_wait_us > 0
                            ? static_cast<uint64_t>(taps->ready_wait_us) * 1000u
                            : 2000000000ull;
  }
  GemmArgs a2{};
  a2.mode = 2;
  a2.E = E;
  a2.K = I;
  a2.N = H;
  a2.I = I;
  a2.n_tiles = H / 256;
  a2.expert_offsets = expert_offsets;
  a2.expert_counts = expert_counts;
  a2.a_sf = b.hsf;
  a2.b_sf = w->w2_sf;
  a2.gs_a = b.gs_h;
  a2.gs_b = w->gs_w2;
  a2.gs_mid = w->gs_mid;
  a2.out = static_cast<float*>(slot_out);
  a2.out_dtype = slot_out_dtype;
  a2.tap = nullptr;
  a2.amax_partial = nullptr;
  a2.partials = b.pieces;
  a2.counters = b.counters + kMaxSplitTiles;
  a2.status = b.status;
  a2.rows = rows;

  // Tiles that can exist, from the host-side bound on expert segments.
  const int64_t S = T * k;
  const int64_t mt_bound = S / kTileRows + (S < E ? S : E);
  const int64_t tiles1 = mt_bound * a1.n_tiles, tiles2 = mt_bound * a2.n_tiles;
  // and the tiles that exist whatever the routing: every segment of c rows
  // takes ceil(c / 128) m-tiles, at least ceil(S / 128) over all experts
  const int64_t mt_min = (S + kTileRows - 1) / kTileRows;
  auto grid_for = [&](int64_t tiles) {
    int64_t g = tiles < nsm ? tiles : nsm;
    return static_cast<int>(g < 1 ? 1 : g);
  };
  // Few tiles (decode): one cooperative kernel for L1 -> requantise -> L2.
  const bool fused = path == NVMOE_PATH_FUSED ||
                     (path == NVMOE_PATH_AUTO && tiles1 < 4 * int64_t(nsm) && tiles2 < 4 * int64_t(nsm));
  const bool timed = ev[0] && ev[1] && ev[2] && ev[3];
  if (timed && note(cudaEventRecord(ev[0], stream)) != cudaSuccess) return NVMOE_ERR_CUDA;
  if (layer != nullptr) {
    layer->hq = b.hq;
    layer->hsf = b.hsf;
    layer->gs_h = b.gs_h;
    const int g = grid_for(tiles1 > tiles2 ? tiles1 : tiles2);
    cudaError_t e = counted(launch_layer(a1, a2, map_x, map_w1, map_h, map_w2, *layer, g, stream), 1);
    if (e != cudaSuccess) return fail(e);
    if (timed)
      for (int i = 1; i < 4; ++i)
        if (note(cudaEventRecord(ev[i], stream)) != cudaSuccess) return NVMOE_ERR_CUDA;
    return NVMOE_OK;
  }
  if (fused) {
    const int g = grid_for(tiles1 > tiles2 ? tiles1 : tiles2);
    cudaError_t e = counted(launch_fused_ffn(a1, a2, map_x, map_w1, map_h, map_w2, b.grid_bar,
                                             row_token, b.hq, b.hsf, b.gs_h, g, stream), 1);
    if (e != cudaSuccess) return fail(e);
    if (timed) {
      // one kernel: L1, requantisation and L2 are not separable
      for (int i = 1; i < 4; ++i)
        if (note(cudaEventRecord(ev[i], stream)) != cudaSuccess) return NVMOE_ERR_CUDA;
    }
    return NVMOE_OK;
  }
  const int g1 = grid_for(tiles1);
  cudaError_t e = cudaSuccess;
  if (phase != 2) {
    e = counted(launch_gemm(a1, map_x, map_w1, g1, mt_min * a1.n_tiles, allow_pair, stream), 1);
    if (e != cudaSuccess) return fail(e);
    if (timed && note(cudaEventRecord(ev[1], stream)) != cudaSuccess) return NVMOE_ERR_CUDA;
  }
  if (phase == 1) {
    // max |h| of this call's rows, for the caller to reduce before phase 2
    return status_of(counted(launch_max_reduce(b.amax, g1, amax_h, stream), 1));
  }
  if (w->gs_mid == nullptr) {
    // requantise h over the valid rows (global amax from the L1 partials, or
    // in phase 2 the caller's amax); with a static intermediate scale the L1
    // epilogue has done it
    const float* amax_src = phase == 2 ? amax_h : b.amax;
    const int n_amax = phase == 2 ? 1 : g1;
    e = counted(launch_quant_pack(b.h, NVMOE_F32, rows, I, nullptr, 1, row_token, amax_src, n_amax,
                                  b.hq, nullptr, b.hsf, b.gs_h, rows, b.status, stream), 1);
    if (e != cudaSuccess) return fail(e);
  }
  if (timed && note(cudaEventRecord(ev[2], stream)) != cudaSuccess) return NVMOE_ERR_CUDA;
  e = counted(launch_gemm(a2, map_h, map_w2, grid_for(tiles2), mt_min * a2.n_tiles, allow_pair,
                                  stream), 1);
  if (e != cudaSuccess) return fail(e);
  if (timed && note(cudaEventRecord(ev[3], stream)) != cudaSuccess) return NVMOE_ERR_CUDA;
  return NVMOE_OK;
}

// --------------------------------------------------- expert parallel ----
namespace {
struct EpBuffers {
  uint8_t* route_ws;
  size_t route_ws_bytes;
  int32_t* dest;
  int32_t* padded;
  int32_t* offsets;
  int32_t* row_token;
};

size_t ep_layout(int64_t T, int k, int G, uint8_t* base, EpBuffers* b) {
  const int64_t S = T * k;
  Carve c{base};
  b->route_ws_bytes = moe_route_workspace_size(T, k, G);
  b->route_ws = c.take<uint8_t>(b->route_ws_bytes);          // its status word comes first
  b->dest = c.take<int32_t>(static_cast<size_t>(S > 0 ? S : 1) * sizeof(int32_t));
  b->padded = c.take<int32_t>(static_cast<size_t>(S > 0 ? S : 1) * sizeof(int32_t));
  b->offsets = c.take<int32_t>(static_cast<size_t>(G + 1) * sizeof(int32_t));
  const int64_t rows = rows_bound(T, k, G);
  b->row_token = c.take<int32_t>(static_cast<size_t>(rows > 0 ? rows : 1) * sizeof(int32_t));
  return c.off;
}
}  // namespace

size_t moe_ep_dispatch_workspace_size(int64_t T, int k, int G) {
  if (T < 0 || k < 1 || G < 1 || G > kMaxExperts || !slots_fit(T, k)) return 0;
  EpBuffers b;
  return ep_layout(T, k, G, nullptr, &b);
}

int moe_ep_dispatch(const int32_t* topk_ids, int64_t T, int k, int E, int G, const uint8_t* q_tok,
                    const uint8_t* sf_tok, int H, int32_t* send_counts, int32_t* send_pos,
                    uint8_t* send_rows, int32_t* send_expert, void* ws, size_t ws_bytes,
                    cudaStream_t stream) {
  const NvtxRange nvtx_range("moe_ep_dispatch");
  if (T < 0 || k < 1 || k > kMaxTopK || E < 1 || E > kMaxExperts || G < 1 || G > E || E % G != 0)
    return NVMOE_ERR_INVALID_ARG;
  if (H < 1 || H % 256 != 0 || !slots_fit(T, k)) return NVMOE_ERR_UNSUPPORTED_SHAPE;
  if (send_counts == nullptr || ws == nullptr) return NVMOE_ERR_INVALID_ARG;
  if (T > 0 && (topk_ids == nullptr || q_tok == nullptr || sf_tok == nullptr ||
                send_pos == nullptr || send_rows == nullptr || send_expert == nullptr))
    return NVMOE_ERR_INVALID_ARG;
  if (!aligned16(q_tok) || !aligned16(sf_tok) || !aligned16(send_rows) || !aligned16(ws))
    return NVMOE_ERR_MISALIGNED;
  if (ws_bytes < moe_ep_dispatch_workspace_size(T, k, G)) return NVMOE_ERR_WORKSPACE_TOO_SMALL;
  EpBuffers b;
  ep_layout(T, k, G, static_cast<uint8_t*>(ws), &b);
  const int64_t S = T * k;
  int* status = reinterpret_cast<int*>(b.route_ws);
  if (S > 0) {
    const cudaError_t e = counted(launch_ep_dest(topk_ids, S, E, G, b.dest, status, stream), 1);
    if (e != cudaSuccess) return fail(e);
  }
  // counting sort of the slots by destination (stable in t*k + j), the
  // routing kernels with ranks for experts; send_counts = the true counts
  const int st = moe_route_permute(b.dest, T, k, G, b.offsets, send_counts, b.row_token, b.padded,
                                   b.route_ws, b.route_ws_bytes, stream);
  if (st != NVMOE_OK || S == 0) return st;
  return status_of(counted(launch_ep_pack(topk_ids, b.padded, b.dest, b.offsets, send_counts, S, k,
                                          E, G, q_tok, sf_tok, H, send_pos, send_rows,
                                          send_expert, stream), 1));
}

int moe_ep_scatter(const uint8_t* recv_rows, int64_t n, int H, const int32_t* slot_of,
                   int64_t out_rows, uint8_t* xq, uint8_t* xsf_mma, int* status,
                   cudaStream_t stream) {
  const NvtxRange nvtx_range("moe_ep_scatter");
  if (n < 0 || out_rows < 0) return NVMOE_ERR_INVALID_ARG;
  if (H < 1 || H % 256 != 0 || !elems_fit(out_rows, H)) return NVMOE_ERR_UNSUPPORTED_SHAPE;
  if (n == 0) return NVMOE_OK;
  if (recv_rows == nullptr || slot_of == nullptr || xq == nullptr || xsf_mma == nullptr)
    return NVMOE_ERR_INVALID_ARG;
  if (!aligned16(recv_rows) || !aligned16(xq) || !aligned16(xsf_mma)) return NVMOE_ERR_MISALIGNED;
  const int k_atoms = static_cast<int>(round_up(H, kStageK) / 64);
  return status_of(counted(launch_ep_scatter(recv_rows, n, H, slot_of, out_rows, xq, xsf_mma,
                                             k_atoms, status, stream), 1));
}

int moe_ep_gather(const void* slot_out, int slot_out_dtype, int H, int64_t slot_rows,
                  const int32_t* slot_of, int64_t n, void* out_rows, int* status,
                  cudaStream_t stream) {
  const NvtxRange nvtx_range("moe_ep_gather");
  if (n < 0 || H < 1 || slot_rows < 0) return NVMOE_ERR_INVALID_ARG;
  if (slot_out_dtype != NVMOE_BF16 && slot_out_dtype != NVMOE_F32 && slot_out_dtype != NVMOE_F16)
    return NVMOE_ERR_INVALID_ARG;
  const int64_t row_bytes = static_cast<int64_t>(H) * (slot_out_dtype == NVMOE_F32 ? 4 : 2);
  if (row_bytes % 16 != 0) return NVMOE_ERR_UNSUPPORTED_SHAPE;
  if (n == 0) return NVMOE_OK;
  if (slot_out == nullptr || slot_of == nullptr || out_rows == nullptr) return NVMOE_ERR_INVALID_ARG;
  if (!aligned16(slot_out) || !aligned16(out_rows)) return NVMOE_ERR_MISALIGNED;
  return status_of(counted(launch_ep_gather(slot_out, row_bytes, slot_rows, slot_of, n, out_rows,
                                            status, stream), 1));
}

// ------------------------------------------------------------ router ----
size_t moe_router_workspace_size(int64_t T, int H, int E) {
  if (T < 0 || H < 1 || E < 1 || !elems_fit(T, H)) return 0;
  return kStatusBytes + align_up(router_workspace_bytes(T, H, E));
}

int moe_router_topk(const void* x, const void* w_router, int64_t T, int H, int E, int k,
                    int softmax_mode, int32_t* topk_ids, float* topk_w, void* ws,
                    size_t ws_bytes, cudaStream_t stream) {
  const NvtxRange nvtx_range("moe_router_topk");
  if (T < 0 || H < 1 || E < 1 || E > kMaxExperts || k < 1 || k > kMaxTopK || k > E)
    return NVMOE_ERR_INVALID_ARG;
  if (softmax_mode != NVMOE_ROUTER_SELECTED && softmax_mode != NVMOE_ROUTER_ALL)
    return NVMOE_ERR_INVALID_ARG;
  if (H % 128 != 0 || !elems_fit(T, H) || !slots_fit(T, E)) return NVMOE_ERR_UNSUPPORTED_SHAPE;
  if (T == 0) return NVMOE_OK;
  if (x == nullptr || w_router == nullptr || topk_ids == nullptr || topk_w == nullptr ||
      ws == nullptr)
    return NVMOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(w_router) || !aligned16(ws)) return NVMOE_ERR_MISALIGNED;
  if (ws_bytes < moe_router_workspace_size(T, H, E)) return NVMOE_ERR_WORKSPACE_TOO_SMALL;
  // x and the weight as byte matrices [rows, 2H]: 64 bf16 per 128-byte box
  // row; the weight box spans E rounded up to 16 rows (the rows past E are
  // filled with zeros)
  CUtensorMap map_x, map_w;
  if (!make_map(&map_x, x, int64_t{2} * H, T, 128) ||
      !make_map(&map_w, w_router, int64_t{2} * H, E, static_cast<uint32_t>((E + 15) / 16 * 16)))
    return fail(cudaErrorInvalidValue);  // tensor-map encoding refused
  Carve c{static_cast<uint8_t*>(ws)};
  int* status = c.take<int>(kStatusBytes);
  float* partials = c.take<float>(router_workspace_bytes(T, H, E));
  return status_of(counted(launch_router(map_x, map_w, T, H, E, k, softmax_mode, topk_ids,
                                         topk_w, partials, status, stream),
                           2));
}

// ------------------------------------------------------------ reduce ----
int moe_unpermute_reduce(const void* slot_out, int slot_out_dtype, const int32_t* slot_of,
                         const float* topk_w, int64_t T, int k, int64_t H, void* y, int y_dtype,
                         cudaStream_t stream) {
  const NvtxRange nvtx_range("moe_unpermute_reduce");
  if (T < 0 || k < 1 || k > kMaxTopK || H < 1) return NVMOE_ERR_INVALID_ARG;
  if (y_dtype != NVMOE_BF16 && y_dtype != NVMOE_F32) return NVMOE_ERR_INVALID_ARG;
  if (slot_out_dtype != NVMOE_BF16 && slot_out_dtype != NVMOE_F32 && slot_out_dtype != NVMOE_F16)
    return NVMOE_ERR_INVALID_ARG;
  if (H % 8 != 0 || !slots_fit(T, k) || !elems_fit(T, H)) return NVMOE_ERR_UNSUPPORTED_SHAPE;
  if (T == 0) return NVMOE_OK;
  if (slot_out == nullptr || slot_of == nullptr || topk_w == nullptr || y == nullptr)
    return NVMOE_ERR_INVALID_ARG;
  if (!aligned16(slot_out) || !aligned16(y)) return NVMOE_ERR_MISALIGNED;
  return status_of(counted(launch_reduce(slot_out, slot_out_dtype, slot_of, topk_w, T, k, H, y,
                                         y_dtype, stream), 1));
}

// ------------------------------------------------------------- layer ----
struct LayerBuffers {
  uint8_t* fwd_ws;        // first: its status word is the layer workspace's
  size_t fwd_ws_bytes;
  int32_t* offsets;
  int32_t* counts;
  int32_t* row_token;
  int32_t* slot_of;
  uint8_t* route_ws;
  size_t route_ws_bytes;
  uint8_t* xq;
  uint8_t* xsf;
  float* gs_x;
  uint8_t* quant_ws;
  size_t quant_ws_bytes;
  void* slot_out;          // fp32 (single-kernel path) or bf16 rows
  int* grid_bar;
  int* ycnt;
};

static size_t layer_layout(int64_t T, int k, int E, int H, int I, uint8_t* base,
                           LayerBuffers* b) {
  Carve c{base};
  const int64_t rows = rows_bound(T, k, E);
  b->fwd_ws_bytes = moe_nvfp4_workspace_size(T, k, E, H, I);
  b->fwd_ws = c.take<uint8_t>(b->fwd_ws_bytes);
  b->offsets = c.take<int32_t>((E + 1) * sizeof(int32_t));
  b->counts = c.take<int32_t>(E * sizeof(int32_t));
  b->row_token = c.take<int32_t>((rows > 0 ? rows : 1) * sizeof(int32_t));
  b->slot_of = c.take<int32_t>((T * k > 0 ? T * k : 1) * sizeof(int32_t));
  b->route_ws_bytes = moe_route_workspace_size(T, k, E);
  b->route_ws = c.take<uint8_t>(b->route_ws_bytes);
  b->xq = c.take<uint8_t>(static_cast<size_t>(rows) * (H / 2));
  b->xsf = c.take<uint8_t>(sf_mma_bytes(rows, H));
  b->gs_x = c.take<float>(sizeof(float));
  b->quant_ws_bytes = nvfp4_quantize_workspace_size(T, H);
  b->quant_ws = c.take<uint8_t>(b->quant_ws_bytes);
  b->slot_out = c.take<uint8_t>(static_cast<size_t>(rows) * H * sizeof(float));
  b->grid_bar = c.take<int>(kLayerBarWords * sizeof(int));
  b->ycnt = c.take<int>(static_cast<size_t>(T > 0 ? T : 1) * (H / 256 + 1) * sizeof(int));
  return c.off;
}

size_t moe_nvfp4_layer_workspace_size(int64_t T, int k, int E, int H, int I) {
  if (T < 0 || k < 1 || E < 1 || H < 1 || I < 1 || !slots_fit(T, k)) return 0;
  LayerBuffers b;
  return layer_layout(T, k, E, H, I, nullptr, &b);
}

int moe_nvfp4_layer_forward(const nvmoe_weights* w, const void* x, int x_dtype,
                            const int32_t* topk_ids, const float* topk_w, int64_t T, int k,
                            void* y, int y_dtype, const nvmoe_taps* taps, void* ws,
                            size_t ws_bytes, cudaStream_t stream) {
  const NvtxRange nvtx_range("moe_nvfp4_layer_forward");
  if (w == nullptr || T < 0 || k < 1 || k > kMaxTopK) return NVMOE_ERR_INVALID_ARG;
  const int E = w->E, H = w->H, I = w->I;
  if (E < 1 || E > kMaxExperts || H < 1 || I < 1) return NVMOE_ERR_INVALID_ARG;
  if (x_dtype != NVMOE_BF16 && x_dtype != NVMOE_F32) return NVMOE_ERR_INVALID_ARG;
  if (y_dtype != NVMOE_BF16 && y_dtype != NVMOE_F32) return NVMOE_ERR_INVALID_ARG;
  if (H % 256 != 0 || I % 128 != 0 || !slots_fit(T, k)) return NVMOE_ERR_UNSUPPORTED_SHAPE;
  if (ws == nullptr) return NVMOE_ERR_INVALID_ARG;
  if (T > 0 && (x == nullptr || topk_ids == nullptr || topk_w == nullptr || y == nullptr))
    return NVMOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(y) || !aligned16(ws)) return NVMOE_ERR_MISALIGNED;
  if (ws_bytes < moe_nvfp4_layer_workspace_size(T, k, E, H, I))
    return NVMOE_ERR_WORKSPACE_TOO_SMALL;
  const int path = taps != nullptr ? taps->path : NVMOE_PATH_AUTO;
  if (taps != nullptr && taps->ready_flag != nullptr) return NVMOE_ERR_INVALID_ARG;
  if (T == 0) return NVMOE_OK;
  LayerBuffers b;
  layer_layout(T, k, E, H, I, static_cast<uint8_t*>(ws), &b);
  int32_t* slot_of = (taps != nullptr && taps->slot_of != nullptr) ? taps->slot_of : b.slot_of;
  const int64_t S = T * k;
  const int64_t rows = rows_bound(T, k, E);

  int nsm = sm_count();
  if (nsm <= 0) return fail(cudaErrorNoDevice);
  const int64_t mt_bound = S / kTileRows + (S < E ? S : E);
  const bool small = x_dtype == NVMOE_BF16 && S <= kLayerMaxSlots &&
                     T * H <= kQuantSmallElems && mt_bound * (I / 128) < 4 * int64_t(nsm) &&
                     mt_bound * (H / 256) < 4 * int64_t(nsm);
  if (path == NVMOE_PATH_LAYER && !small) return NVMOE_ERR_UNSUPPORTED_SHAPE;
  if (path == NVMOE_PATH_LAYER || (path == NVMOE_PATH_AUTO && small)) {
    LayerLaunch l{};
    l.x = x;
    l.topk_ids = topk_ids;
    l.topk_w = topk_w;
    l.T = static_cast<int>(T);
    l.k = k;
    l.rows = rows;
    l.xq = b.xq;
    l.xsf = b.xsf;
    l.gs_x = b.gs_x;
    l.expert_offsets = b.offsets;
    l.expert_counts = b.counts;
    l.row_token = b.row_token;
    l.slot_of = slot_of;
    l.grid_bar = b.grid_bar;
    l.ycnt = b.ycnt;
    l.y = y;
    l.y_dtype = y_dtype;
    return forward_impl(w, b.xq, b.xsf, b.gs_x, b.offsets, b.counts, b.row_token, T, k,
                        b.slot_out, NVMOE_F32, taps, b.fwd_ws, b.fwd_ws_bytes, stream, &l);
  }
  int st = moe_route_permute(topk_ids, T, k, E, b.offsets, b.counts, b.row_token, slot_of,
                             b.route_ws, b.route_ws_bytes, stream);
  if (st != NVMOE_OK) return st;
  // the row-major scales go to the slot-row buffer, which the L2 GEMM
  // overwrites only after they have been staged
  st = nvfp4_quantize_act(x, x_dtype, T, H, slot_of, k, rows, b.xq,
                          static_cast<uint8_t*>(b.slot_out), b.xsf, b.gs_x, b.quant_ws,
                          b.quant_ws_bytes, stream);
  if (st != NVMOE_OK) return st;
  // slot rows in fp16: half the bytes of the L2 epilogue's stores and of the
  // reduce's loads; the rounding (at most 2^-11 relative) stays well inside
  // the 2e-3 * row-amax tolerance of a GEMM output, and a value beyond the
  // fp16 range is reported (NVMOE_ERR_RANGE), never clamped
  st = forward_impl(w, b.xq, b.xsf, b.gs_x, b.offsets, b.counts, b.row_token, T, k, b.slot_out,
                    NVMOE_F16, taps, b.fwd_ws, b.fwd_ws_bytes, stream, nullptr);
  if (st != NVMOE_OK) return st;
  return moe_unpermute_reduce(b.slot_out, NVMOE_F16, slot_of, topk_w, T, k, H, y, y_dtype,
                              stream);
}

}  // extern "C"
