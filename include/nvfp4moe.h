/*
 * nvfp4moe.h — C ABI of the GB300 (sm_103a) NVFP4 MoE expert FFN library
 * (libnvfp4moe.so).
 *
 * The forward pass of one mixture-of-experts expert FFN with NVFP4 (E2M1
 * values, 16-element E4M3 block scales, fp32 global scales), as described by
 * the "NVFP4 MegaMoE Debug Log" (Architecture Notes, "NVFP4 MoE Pipeline"):
 *
 *   1. moe_route_permute      group the T*k (token, choice) slots by expert
 *   2. nvfp4_quantize_act     dynamic activation quantisation (stage_activation)
 *   3-6. moe_nvfp4_forward    L1 grouped GEMM over [gate; up], SiLU(gate)*up,
 *                             requantisation, L2 grouped GEMM, per-expert alpha
 *   7. moe_unpermute_reduce   top-k weighted reduce back to token order
 *
 * plus two offline weight helpers (nvfp4_quantize_weights,
 * moe_nvfp4_prepare_weights).
 *
 * Conventions (all entry points):
 *  - Every pointer argument is a DEVICE pointer owned by the caller, unless
 *    stated otherwise.  The library never allocates or frees device memory,
 *    never synchronises the host and keeps no state between calls except a
 *    per-device cache of kernel attributes (each kernel's shared-memory size,
 *    set on its first launch on a device) and the per-device address of the
 *    allocation-free routing array.  One process may drive several GPUs:
 *    every call works on the current device.
 *  - Work is enqueued on `stream`; a call returns once its kernels are
 *    enqueued.  Calls are stream-ordered and may be captured in a CUDA graph.
 *  - The return value is an nvmoe_status.  Host-side argument checks run
 *    before anything is enqueued; a nonzero status means nothing was enqueued
 *    (except NVMOE_ERR_CUDA, returned when a launch fails).  No C++ exception
 *    crosses the ABI.
 *  - Faults detected on the device (a wait that exceeded its time limit, an
 *    expert id out of range) do not trap: the kernel records a status code in
 *    a caller-visible status word and returns (see nvmoe_read_status).
 *  - Pointers must be 16-byte aligned.
 *
 * Slot layout.  Routing produces a grouped "row" layout: expert e owns rows
 * [expert_offsets[e], expert_offsets[e] + expert_counts[e]), and every
 * expert_offsets[e] is a multiple of NVMOE_TILE_ROWS (128); rows between an
 * expert's last slot and the next multiple of 128 are padding.  Within an
 * expert, slots are in ascending flat order t*k + j (stable counting sort).
 *
 * Block-scale staging ("MMA layout").  Block scales consumed by the tensor
 * cores are stored in 512-byte atoms covering 128 rows x 64 elements
 * (4 scale bytes per row).  For a matrix with R rows (R padded up to a
 * multiple of 128) and K elements per row (K padded up to a multiple of 256,
 * K_pad), the scale byte of (row r, 16-element group g) lives at
 *   ((r / 128) * (K_pad / 64) + g / 4) * 512
 *     + (r % 32) * 16 + ((r % 128) / 32) * 4 + (g % 4).
 * nvfp4_sf_mma_bytes() gives the buffer size.  Padding bytes are unspecified.
 */
#ifndef NVFP4MOE_H
#define NVFP4MOE_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

#define NVMOE_TILE_ROWS 128

typedef enum {
  NVMOE_OK = 0,
  NVMOE_ERR_INVALID_ARG = 1,        /* null pointer, negative size, bad enum */
  NVMOE_ERR_UNSUPPORTED_SHAPE = 2,  /* shape outside the supported set      */
  NVMOE_ERR_MISALIGNED = 3,         /* pointer not 16-byte aligned           */
  NVMOE_ERR_WORKSPACE_TOO_SMALL = 4,
  NVMOE_ERR_CUDA = 5,               /* a CUDA runtime/driver call failed     */
  NVMOE_ERR_TIMEOUT = 6,            /* device: a bounded wait ran out        */
  NVMOE_ERR_DEVICE_BAD_INDEX = 7,   /* device: expert id out of [0, E)       */
  NVMOE_ERR_RANGE = 8,              /* device: a value exceeded the range of
                                       its storage type (fp16 slot rows)     */
  NVMOE_ERR_DEVICE_BOUNDS = 9       /* device, NVMOE_DEBUG_BOUNDS build only:
                                       an index outside its buffer; the
                                       access was skipped                    */
} nvmoe_status;

/* Element types of activation / output buffers. */
typedef enum { NVMOE_BF16 = 0, NVMOE_F32 = 1, NVMOE_F16 = 2 } nvmoe_dtype;

/* Programmatic dependent launch on the multi-launch path (routing,
 * quantisation, both GEMMs, requantisation, reduce): each kernel is launched
 * with programmatic stream serialization, starts its prologue (barriers, TMEM,
 * tensor-map prefetch) while the kernel before it finishes, and waits
 * (griddepcontrol.wait) before touching any memory an earlier kernel used,
 * so results are unchanged.  enable 1 turns it on (process-wide); returns the
 * previous setting.  Default off: measured inside a CUDA graph on the large
 * prefill step it was 2 % slower (4.29 against 4.21 ms), whether the kernels
 * let their dependents launch at entry or after their work.  Host only. */
int nvmoe_set_pdl(int enable);

/* Human-readable name of a status code (static string, never NULL). */
const char* nvmoe_status_str(int status);

/* Name of the CUDA error (e.g. "cudaErrorInvalidValue") behind the last
   NVMOE_ERR_CUDA returned on the calling host thread, or "" if there was
   none.  Static string, never NULL; the record is per thread and is
   overwritten by the next failing call.  Host only, no device work. */
const char* nvmoe_last_cuda_error(void);

/* Library ABI version (major * 100 + minor): 200 (nvmoe_taps gained the
 * ready-flag members). */
int nvmoe_version(void);

/* Number of kernels this library has enqueued in this process so far (all
 * entry points; a replay of a captured CUDA graph enqueues nothing new).
 * For accounting and tests; no synchronisation. */
uint64_t nvmoe_kernel_launch_count(void);

/* Read (and optionally clear) the device status word that a workspace
 * carries at its start.  Synchronises `stream`.  `status_out` is a HOST
 * pointer.  Every workspace-taking call writes only nonzero codes there; a
 * fresh workspace must start zeroed (nvmoe_clear_status). */
int nvmoe_read_status(const void* workspace, cudaStream_t stream, int* status_out);
int nvmoe_clear_status(void* workspace, cudaStream_t stream);

/* Size in bytes of a staged (MMA layout) block-scale buffer for `rows` rows
 * of `cols` elements. */
size_t nvfp4_sf_mma_bytes(int64_t rows, int64_t cols);

/* ------------------------------------------------------- measurement --
 * nvmoe_fp4_mma_probe — dense NVFP4 tensor-core throughput probe.  No
 * counterpart in the source pages: the workloads' prefill figure is a
 * fraction of the dense FP4 tensor peak, and this measures that peak on the
 * GPU at hand instead of taking a datasheet number.  Each CTA issues `iters`
 * back-to-back tcgen05.mma kind::mxf4nvf4 block_scale.scale_vec::4X (K = 64
 * each, operands resident in shared memory, fp32 accumulator in TMEM) and
 * records the SM clock cycles from its first issue to the completion of the
 * last MMA.  FLOPs per CTA = iters * 2 * 128 * N * 64 (N = 256, or 128 with
 * bit 2); the caller times the launch with CUDA events.
 *   variant  bit 1: CTA pairs (cta_group::2, M = 256 over two SMs); bit 2:
 *            N = 128; bit 4: per MMA the 32x128b.warpx4 scale copies of a
 *            one-atom-per-k-block staging (1 for A, N/128 for B); bit 8: per
 *            four MMAs 128x256b scale copies (1 for A, N/64 for B).  Bits 4
 *            and 8 are exclusive.  Bit 16: the MMAs alternate between two
 *            accumulators; bit 32 (N = 128 only): between four; bit 64: no
 *            MMA adds to the previous one's result; bit 128: the scale
 *            copies alone (with bit 4 or 8), no MMA; with bit 8, bit 256:
 *            only the A copy, bit 512: the next four MMAs' copies issued
 *            after the second MMA of the current four.  Bit 1024 (with at
 *            most bit 2; iters a multiple of 4): one CTA whose scales reach
 *            TMEM by tcgen05.st from four warps, a stage of four MMAs at a
 *            time, while a fifth warp issues the MMAs.
 *   iters    1 .. 2^20;  grid  CTAs (even with bit 1), one per SM at most
 *   cycles   int64 [grid] out (device): cycles of each issuing CTA (-1 for
 *            the odd CTA of a pair)
 *   workspace  >= 256 bytes, zeroed; its first word is the status word
 * Operand values are fixed (E2M1 1.0, scales 1.0); nothing else is read. */
int nvmoe_fp4_mma_probe(int variant, int iters, int grid, long long* cycles,
                        void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* ---------------------------------------------------------------- step 1 --
 * moe_route_permute — per-expert histogram, prefix sum and stable slot
 * assignment of the top-k routing choice ("NVFP4 MegaMoE Debug Log":
 * pipeline trace "slots=", later log "L2 slot_token"; the scatter with routing
 * weights of the NVFP4 MoE Pipeline needs the inverse map slot_of).
 *
 *   topk_ids        int32 [T, k], row-major; each entry in [0, E).  An entry
 *                   outside that range sets NVMOE_ERR_DEVICE_BAD_INDEX in the
 *                   workspace status word and is dropped.
 *   expert_offsets  int32 [E + 1] out: first row of each expert (multiples of
 *                   128); expert_offsets[E] = number of rows in use.
 *   expert_counts   int32 [E] out: slots per expert.
 *   row_token       int32 [moe_route_rows_bound(T,k,E)] out: token of each
 *                   row, -1 on padding rows and on rows past expert_offsets[E].
 *   slot_of         int32 [T * k] out: row of (token t, choice j) at t*k + j.
 * Limits: 1 <= k <= 32, 1 <= E <= 256, T*k < 2^31.  T = 0 is valid (no-op
 * apart from zero offsets/counts and -1 row tokens).
 */
int64_t moe_route_rows_bound(int64_t T, int k, int E);
size_t moe_route_workspace_size(int64_t T, int k, int E);
int moe_route_permute(const int32_t* topk_ids, int64_t T, int k, int E,
                      int32_t* expert_offsets, int32_t* expert_counts,
                      int32_t* row_token, int32_t* slot_of,
                      void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* moe_route_permute_noalloc — the same routing permutation for callers that
 * cannot hand the library a device workspace.  No counterpart in the source
 * pages: it exists for callers that may not allocate device memory at all,
 * e.g. a serving engine that reserves every byte of HBM up front for its own
 * pools, or a plug-in host that owns all allocation, where a cudaMalloc
 * (which also synchronises the device) is not permitted.
 *
 * Same arguments and results as moe_route_permute, without the workspace.
 * The per-chunk histograms live in a fixed array inside the library
 * (NVMOE_NOALLOC_ROUTE_WORDS 32-bit words, 256 KiB, held on every GPU that
 * loads the library until the process exits); the call allocates nothing.
 *   - Limit: ceil(T*k / 4096) * E <= NVMOE_NOALLOC_ROUTE_WORDS (for example
 *     T*k up to 5.5 million slots with E = 48); larger inputs return
 *     NVMOE_ERR_UNSUPPORTED_SHAPE before anything is enqueued.
 *   - The first call on a device looks up the array's device address (once
 *     per device, with that device current); make that first call before
 *     any stream capture.
 *   - Every call shares the one array: calls whose kernels can overlap on the
 *     GPU (different streams without ordering, or several host threads) race
 *     and give wrong results.  Order them on one stream.
 *   - An expert id outside [0, E) is dropped (slot_of = -1) but no status
 *     word is written (there is no workspace to hold it).
 */
#define NVMOE_NOALLOC_ROUTE_WORDS (64 * 1024)
int moe_route_permute_noalloc(const int32_t* topk_ids, int64_t T, int k, int E,
                              int32_t* expert_offsets, int32_t* expert_counts,
                              int32_t* row_token, int32_t* slot_of, cudaStream_t stream);

/* ---------------------------------------------------------------- step 2 --
 * nvfp4_quantize_act — dynamic NVFP4 quantisation of activations
 * ("NVFP4 MegaMoE Debug Log", Hypotheses §6 steps 1-5 and §5 packing; commit
 * message "Three bugs fixed" on src).  In IEEE fp32, round-to-nearest-even:
 *   amax = max |x| over the whole input;  gs = amax / 2688  (1.0 if amax = 0)
 *   per 16-element block along a row:  b = max |x_i|,
 *     sf = E4M3_satfinite(b / (6 * gs)),  d = dec(sf) * gs,
 *     nibble_i = E2M1_satfinite(|x_i| / d) with bit 3 = sign bit of x_i
 *     (all nibbles 0 when d == 0)
 *   element 2j goes to the low nibble of byte j, 2j+1 to the high nibble.
 *
 *   x            [rows, cols] row-major, x_dtype = NVMOE_BF16 or NVMOE_F32.
 *   row_dst      optional int32 [rows * fanout]: input row r is written to
 *                output rows row_dst[r*fanout + j], j < fanout (use the
 *                slot_of of moe_route_permute with fanout = k to quantise
 *                straight into the grouped slot layout).  NULL: row r -> r.
 *   out_rows     number of output rows (>= rows when row_dst is NULL).
 *   q            uint8 [out_rows, cols/2] packed nibbles.
 *   sf_rowmajor  optional uint8 [out_rows, cols/16] scale bytes, row-major.
 *   sf_mma       optional staged scales, nvfp4_sf_mma_bytes(out_rows, cols).
 *   gs_out       float [1]: gs.
 * Output rows not written by any input row are left untouched, except that
 * when both scale layouts are given (cols % 256 == 0, sf_rowmajor 16-byte
 * aligned, rows * cols > 65536) the staged scales are written
 * by a second pass over sf_rowmajor: every 128-row tile of sf_mma is then
 * rewritten whole, an unwritten row's staged bytes being whatever its
 * sf_rowmajor row holds (zero past out_rows).  The bytes of written rows are
 * the same either way.
 * Limits: cols % 64 == 0, 1 <= fanout <= 32.  rows = 0 writes gs = 1.
 */
size_t nvfp4_quantize_workspace_size(int64_t rows, int64_t cols);
int nvfp4_quantize_act(const void* x, int x_dtype, int64_t rows, int64_t cols,
                       const int32_t* row_dst, int fanout, int64_t out_rows,
                       uint8_t* q, uint8_t* sf_rowmajor, uint8_t* sf_mma,
                       float* gs_out, void* workspace, size_t workspace_bytes,
                       cudaStream_t stream);

/* ------------------------------------------------------ offline weights --
 * nvfp4_quantize_weights — NVFP4 quantisation of fp32 expert weights into
 * the checkpoint layout ("NVFP4 MegaMoE Debug Log", Hypotheses §6 steps 1-5
 * and §2 shapes): per expert e, gs[e] = amax(W_e) / 2688; 16-element blocks
 * run along K for each output column n; same arithmetic as step 2.
 *   w    float [E, K, N] row-major (math layout, K = reduction dim)
 *   q    uint8 [E, K/2, N]: byte (j, n) = element (2j, n) low, (2j+1, n) high
 *   sf   uint8 [E, K/16, N]
 *   gs   float [E]
 * Limits: K % 64 == 0, N >= 1.
 */
size_t nvfp4_quantize_weights_workspace_size(int E, int K, int N);
int nvfp4_quantize_weights(const float* w, int E, int K, int N, uint8_t* q,
                           uint8_t* sf, float* gs, void* workspace,
                           size_t workspace_bytes, cudaStream_t stream);

/* moe_nvfp4_prepare_weights — checkpoint layout -> tensor-core layout (the
 * B-operand byte transpose of "NVFP4 MegaMoE Debug Log", Hypotheses §8 and the
 * later log's "B ColumnMajor" point; scale staging replaces the SF remap of
 * the commit messages on src).  Nibble pairs stay along K.
 *   q_ckpt  uint8 [E, K/2, N],  sf_ckpt uint8 [E, K/16, N]
 *   q_out   K-major B-operand tiles of the [E*N, K] matrix: with
 *           KT = ceil(K/256), row n (= e*N + column) and K-stage kt, the
 *           contiguous 16 KB tile ((n/128)*KT + kt) holds 128 rows of 128
 *           bytes; byte j of row n%128 packs elements 256*kt + 2j (low
 *           nibble) and 256*kt + 2j + 1 (high); bytes past K/2 are zero.
 *           Size moe_nvfp4_prepared_bytes(E, K, N) = E*N*KT*128.
 *   sf_out  staged scales of the [E*N, K] matrix: nvfp4_sf_mma_bytes(E*N, K)
 * Limits: K % 64 == 0, N % 128 == 0.
 */
size_t moe_nvfp4_prepared_bytes(int E, int K, int N);
int moe_nvfp4_prepare_weights(const uint8_t* q_ckpt, const uint8_t* sf_ckpt,
                              int E, int K, int N, uint8_t* q_out,
                              uint8_t* sf_out, cudaStream_t stream);

/* ------------------------------------------------------------ steps 3-6 --
 * Prepared expert weights (all device pointers):
 *   w1     B tiles of the [E*2I, H] matrix (moe_nvfp4_prepare_weights):
 *          L1 [gate; up] rows: gate = rows [0, I), up = rows [I, 2I) of
 *          each expert (plain concatenation, commit message on the removed
 *          2-CTA interleave)
 *   w1_sf  staged, nvfp4_sf_mma_bytes(E*2I, H);  gs_w1 float [E]
 *   w2     B tiles of the [E*H, I] matrix;  w2_sf staged,
 *          nvfp4_sf_mma_bytes(E*H, I);
 *   gs_w2  float [E]
 *   gs_w1_up  float [E] or NULL.  Checkpoints that quantise gate_proj and
 *          up_proj separately carry one global scale per half ("NVFP4
 *          MegaMoE Debug Log", code-review point 5, gate/up correction:
 *          equivalent to a per-column alpha).  When given, the gate columns
 *          use alpha = gs_x * gs_w1[e] and the up columns alpha = gs_x *
 *          gs_w1_up[e]; when NULL both halves use gs_w1[e].
 *   gs_mid float [E] or NULL.  A static global scale per expert for the
 *          requantisation of h (like a checkpoint's calibrated w2 input
 *          scale), in place of the pages' dynamic one (amax of h over all
 *          slots / 2688, "NVFP4 MegaMoE Debug Log", NVFP4 MoE Pipeline).
 *          With it no step waits for the whole L1 output: each CTA
 *          requantises the h tiles it has just produced, and L2 uses
 *          alpha = gs_mid[e] * gs_w2[e].  taps->gs_h is not written.
 */
typedef struct {
  int E, H, I;
  const uint8_t* w1;
  const uint8_t* w1_sf;
  const float* gs_w1;
  const uint8_t* w2;
  const uint8_t* w2_sf;
  const float* gs_w2;
  const float* gs_w1_up;
  const float* gs_mid;
} nvmoe_weights;

/* Optional outputs of intermediate results (any member may be NULL).
 *   l1_out   float [rows, 2I]: alpha-scaled L1 output, [gate | up]
 *   h        float [rows, I]:  SiLU(gate) * up (fp32)
 *   hq       uint8 [rows, I/2]; hsf_mma staged nvfp4_sf_mma_bytes(rows, I)
 *   gs_h     float [1]
 *   stage_events  caller-created CUDA events recorded on `stream`: [0]
 *            before the L1 GEMM, [1] after it, [2] after the requantisation,
 *            [3] after the L2 GEMM (all four or none; on the fused path
 *            [1..3] are all recorded after the single kernel).
 *   path     NVMOE_PATH_AUTO (0, default), NVMOE_PATH_SEPARATE (three
 *            launches: L1, requantisation, L2), NVMOE_PATH_FUSED (one
 *            cooperative kernel with two grid barriers) or
 *            NVMOE_PATH_SEPARATE_SINGLE (three launches, every GEMM on
 *            one-CTA tiles).  AUTO takes the fused kernel when both GEMMs
 *            have fewer than 4 tiles per SM.  On the three-launch path a
 *            GEMM with at least 4 tiles per SM whatever the routing runs on
 *            clusters of two CTAs (one tcgen05 MMA over both SMs, M = 256),
 *            unless SEPARATE_SINGLE.  Every path computes identical
 *            results.
 * rows = moe_route_rows_bound(T, k, E); padding rows are unspecified.
 * When h / hq / hsf_mma / gs_h are given they replace the workspace buffers
 * of the same name (no extra traffic); l1_out costs one extra store. */
#define NVMOE_PATH_AUTO 0
#define NVMOE_PATH_SEPARATE 1
#define NVMOE_PATH_FUSED 2
#define NVMOE_PATH_LAYER 3     /* moe_nvfp4_layer_forward only */
#define NVMOE_PATH_SEPARATE_SINGLE 4
typedef struct {
  float* l1_out;
  float* h;
  uint8_t* hq;
  uint8_t* hsf_mma;
  float* gs_h;
  cudaEvent_t stage_events[4];
  int path;
  int32_t* slot_of;       /* moe_nvfp4_layer_forward: int32 [T*k] row of each slot */
  /* moe_nvfp4_forward only (moe_nvfp4_layer_forward rejects it with
   * NVMOE_ERR_INVALID_ARG): the activation rows xq / xsf_mma are produced by
   * another stream or device and are ready once *ready_flag >= ready_value
   * (an int32 device word; gs_x and the routing tables must be ready at
   * launch).  The L1 kernel waits for the flag before its first load, at
   * most ready_wait_us microseconds (<= 0: 2 s); a wait that runs out
   * records NVMOE_ERR_TIMEOUT in the workspace status word and the call's
   * kernels return without producing results.  The workspace is left ready
   * for the next call.  NULL = ready at launch. */
  const int32_t* ready_flag;
  int ready_value;
  int ready_wait_us;
} nvmoe_taps;

/* moe_nvfp4_forward — the expert FFN on grouped slots ("NVFP4 MegaMoE Debug
 * Log", NVFP4 MoE Pipeline; Hypotheses §3 for alpha):
 *   l1[r, :]  = (gs_x * gs_w1[e]) * sum_k dec(xq) dec(xsf) dec(w1) dec(w1_sf)
 *               (up columns: gs_w1_up[e] in place of gs_w1[e] when given)
 *   h[r, c]   = silu(l1[r, c]) * l1[r, I + c]          (fp32)
 *   hq, hsf, gs_h = step-2 quantisation of h over all valid rows
 *   out[r, :] = (gs_h * gs_w2[e]) * sum_k dec(hq) dec(hsf) dec(w2) dec(w2_sf)
 * Alpha is applied to the fp32 accumulator, never folded into block scales.
 *   xq        uint8 [rows, H/2] activations in the grouped slot layout
 *   xsf_mma   staged scales of xq: nvfp4_sf_mma_bytes(rows, H)
 *   gs_x      float [1]
 *   expert_offsets, expert_counts, row_token: from moe_route_permute
 *   slot_out  [rows, H] of slot_out_dtype: NVMOE_F32, NVMOE_F16 or NVMOE_BF16
 *             (the fp32 alpha-scaled result rounded to nearest even: half the
 *             bytes written here and read by the reduce; fp16 is within
 *             2^-11 relative, bf16 within 2^-8).  With fp16 a value of
 *             magnitude above 65504 records NVMOE_ERR_RANGE in the status
 *             word (the stored value is then inf).
 *             (padding rows unspecified)
 * rows = moe_route_rows_bound(T, k, E).
 * Workspace: moe_nvfp4_workspace_size bytes, zero-filled before its first
 * use; the call leaves it ready for the next call (split-tile counters are
 * reset by the kernel that uses them).  One workspace per stream: calls that
 * overlap on the device must not share one.
 * Work split: with fewer than 4 tiles per SM (decode) the tiles x K-stages
 * sequence is divided evenly between the SMs; a tile shared by several SMs
 * is summed in ascending K order by the last SM to finish its piece, so the
 * result does not depend on timing.
 * Limits: H % 256 == 0, I % 128 == 0, E <= 256.
 */
size_t moe_nvfp4_workspace_size(int64_t T, int k, int E, int H, int I);
int moe_nvfp4_forward(const nvmoe_weights* weights, const uint8_t* xq,
                      const uint8_t* xsf_mma, const float* gs_x,
                      const int32_t* expert_offsets, const int32_t* expert_counts,
                      const int32_t* row_token, int64_t T, int k,
                      void* slot_out, int slot_out_dtype, const nvmoe_taps* taps,
                      void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* moe_nvfp4_forward_phase — moe_nvfp4_forward in two calls, for callers whose
 * h spans several processes (expert parallelism): the requantisation's global
 * scale is gs_h = amax(h)/2688 over ALL of h ("NVFP4 MoE Pipeline" step 4), so
 * the amax of every process's h must be reduced before any h is requantised.
 *   phase 1  L1 GEMM + SiLU*up: h into the workspace, and *amax_h (device
 *            float) = max |h| over this call's valid rows (0 for T == 0).
 *   phase 2  requantise h with gs_h = *amax_h/2688 (the caller's reduced
 *            amax: 0 gives gs 1, as for an all-zero tensor), then the L2 GEMM
 *            into slot_out.
 * The arguments are those of moe_nvfp4_forward, the same in both calls, with
 * the same workspace (it carries h between them).  Always the three-launch
 * path (the fused kernels need the amax inside).  With weights->gs_mid (a
 * static intermediate scale) phase 1 requantises in the L1 epilogue and phase
 * 2 runs L2 alone; *amax_h is then unused by phase 2.  With one process,
 * phase 1 then phase 2 on the same *amax_h equals moe_nvfp4_forward bit for
 * bit.  Errors as moe_nvfp4_forward; NVMOE_ERR_INVALID_ARG for phase not 1
 * or 2 or amax_h NULL. */
int moe_nvfp4_forward_phase(const nvmoe_weights* weights, const uint8_t* xq,
                            const uint8_t* xsf_mma, const float* gs_x,
                            const int32_t* expert_offsets, const int32_t* expert_counts,
                            const int32_t* row_token, int64_t T, int k, void* slot_out,
                            int slot_out_dtype, int phase, float* amax_h,
                            const nvmoe_taps* taps, void* workspace, size_t workspace_bytes,
                            cudaStream_t stream);

/* ----------------------------------------------------- expert parallelism --
 * The pages' 48 experts are one tensor-parallel rank's share of a larger MoE
 * ("NVFP4 MoE Debug Log (early)", Symptoms: all 8 TP ranks hold the same
 * weight shapes; Hypotheses section 7, the per-rank table).  Split the E
 * experts over G processes instead (E % G == 0; process d owns experts
 * [d*E/G, (d+1)*E/G)), and a token's slot goes to the owner of its expert:
 *
 *   every process: amax of its tokens (nvfp4_amax) -> MAX over processes ->
 *     quantise its tokens once with that amax (nvfp4_quantize_act_amax,
 *     row_dst NULL: token rows, row-major scales) -> moe_ep_dispatch ->
 *     all-to-all of the packed rows and their local expert ids (counts from
 *     send_counts) ->
 *   owner: moe_route_permute of the received local expert ids (T = rows
 *     received, k = 1) -> moe_ep_scatter -> moe_nvfp4_forward_phase 1 ->
 *     MAX of amax_h over processes -> phase 2 -> moe_ep_gather ->
 *     all-to-all back (the reverse counts) ->
 *   every process: moe_unpermute_reduce of the returned rows with
 *     slot_of = send_pos.
 *
 * The exchanges are the caller's collectives (NCCL / torch.distributed).
 * With the tokens split over the processes in order, every expert sees its
 * slots in the one-process order and the same global scales, so the result
 * equals the one-process forward of the whole batch bit for bit.  The
 * library never synchronises with the host: send_counts must be copied out
 * by the caller to size the exchange. */

/* Max |x| of a [rows, cols] bf16/fp32 matrix into *amax_out (device float;
 * 0 for rows == 0).  Workspace: nvfp4_quantize_workspace_size(rows, cols).
 * Errors as nvfp4_quantize_act. */
int nvfp4_amax(const void* x, int x_dtype, int64_t rows, int64_t cols, float* amax_out,
               void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* nvfp4_quantize_act with the amax given (*amax_in, device float) instead of
 * computed: gs = amax/2688 written to *gs_out; no workspace.  The same
 * arguments and results as nvfp4_quantize_act otherwise (its results equal
 * nvfp4_quantize_act's when *amax_in is the matrix's own amax).  Having no
 * status word, the NVMOE_DEBUG_BOUNDS build skips a row_dst >= out_rows
 * without a record. */
int nvfp4_quantize_act_amax(const void* x, int x_dtype, int64_t rows, int64_t cols,
                            const int32_t* row_dst, int fanout, int64_t out_rows,
                            const float* amax_in, uint8_t* q, uint8_t* sf_rowmajor,
                            uint8_t* sf_mma, float* gs_out, cudaStream_t stream);

/* Dispatch of T tokens' k slots to G processes.
 *   topk_ids  int32 [T, k] global expert ids (an id outside [0, E) is
 *             recorded as NVMOE_ERR_DEVICE_BAD_INDEX in the workspace status
 *             and its slot sent nowhere: send_pos -1)
 *   q_tok     uint8 [T, H/2] E2M1 token rows; sf_tok uint8 [T, H/16]
 *             row-major E4M3 scales (nvfp4_quantize_act_amax, row_dst NULL)
 *   send_counts  int32 [G] out: slots for each process
 *   send_pos  int32 [T*k] out: row of slot t*k+j in send_rows; the rows of
 *             process d are [sum of counts before d, +counts[d]), in
 *             ascending t*k+j
 *   send_rows uint8 [T*k, H/2 + H/16] out: nibbles then scales per row
 *   send_expert int32 [T*k] out: the row's expert index on its process
 *   workspace moe_ep_dispatch_workspace_size(T, k, G), status word first.
 * Limits: E % G == 0, G <= E <= 256, H % 256 == 0.  16-byte alignment of
 * q_tok, sf_tok, send_rows, workspace. */
size_t moe_ep_dispatch_workspace_size(int64_t T, int k, int G);
int moe_ep_dispatch(const int32_t* topk_ids, int64_t T, int k, int E, int G,
                    const uint8_t* q_tok, const uint8_t* sf_tok, int H, int32_t* send_counts,
                    int32_t* send_pos, uint8_t* send_rows, int32_t* send_expert,
                    void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* Received rows (moe_ep_dispatch's row format, n of them) into the slot
 * layout of moe_nvfp4_forward: row i's nibbles to xq[slot_of[i]] (xq has
 * out_rows rows) and its scales to their staged offsets in xsf_mma
 * (nvfp4_sf_mma_bytes(out_rows, H)); slot_of from moe_route_permute of the
 * received expert ids (k = 1); rows with slot_of < 0 are skipped.  status:
 * nullable device int where the NVMOE_DEBUG_BOUNDS build records
 * NVMOE_ERR_DEVICE_BOUNDS for a slot_of >= out_rows (that row is skipped).
 * 16-byte alignment of recv_rows, xq, xsf_mma. */
int moe_ep_scatter(const uint8_t* recv_rows, int64_t n, int H, const int32_t* slot_of,
                   int64_t out_rows, uint8_t* xq, uint8_t* xsf_mma, int* status,
                   cudaStream_t stream);

/* out_rows[i] = slot_out[slot_of[i]] for i < n (slot_out: slot_rows rows of
 * H elements of slot_out_dtype; a row with slot_of < 0 is zero): the owner's
 * slot outputs in received order, for the return exchange.  status as for
 * moe_ep_scatter (a slot_of >= slot_rows gives a zero row in that build).
 * 16-byte alignment. */
int moe_ep_gather(const void* slot_out, int slot_out_dtype, int H, int64_t slot_rows,
                  const int32_t* slot_of, int64_t n, void* out_rows, int* status,
                  cudaStream_t stream);

/* -------------------------------------------------------- router front end --
 * moe_router_topk — the step before the routing permutation.  The pages keep
 * the router ("gate") weight in BF16 ("NVFP4 MegaMoE Debug Log", Checkpoint
 * Layers) and route each token to its top-k experts with softmax weights:
 *   logits[t, e] = sum_h x[t, h] * w_router[e, h]   (bf16 inputs, fp32 sums;
 *                  the h order is fixed, so results do not depend on timing)
 *   topk_ids[t, j]  the expert with the j-th largest logit (ties: the lower
 *                   expert id first)
 *   topk_w[t, j]    softmax_mode NVMOE_ROUTER_SELECTED: softmax over the k
 *                   selected logits; NVMOE_ROUTER_ALL: the full softmax's
 *                   probability of the selected expert
 *   x bf16 [T, H];  w_router bf16 [E, H];  topk_ids int32 [T, k];
 *   topk_w float [T, k]
 * The logits run on the tensor cores (tcgen05.mma kind::f16, fp32
 * accumulation in TMEM): a CTA takes 128 tokens and one range of H, and the
 * ranges' partial logits are added in range order (so results do not depend
 * on timing); small batches split H over several CTAs.
 * Workspace: moe_router_workspace_size(T, H, E) bytes; its first word is a
 * status word (nvmoe_read_status), zero before the first use.
 * Limits: H % 128 == 0, 1 <= E <= 256, 1 <= k <= min(E, 32); x and w_router
 * 16-byte aligned.
 */
#define NVMOE_ROUTER_SELECTED 0
#define NVMOE_ROUTER_ALL 1
size_t moe_router_workspace_size(int64_t T, int H, int E);
int moe_router_topk(const void* x, const void* w_router, int64_t T, int H, int E, int k,
                    int softmax_mode, int32_t* topk_ids, float* topk_w, void* workspace,
                    size_t workspace_bytes, cudaStream_t stream);

/* ---------------------------------------------------------------- step 7 --
 * moe_unpermute_reduce — "scatter with routing weights" of the NVFP4 MoE
 * Pipeline, written as a deterministic gather:
 *   y[t, :] = sum_{j = 0..k-1} topk_w[t, j] * slot_out[slot_of[t*k + j], :]
 * accumulated in fp32 in ascending j, stored once as y_dtype (bf16 rounds to
 * nearest even).
 *   slot_out [rows, H] of slot_out_dtype (NVMOE_F32, NVMOE_F16 or
 *            NVMOE_BF16; both 16-bit types widen exactly);  slot_of int32
 *            [T*k];  topk_w float [T, k]
 *   y        [T, H] of y_dtype (NVMOE_BF16 or NVMOE_F32)
 * Limits: H % 8 == 0, 1 <= k <= 32.
 */
int moe_unpermute_reduce(const void* slot_out, int slot_out_dtype,
                         const int32_t* slot_of, const float* topk_w, int64_t T, int k,
                         int64_t H, void* y, int y_dtype, cudaStream_t stream);

/* ----------------------------------------------------------- steps 1-7 --
 * moe_nvfp4_layer_forward — the whole layer in one call: the four steps
 * above on buffers carved from one workspace, with the same results.
 *   x        [T, H] of x_dtype (NVMOE_BF16 or NVMOE_F32)
 *   topk_ids int32 [T, k];  topk_w float [T, k]
 *   y        [T, H] of y_dtype
 * Small batches (bf16 x, T*k <= 128, T*H <= 65536, fewer than 4 tiles per SM
 * in both GEMMs) run as ONE cooperative kernel: every CTA builds the routing
 * tables and computes gs_x itself, so weight streaming starts at once; the
 * activation blocks are quantised once, 1/G of them per CTA, and each CTA's
 * activation loads wait for the count of finished shares; a single grid
 * barrier separates L1 from the requantisation (the intermediate global
 * scale needs every h), which is spread over the grid the same way; the
 * top-k reduce of a (token, 256-column tile) is done by the CTA that writes
 * its last slot row.  taps->path = NVMOE_PATH_LAYER forces that kernel
 * (NVMOE_ERR_UNSUPPORTED_SHAPE when the batch is too large); SEPARATE / FUSED
 * select the paths of moe_nvfp4_forward after separate routing and
 * quantisation launches.  taps->slot_of, when given, receives the slot row
 * of every (token, choice).
 * Above the single-kernel limits the slot rows between the L2 GEMM and the
 * reduce are held in fp16 (see moe_nvfp4_forward: NVMOE_ERR_RANGE reports a
 * value beyond its range).
 * Workspace: moe_nvfp4_layer_workspace_size bytes, zero-filled before first
 * use; its status word (nvmoe_read_status) is the forward's.  The kernel
 * leaves its barrier words and reduce counters at zero for the next call;
 * after a call that recorded a non-zero status (an expert id outside
 * [0, E), a timed-out wait) they may be left mid-count: zero the workspace
 * again before reusing it.
 */
size_t moe_nvfp4_layer_workspace_size(int64_t T, int k, int E, int H, int I);
int moe_nvfp4_layer_forward(const nvmoe_weights* weights, const void* x, int x_dtype,
                            const int32_t* topk_ids, const float* topk_w, int64_t T, int k,
                            void* y, int y_dtype, const nvmoe_taps* taps, void* workspace,
                            size_t workspace_bytes, cudaStream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* NVFP4MOE_H */
