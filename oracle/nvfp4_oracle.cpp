// CPU oracle of the NVFP4 MoE expert FFN, in plain C++17 — TEST
// INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the CPU
// baseline of the benchmark load it; the library never does, and the two
// share no code, header, table or helper.
//
// What it computes, and where the pages say so:
//   * E2M1 nibbles: sign-magnitude, bit 3 = sign, bits 2:0 index the
//     magnitudes {0, 0.5, 1, 1.5, 2, 3, 4, 6}; a value snaps to the nearest
//     magnitude (commit message "Three bugs fixed" on src).
//   * Packing: element 2j in the low nibble, 2j+1 in the high nibble
//     ("NVFP4 MegaMoE Debug Log", Hypotheses §5); weight bytes pair elements
//     along K (Hypotheses §8 and the weight-unpack passage).
//   * E4M3 scale bytes are read by their bit pattern (commit message on the
//     FP8 view-vs-convert bug), OCP E4M3: bias 7, no infinities, S.1111.111 NaN.
//   * Quantiser (Hypotheses §6 steps 1-5), IEEE fp32 in this order:
//       gs = amax / (6*448);  per 16-block b = max|v|;  sf = E4M3(b / (6 gs));
//       d = dec(sf) gs;  nibble = E2M1(v / d)
//   * L1 / L2 GEMMs with per-expert alpha = activation gs * weight gs applied
//     to the fp64 accumulator, never folded into the block scales (Hypotheses
//     §3; NVFP4 MoE Pipeline); SiLU(gate)*up on the plain [gate; up] halves
//     (commit message on the removed 2-CTA interleave); requantisation of h
//     with its own dynamic global scale; the top-k weighted scatter back to
//     token order (NVFP4 MoE Pipeline).
// Readings where the pages are silent (the same as the library's, stated
// independently here): ties round to the even code; both encoders saturate
// (6, 448); the nibble divisor uses the stored scale; a block whose scale
// decodes to 0 gets nibbles 0x0; an all-zero tensor gets gs = 1; a negative
// value that rounds to magnitude 0 keeps its sign bit.
//
// Accumulation is fp64 (sums in ascending K); h is rounded to fp32 before it
// is requantised; y is rounded once to bf16 by the caller's choice.
// Build: g++ -std=c++17 -O3 -fopenmp -ffp-contract=off -shared -fPIC (no
// fast-math: every fp32 step must be the IEEE operation it names).
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <vector>

#include <omp.h>

namespace {

// ------------------------------------------------------------ E2M1 ----
const double kE2M1Mag[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};

double e2m1_value(unsigned nib) {
  const double m = kE2M1Mag[nib & 7u];
  return (nib & 8u) ? -m : m;
}

// Nearest magnitude by walking up the grid while |v| lies above the midpoint
// to the next magnitude; on a midpoint the even code wins; saturates at 6.
// (An fp32 argument widens to double exactly; the midpoints are exact.)
unsigned e2m1_code(double v) {
  double a = std::fabs(v);
  if (!(a <= 6.0)) a = 6.0;
  unsigned c = 0;
  while (c < 7) {
    const double mid = 0.5 * (kE2M1Mag[c] + kE2M1Mag[c + 1]);
    if (a > mid || (a == mid && ((c + 1) % 2 == 0)))
      ++c;
    else
      break;
  }
  return c | (std::signbit(v) ? 8u : 0u);
}

// ------------------------------------------------------------ E4M3 ----
double e4m3_value(unsigned byte) {
  const unsigned s = (byte >> 7) & 1u, e = (byte >> 3) & 15u, m = byte & 7u;
  double mag;
  if (e == 15u && m == 7u)
    mag = std::nan("");
  else if (e == 0u)
    mag = std::ldexp(static_cast<double>(m), -9);           // (m/8) 2^-6
  else
    mag = std::ldexp(8.0 + m, static_cast<int>(e) - 10);   // (1 + m/8) 2^(e-7)
  return s ? -mag : mag;
}

// The 127 non-negative finite values, ascending with the byte 0x00..0x7E.
struct E4M3Table {
  double v[127];
  E4M3Table() {
    for (unsigned b = 0; b < 127; ++b) v[b] = e4m3_value(b);
  }
};
const E4M3Table kE4M3;

// Nearest non-negative E4M3 byte (ties to the even byte), saturating at 448.
unsigned e4m3_code_nonneg(double a) {
  if (a >= kE4M3.v[126]) return 126u;
  // largest byte whose value is <= a
  unsigned lo = 0, hi = 126;
  while (hi - lo > 1) {
    const unsigned mid = (lo + hi) / 2;
    if (kE4M3.v[mid] <= a) lo = mid; else hi = mid;
  }
  if (kE4M3.v[lo] == a) return lo;
  const double midpoint = 0.5 * (kE4M3.v[lo] + kE4M3.v[lo + 1]);
  if (a > midpoint) return lo + 1;
  if (a < midpoint) return lo;
  return (lo % 2 == 0) ? lo : lo + 1;
}

// ------------------------------------------------------------ scales ----
float global_scale_of(float amax) {
  if (amax == 0.0f) return 1.0f;
  return amax / 2688.0f;          // 6 * 448
}

// One 16-element block: scale byte, and the 16 nibbles.
unsigned quantise_block(const float* v, float gs, unsigned* nib) {
  float b = 0.0f;
  for (int i = 0; i < 16; ++i) b = std::max(b, std::fabs(v[i]));
  const float denom = 6.0f * gs;
  const float t = b / denom;
  const unsigned sf = e4m3_code_nonneg(static_cast<double>(t));
  const float d = static_cast<float>(e4m3_value(sf)) * gs;
  for (int i = 0; i < 16; ++i) {
    const float ratio = v[i] / d;             // one fp32 division
    nib[i] = d == 0.0f ? 0u : e2m1_code(static_cast<double>(ratio));
  }
  return sf;
}

float tensor_amax(const float* v, int64_t n) {
  float m = 0.0f;
#pragma omp parallel for reduction(max : m)
  for (int64_t i = 0; i < n; ++i) m = std::max(m, std::fabs(v[i]));
  return m;
}

}  // namespace

extern "C" {

// ---------------------------------------------------------- codecs ----
double nvo_e2m1_decode(int nib) { return e2m1_value(static_cast<unsigned>(nib)); }
int nvo_e2m1_encode(double v) { return static_cast<int>(e2m1_code(v)); }
double nvo_e4m3_decode(int byte) { return e4m3_value(static_cast<unsigned>(byte)); }
// v must be finite and >= 0
int nvo_e4m3_encode_nonneg(double v) { return static_cast<int>(e4m3_code_nonneg(v)); }
float nvo_global_scale(float amax) { return global_scale_of(amax); }

void nvo_e2m1_decode_n(const uint8_t* nib, int64_t n, double* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = e2m1_value(nib[i]);
}
void nvo_e2m1_encode_n(const double* v, int64_t n, uint8_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = static_cast<uint8_t>(e2m1_code(v[i]));
}
void nvo_e4m3_decode_n(const uint8_t* b, int64_t n, double* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = e4m3_value(b[i]);
}
void nvo_e4m3_encode_nonneg_n(const double* v, int64_t n, uint8_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = static_cast<uint8_t>(e4m3_code_nonneg(v[i]));
}

// --------------------------------------------------------- packing ----
// [R, K] nibbles -> [R, K/2] bytes: element 2j low, 2j+1 high.
void nvo_pack_nibbles(const uint8_t* nib, int64_t R, int64_t K, uint8_t* out) {
  for (int64_t r = 0; r < R; ++r)
    for (int64_t j = 0; j < K / 2; ++j)
      out[r * (K / 2) + j] = static_cast<uint8_t>((nib[r * K + 2 * j] & 15u) |
                                                  ((nib[r * K + 2 * j + 1] & 15u) << 4));
}
void nvo_unpack_nibbles(const uint8_t* packed, int64_t R, int64_t K, uint8_t* nib) {
  for (int64_t r = 0; r < R; ++r)
    for (int64_t j = 0; j < K / 2; ++j) {
      const uint8_t b = packed[r * (K / 2) + j];
      nib[r * K + 2 * j] = b & 15u;
      nib[r * K + 2 * j + 1] = b >> 4;
    }
}
// checkpoint weight bytes (K/2, N) -> nibbles (K, N): pairs along K
void nvo_unpack_weight_k(const uint8_t* packed, int64_t K, int64_t N, uint8_t* nib) {
  for (int64_t j = 0; j < K / 2; ++j)
    for (int64_t n = 0; n < N; ++n) {
      const uint8_t b = packed[j * N + n];
      nib[(2 * j) * N + n] = b & 15u;
      nib[(2 * j + 1) * N + n] = b >> 4;
    }
}

// ------------------------------------------------------- quantiser ----
// Rows of [R, K] fp32 along K.  has_gs = 0: gs from the amax of the whole
// input; else gs_in.  q [R, K/2], sf [R, K/16]; *gs_out = gs.
void nvo_quantize_rows(const float* v, int64_t R, int64_t K, int has_gs, float gs_in,
                       uint8_t* q, uint8_t* sf, float* gs_out) {
  const float gs = has_gs ? gs_in : global_scale_of(tensor_amax(v, R * K));
  *gs_out = gs;
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < R; ++r) {
    unsigned nib[16];
    for (int64_t g = 0; g < K / 16; ++g) {
      const float* blk = v + r * K + g * 16;
      sf[r * (K / 16) + g] = static_cast<uint8_t>(quantise_block(blk, gs, nib));
      for (int j = 0; j < 8; ++j)
        q[r * (K / 2) + g * 8 + j] = static_cast<uint8_t>(nib[2 * j] | (nib[2 * j + 1] << 4));
    }
  }
}

// q [R, K/2] + sf [R, K/16] -> fp64 [R, K] without the global scale
void nvo_dequantize_rows(const uint8_t* q, const uint8_t* sf, int64_t R, int64_t K,
                         double* out) {
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < R; ++r)
    for (int64_t k = 0; k < K; ++k) {
      const uint8_t b = q[r * (K / 2) + k / 2];
      const unsigned nib = (k % 2 == 0) ? (b & 15u) : (b >> 4);
      out[r * K + k] = e2m1_value(nib) * e4m3_value(sf[r * (K / 16) + k / 16]);
    }
}

// One expert's weight (K, N) fp32: blocks of 16 along K for each column n,
// gs from the whole matrix.  q (K/2, N), sf (K/16, N).  The same block
// arithmetic as quantise_block, taken one 16-row band at a time so that the
// rows of w are read in order.
void nvo_quantize_weight(const float* w, int64_t K, int64_t N, uint8_t* q, uint8_t* sf,
                         float* gs_out) {
  const float gs = global_scale_of(tensor_amax(w, K * N));
  *gs_out = gs;
  const float denom = 6.0f * gs;
#pragma omp parallel
  {
    std::vector<float> bmax(static_cast<size_t>(N)), d(static_cast<size_t>(N));
#pragma omp for schedule(static)
    for (int64_t g = 0; g < K / 16; ++g) {
      const float* band = w + g * 16 * N;
      for (int64_t n = 0; n < N; ++n) bmax[n] = 0.0f;
      for (int i = 0; i < 16; ++i)
        for (int64_t n = 0; n < N; ++n) bmax[n] = std::max(bmax[n], std::fabs(band[i * N + n]));
      for (int64_t n = 0; n < N; ++n) {
        const float t = bmax[n] / denom;
        const unsigned code = e4m3_code_nonneg(static_cast<double>(t));
        sf[g * N + n] = static_cast<uint8_t>(code);
        d[n] = static_cast<float>(e4m3_value(code)) * gs;
      }
      for (int j = 0; j < 8; ++j)
        for (int64_t n = 0; n < N; ++n) {
          unsigned nib[2];
          for (int h = 0; h < 2; ++h) {
            const float ratio = band[(2 * j + h) * N + n] / d[n];
            nib[h] = d[n] == 0.0f ? 0u : e2m1_code(static_cast<double>(ratio));
          }
          q[(g * 8 + j) * N + n] = static_cast<uint8_t>(nib[0] | (nib[1] << 4));
        }
    }
  }
}

void nvo_dequantize_weight(const uint8_t* q, const uint8_t* sf, int64_t K, int64_t N,
                           double* out) {
#pragma omp parallel for schedule(static)
  for (int64_t k = 0; k < K; ++k)
    for (int64_t n = 0; n < N; ++n) {
      const uint8_t b = q[(k / 2) * N + n];
      const unsigned nib = (k % 2 == 0) ? (b & 15u) : (b >> 4);
      out[k * N + n] = e2m1_value(nib) * e4m3_value(sf[(k / 16) * N + n]);
    }
}

// ------------------------------------------------------------ GEMM ----
// acc[m, n] = sum over k (ascending) of A[m, k] W[k, n] in fp64, with A and
// W already dequantised (every product of E2M1 and E4M3 values is exact).
// The loops run over blocks of rows and columns so that a slice of W is
// reused from cache; every output still adds its K terms in ascending order.
void nvo_matmul_f64(const double* A, const double* W, int64_t M, int64_t K, int64_t N,
                    double* C) {
  const int64_t MB = 16, NB = 256;
  const int64_t mblocks = (M + MB - 1) / MB, nblocks = (N + NB - 1) / NB;
#pragma omp parallel for schedule(dynamic)
  for (int64_t blk = 0; blk < mblocks * nblocks; ++blk) {
    const int64_t m0 = (blk / nblocks) * MB, n0 = (blk % nblocks) * NB;
    const int64_t m1 = std::min(M, m0 + MB), n1 = std::min(N, n0 + NB);
    for (int64_t m = m0; m < m1; ++m)
      for (int64_t n = n0; n < n1; ++n) C[m * N + n] = 0.0;
    for (int64_t k = 0; k < K; ++k)
      for (int64_t m = m0; m < m1; ++m) {
        const double a = A[m * K + k];
        if (a == 0.0) continue;          // adds +0 * w: no change to any sum
        const double* wr = W + k * N;
        double* cr = C + m * N;
        for (int64_t n = n0; n < n1; ++n) cr[n] += a * wr[n];
      }
  }
}

// acc[m, n] = sum_k dec(a) dec(sfa) dec(w) dec(sfw), global scales not applied.
// a_q [M, K/2], a_sf [M, K/16]; w_q (K/2, N), w_sf (K/16, N).
void nvo_block_scaled_matmul(const uint8_t* a_q, const uint8_t* a_sf, int64_t M, int64_t K,
                             const uint8_t* w_q, const uint8_t* w_sf, int64_t N, double* acc) {
  std::vector<double> A(static_cast<size_t>(M * K)), W(static_cast<size_t>(K * N));
  nvo_dequantize_rows(a_q, a_sf, M, K, A.data());
  nvo_dequantize_weight(w_q, w_sf, K, N, W.data());
  nvo_matmul_f64(A.data(), W.data(), M, K, N, acc);
}

// -------------------------------------------------------- routing ----
// Counting sort of the T*k (token, choice) pairs by expert, stable in the
// flat index t*k + j.  Returns -1 (and writes nothing) on an id outside
// [0, E).  counts [E], offsets [E+1], slot_flat [S] (dense slot -> flat
// index), slot_of [S] (flat index -> dense slot).
int nvo_route(const int32_t* ids, int64_t T, int k, int E, int64_t* counts, int64_t* offsets,
              int64_t* slot_flat, int64_t* slot_of) {
  const int64_t S = T * k;
  for (int64_t i = 0; i < S; ++i)
    if (ids[i] < 0 || ids[i] >= E) return -1;
  for (int e = 0; e < E; ++e) counts[e] = 0;
  for (int64_t i = 0; i < S; ++i) ++counts[ids[i]];
  offsets[0] = 0;
  for (int e = 0; e < E; ++e) offsets[e + 1] = offsets[e] + counts[e];
  std::vector<int64_t> next(offsets, offsets + E);
  for (int64_t i = 0; i < S; ++i) {
    const int64_t s = next[ids[i]]++;
    slot_flat[s] = i;
    slot_of[i] = s;
  }
  return 0;
}

// Dense slots -> the grouped row layout whose expert segments start at
// multiples of tile_rows.  row_offsets [E+1]; row_of [S] (flat index -> row);
// row_token [rows] (-1 on padding).  Returns the number of rows.
int64_t nvo_padded_layout(const int64_t* counts, const int64_t* offsets, const int64_t* slot_flat,
                          const int64_t* slot_of, int64_t S, int E, int k, int tile_rows,
                          int64_t* row_offsets, int64_t* row_of, int64_t* row_token,
                          int64_t row_token_len) {
  row_offsets[0] = 0;
  for (int e = 0; e < E; ++e)
    row_offsets[e + 1] = row_offsets[e] + (counts[e] + tile_rows - 1) / tile_rows * tile_rows;
  const int64_t rows = row_offsets[E];
  if (row_token != nullptr)
    for (int64_t r = 0; r < std::min(rows, row_token_len); ++r) row_token[r] = -1;
  std::vector<int64_t> row_of_dense(static_cast<size_t>(S));
  for (int e = 0; e < E; ++e)
    for (int64_t s = offsets[e]; s < offsets[e + 1]; ++s) row_of_dense[s] = row_offsets[e] + (s - offsets[e]);
  for (int64_t i = 0; i < S; ++i) row_of[i] = row_of_dense[slot_of[i]];
  if (row_token != nullptr)
    for (int64_t s = 0; s < S; ++s)
      if (row_of_dense[s] < row_token_len) row_token[row_of_dense[s]] = slot_flat[s] / k;
  return rows;
}

// --------------------------------------------------- activation ----
double nvo_silu(double x) { return x / (1.0 + std::exp(-x)); }

// h = SiLU(gate) * up on [S, 2I] fp64, rounded once to fp32.
void nvo_swiglu(const double* l1, int64_t S, int64_t I, float* h) {
#pragma omp parallel for schedule(static)
  for (int64_t s = 0; s < S; ++s)
    for (int64_t c = 0; c < I; ++c)
      h[s * I + c] = static_cast<float>(nvo_silu(l1[s * 2 * I + c]) * l1[s * 2 * I + I + c]);
}

// ------------------------------------------------------------ reduce ----
// y[t] = sum over j ascending of w[t, j] * out2[slot_of[t*k + j]], fp64.
// (w as fp64: the pipeline's fp32 routing weights widen exactly)
void nvo_unpermute_reduce(const double* out2, int64_t H, const int64_t* slot_of, const double* w,
                          int64_t T, int k, double* y) {
#pragma omp parallel for schedule(static)
  for (int64_t t = 0; t < T; ++t) {
    for (int64_t c = 0; c < H; ++c) y[t * H + c] = 0.0;
    for (int j = 0; j < k; ++j) {
      const double wj = w[t * k + j];
      const double* row = out2 + slot_of[t * k + j] * H;
      for (int64_t c = 0; c < H; ++c) y[t * H + c] += wj * row[c];
    }
  }
}

// Nearest bf16 value of x (ties to even), rounded once from fp64.
double nvo_round_to_bf16(double x) {
  if (x == 0.0 || !std::isfinite(x)) return x;
  int e = 0;
  const double m = std::frexp(x, &e);             // x = m 2^e, 0.5 <= |m| < 1
  return std::ldexp(std::nearbyint(std::ldexp(m, 8)), e - 8);
}

// ----------------------------------------------------------- forward ----
// The whole forward pass (routing -> quantise x -> L1 with alpha -> SiLU*up
// -> requantise h -> L2 with alpha -> top-k reduce), dense slot order.
//   x [T, H] fp32 (bf16 values); ids int32 [T, k]; w fp32 [T, k]
//   w1_q (E, H/2, 2I), w1_sf (E, H/16, 2I), gs_w1 [E] (or [E, 2] gate/up
//   when gs1_split); w2_q (E, I/2, H), w2_sf (E, I/16, H), gs_w2 [E];
//   gs_mid [E] or null (static intermediate scale per expert in place of the
//   dynamic one: h rows of expert e quantised with gs_mid[e], L2 alpha
//   gs_mid[e] gs_w2[e]).
// Outputs (any may be null except y64): l1 [S, 2I] fp64 alpha-scaled, h [S, I]
// fp32, hq [S, I/2], hsf [S, I/16], gs_h [1], gs_x [1], out2 [S, H] fp64,
// y64 [T, H] fp64, slot_of [S].  Returns 0, or -1 on an expert id outside
// [0, E).
int nvo_forward(const float* x, int64_t T, int64_t H, const int32_t* ids, const float* w, int k,
                int E, int64_t I, const uint8_t* w1_q, const uint8_t* w1_sf, const float* gs_w1,
                int gs1_split, const uint8_t* w2_q, const uint8_t* w2_sf, const float* gs_w2,
                const float* gs_mid, double* l1_out, float* h_out, uint8_t* hq_out,
                uint8_t* hsf_out, float* gs_h_out, float* gs_x_out, double* out2_out,
                double* y64, int64_t* slot_of_out) {
  const int64_t S = T * k;
  std::vector<int64_t> counts(E), offsets(E + 1), slot_flat(S), slot_of(S);
  if (nvo_route(ids, T, k, E, counts.data(), offsets.data(), slot_flat.data(), slot_of.data()))
    return -1;
  // step 2: activations
  std::vector<uint8_t> xq(static_cast<size_t>(T * H / 2)), xsf(static_cast<size_t>(T * H / 16));
  float gs_x = 1.0f;
  nvo_quantize_rows(x, T, H, 0, 0.0f, xq.data(), xsf.data(), &gs_x);
  // steps 3 + 6: L1 per expert on its slots' token rows
  std::vector<double> l1(static_cast<size_t>(S * 2 * I), 0.0);
  for (int e = 0; e < E; ++e) {
    const int64_t s0 = offsets[e], n = counts[e];
    if (n == 0) continue;
    std::vector<uint8_t> aq(static_cast<size_t>(n * H / 2)), asf(static_cast<size_t>(n * H / 16));
    for (int64_t i = 0; i < n; ++i) {
      const int64_t t = slot_flat[s0 + i] / k;
      std::memcpy(&aq[i * H / 2], &xq[t * H / 2], H / 2);
      std::memcpy(&asf[i * H / 16], &xsf[t * H / 16], H / 16);
    }
    std::vector<double> acc(static_cast<size_t>(n * 2 * I));
    nvo_block_scaled_matmul(aq.data(), asf.data(), n, H, w1_q + e * (H / 2) * (2 * I),
                            w1_sf + e * (H / 16) * (2 * I), 2 * I, acc.data());
    const double a_gate = static_cast<double>(gs_x) *
                          static_cast<double>(gs1_split ? gs_w1[2 * e] : gs_w1[e]);
    const double a_up = static_cast<double>(gs_x) *
                        static_cast<double>(gs1_split ? gs_w1[2 * e + 1] : gs_w1[e]);
    for (int64_t i = 0; i < n; ++i)
      for (int64_t c = 0; c < 2 * I; ++c)
        l1[(s0 + i) * 2 * I + c] = acc[i * 2 * I + c] * (c < I ? a_gate : a_up);
  }
  // step 4: SiLU(gate) * up, then requantisation
  std::vector<float> h(static_cast<size_t>(S * I));
  nvo_swiglu(l1.data(), S, I, h.data());
  std::vector<uint8_t> hq(static_cast<size_t>(S * I / 2)), hsf(static_cast<size_t>(S * I / 16));
  float gs_h = 1.0f;
  if (gs_mid == nullptr) {
    nvo_quantize_rows(h.data(), S, I, 0, 0.0f, hq.data(), hsf.data(), &gs_h);
  } else {
    for (int e = 0; e < E; ++e) {
      if (counts[e] == 0) continue;
      float unused = 0.0f;
      nvo_quantize_rows(h.data() + offsets[e] * I, counts[e], I, 1, gs_mid[e],
                        hq.data() + offsets[e] * I / 2, hsf.data() + offsets[e] * I / 16, &unused);
    }
  }
  // steps 5 + 6: L2 per expert
  std::vector<double> out2(static_cast<size_t>(S * H), 0.0);
  for (int e = 0; e < E; ++e) {
    const int64_t s0 = offsets[e], n = counts[e];
    if (n == 0) continue;
    std::vector<double> acc(static_cast<size_t>(n * H));
    nvo_block_scaled_matmul(hq.data() + s0 * I / 2, hsf.data() + s0 * I / 16, n, I,
                            w2_q + e * (I / 2) * H, w2_sf + e * (I / 16) * H, H, acc.data());
    const double alpha = static_cast<double>(gs_mid == nullptr ? gs_h : gs_mid[e]) *
                         static_cast<double>(gs_w2[e]);
    for (int64_t i = 0; i < n * H; ++i) out2[s0 * H + i] = acc[i] * alpha;
  }
  // step 7
  std::vector<double> w64(w, w + S);
  nvo_unpermute_reduce(out2.data(), H, slot_of.data(), w64.data(), T, k, y64);

  if (l1_out) std::memcpy(l1_out, l1.data(), l1.size() * sizeof(double));
  if (h_out) std::memcpy(h_out, h.data(), h.size() * sizeof(float));
  if (hq_out) std::memcpy(hq_out, hq.data(), hq.size());
  if (hsf_out) std::memcpy(hsf_out, hsf.data(), hsf.size());
  if (gs_h_out) *gs_h_out = gs_h;
  if (gs_x_out) *gs_x_out = gs_x;
  if (out2_out) std::memcpy(out2_out, out2.data(), out2.size() * sizeof(double));
  if (slot_of_out) std::memcpy(slot_of_out, slot_of.data(), slot_of.size() * sizeof(int64_t));
  return 0;
}

int nvo_max_threads(void) { return omp_get_max_threads(); }
void nvo_set_threads(int n) { omp_set_num_threads(n); }

}  // extern "C"
