// Plain CPU oracle for the IQ4_NL routed-expert MoE layer.
//
// TEST INFRASTRUCTURE. Only the tests, the package smoke check and the
// benchmark's CPU-baseline leg call this code. The CUDA library never links it,
// and this file shares no header, helper or table with that library.
//
// Everything is computed with plain loops in double precision. Results are
// rounded to fp32 only by the caller, at the output. This follows the Red Lite
// page "What we learned", section 7 ("How we know it is correct"): every native
// stage is compared with a CPU reference computed in double precision.
//
// Sources of each definition:
//  * IQ4_NL block (GGML type 20): 32 weights in 18 bytes, as stated in the
//    Overview table of the PocketLLM page "Xing4.0-29B-A4B". The byte layout
//    (little-endian fp16 scale d, then 16 bytes of nibble pairs; the low nibble
//    of byte j is weight j and the high nibble is weight j+16) and the 16-entry
//    table are those of the published GGML format.
//  * Router: the same page's Overview calls the MoE "sigmoid-routed ... with a
//    shared expert". Scores are W_r x; the top-k choice is made on
//    sigmoid(score) + bias (descending, ties to the lower index); the combine
//    weights are the chosen sigmoids, renormalised to sum to one. The bias takes
//    part in the choice only.
//  * Expert: a SwiGLU FFN, h = silu(W_g x) * (W_u x), o = W_d h. The shared
//    expert is always on and has weight 1.
//  * Combine: y_t = sum_j w_tj o(e_tj, x_t) + o_shared(x_t), taken in slot
//    order; the Xing4.0 page's closing list calls this the MoE's
//    "deterministic route reduction".
//  * Invalid routes: the wpnews article "Running Qwen Flash-Next NVFP4 in vLLM"
//    (its passage on invalid expert routes) maps an id outside [0, E) to expert
//    0 and sets its weight to 0.
//
// Mode "mma16" is the same computation with three roundings to fp16
// (round-to-nearest-even, subnormals kept): each dequantised weight d*T[q],
// each activation x, and each h before the down projection. It is the
// reference for the tensor-core prefill path, whose operands are fp16.
//
// Mode "mma8" is the reference for the prefill path with 8-bit operands (the
// Xolotl blog's "Prompts" passage runs its prompt contraction on the 4090's
// int8 tensor cores; the 8-bit format taken here is floating point, the one
// whose tensor rate is fast on the target GPU). The format is E4M3 of the OCP
// 8-bit floating point
// specification (1 sign, 4 exponent bits with bias 7, 3 fraction bits; no
// infinities, S.1111.111 is NaN, largest finite 448), rounded to nearest with
// ties to even and finite overflow saturated to +-448. E4M3 spans fewer
// binades than IQ4_NL weights or activations, so each value is rounded after
// a power-of-two scaling that the contraction's output undoes exactly:
//  * a weight row m (K inputs) is scaled by 2^-E_m, E_m the largest exponent
//    of its blocks' fp16 scales d (-14 for a subnormal or zero d), so that
//    |d*T*2^-E_m| < 254 for every weight of the row: w8 = 2^E_m e4m3(d*T*2^-E_m);
//  * an activation vector v (a token's x, or one (token, expert) pair's h) is
//    scaled by 2^-X, X = floor(log2 max|v|) - 6 (0 for an all-zero vector), so
//    that its largest magnitude lies in [64, 128): v8 = 2^X e4m3(v*2^-X).
// Everything else, as in the exact mode, is a plain double computation.

#include <cmath>
#include <cstdint>
#include <cstring>
#include <vector>
#include <algorithm>
#include <limits>
#ifdef _OPENMP
#include <omp.h>
#endif

namespace {

// The IQ4_NL non-linear table (GGML type 20).
const int kTable[16] = {-127, -104, -83, -65, -49, -35, -22, -10,
                        1,    13,   25,  38,  53,  69,  89,  113};

constexpr int kBlockWeights = 32;
constexpr int kBlockBytes = 18;

// IEEE 754 binary16 bit pattern -> double. Written from the field layout:
// 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits.
double half_to_double(uint16_t h) {
  const int sign = h >> 15;
  const int e = (h >> 10) & 0x1F;
  const int m = h & 0x3FF;
  double v;
  if (e == 0) {
    v = std::ldexp(static_cast<double>(m), -24);              // zero / subnormal
  } else if (e == 31) {
    v = m ? std::numeric_limits<double>::quiet_NaN()
          : std::numeric_limits<double>::infinity();
  } else {
    v = std::ldexp(static_cast<double>(1024 + m), e - 25);    // (1 + m/2^10) 2^(e-15)
  }
  return sign ? -v : v;
}

// bfloat16 bit pattern -> double. bfloat16 is the upper half of an IEEE 754
// binary32: 1 sign bit, 8 exponent bits (bias 127), 7 fraction bits.
double bf16_to_double(uint16_t b) {
  const int sign = b >> 15;
  const int e = (b >> 7) & 0xFF;
  const int m = b & 0x7F;
  double v;
  if (e == 0) {
    v = std::ldexp(static_cast<double>(m), -133);             // zero / subnormal
  } else if (e == 255) {
    v = m ? std::numeric_limits<double>::quiet_NaN()
          : std::numeric_limits<double>::infinity();
  } else {
    v = std::ldexp(static_cast<double>(128 + m), e - 134);    // (1 + m/2^7) 2^(e-127)
  }
  return sign ? -v : v;
}

// double -> binary16 bit pattern, round to nearest, ties to even, with
// subnormals and overflow to infinity.
uint16_t double_to_half(double v) {
  const uint16_t sign = std::signbit(v) ? 0x8000 : 0;
  if (std::isnan(v)) return 0x7E00;
  const double a = std::fabs(v);
  if (std::isinf(a)) return sign | 0x7C00;
  if (a == 0.0) return sign;
  int ex = 0;
  std::frexp(a, &ex);                 // a = f 2^ex, f in [0.5, 1)
  int e = ex - 1;                     // floor(log2 a)
  if (e > 15) return sign | 0x7C00;   // a >= 2^16: beyond every finite half
  if (e < -14) e = -14;               // subnormal range shares the 2^-24 quantum
  const double q = std::ldexp(1.0, e - 10);
  const double n = a / q;             // exact: division by a power of two
  double r = std::floor(n);
  const double frac = n - r;          // exact
  if (frac > 0.5 || (frac == 0.5 && std::fmod(r, 2.0) != 0.0)) r += 1.0;
  long ri = static_cast<long>(r);
  if (ri == 2048) { ri = 1024; e += 1; }
  if (e > 15) return sign | 0x7C00;
  if (ri < 1024) return sign | static_cast<uint16_t>(ri);   // subnormal (e == -14)
  return sign | static_cast<uint16_t>(((e + 15) << 10) | (ri - 1024));
}

double round_to_half(double v) { return half_to_double(double_to_half(v)); }

// E4M3 byte -> double, from the field layout: e = bits 6..3, f = bits 2..0;
// e == 0: subnormal f/8 * 2^-6; else (1 + f/8) * 2^(e-7); S.1111.111 is NaN.
double e4m3_to_double(uint8_t c) {
  const int sgn = (c >> 7) & 1, e = (c >> 3) & 0xF, f = c & 7;
  if (e == 0xF && f == 7) return std::numeric_limits<double>::quiet_NaN();
  const double mag = (e == 0) ? std::ldexp(f / 8.0, -6) : std::ldexp(1.0 + f / 8.0, e - 7);
  return sgn ? -mag : mag;
}

// double -> E4M3, round to nearest with ties to even (on the 3-bit fraction,
// subnormals included), finite overflow saturated to +-448, NaN to 0x7F.
uint8_t double_to_e4m3(double v) {
  if (std::isnan(v)) return 0x7F;
  const uint8_t sgn = std::signbit(v) ? 0x80 : 0x00;
  double a = std::fabs(v);
  if (a >= 448.0) return sgn | 0x7E;               // saturate (the largest finite, 1.110 x 2^8)
  // the quantum of a's binade: 2^(e-3) for normals (e >= -6), 2^-9 below
  int e = 0;
  std::frexp(a, &e);                               // a = m 2^e, m in [0.5, 1)
  int ex = e - 1;                                  // floor(log2 a) for a > 0
  if (a == 0.0 || ex < -6) ex = -6;
  const double q = std::ldexp(1.0, ex - 3);
  double n = a / q;                                // exact: a power-of-two scaling
  double r = std::floor(n);
  const double frac = n - r;
  if (frac > 0.5 || (frac == 0.5 && std::fmod(r, 2.0) != 0.0)) r += 1.0;
  const double rv = r * q;                         // the rounded magnitude
  if (rv >= 448.0) return sgn | 0x7E;
  if (rv == 0.0) return sgn;
  int e2 = 0;
  std::frexp(rv, &e2);
  int ebin = e2 - 1;                               // rv's binade after rounding
  if (ebin < -6) {                                 // subnormal: f/8 * 2^-6
    const int f = static_cast<int>(std::ldexp(rv, 9));
    return sgn | static_cast<uint8_t>(f);
  }
  const int f = static_cast<int>(std::ldexp(rv, 3 - ebin)) - 8;
  return sgn | static_cast<uint8_t>(((ebin + 7) << 3) | f);
}
double round_to_e4m3(double v) { return e4m3_to_double(double_to_e4m3(v)); }

// Exponent of an fp16 scale for the row scaling: floor(log2 |d|) for a normal
// d (its biased exponent field minus 15), -14 for a subnormal or zero d.
int half_exponent(uint16_t dbits) {
  const int f = (dbits >> 10) & 0x1F;
  return f == 0 ? -14 : f - 15;
}

// The row exponent E_m: the largest exponent of the row's block scales.
int row_exponent(const uint8_t* row, int nb) {
  int e = -1000;
  for (int b = 0; b < nb; ++b) {
    const uint8_t* blk = row + static_cast<size_t>(b) * 18;
    const int eb = half_exponent(static_cast<uint16_t>(blk[0] | (blk[1] << 8)));
    e = eb > e ? eb : e;
  }
  return e;
}

// An activation vector's exponent X = floor(log2 max|v|) - 6; 0 when all zero.
int vector_exponent(const double* v, int n) {
  double m = 0.0;
  for (int i = 0; i < n; ++i) m = std::fabs(v[i]) > m ? std::fabs(v[i]) : m;
  if (!(m > 0.0) || !std::isfinite(m)) return 0;
  int e = 0;
  std::frexp(m, &e);
  return (e - 1) - 6;
}

// v <- 2^X e4m3(v 2^-X) with the vector's own exponent.
void round_vector_e4m3(double* v, int n) {
  const int X = vector_exponent(v, n);
  for (int i = 0; i < n; ++i) v[i] = std::ldexp(round_to_e4m3(std::ldexp(v[i], -X)), X);
}

// Dequantise one 18-byte block into 32 doubles.
void dequant_block(const uint8_t* blk, int mode, double* w) {
  const uint16_t dbits = static_cast<uint16_t>(blk[0] | (blk[1] << 8));
  const double d = half_to_double(dbits);
  for (int j = 0; j < 16; ++j) {
    const uint8_t q = blk[2 + j];
    w[j] = d * kTable[q & 0x0F];
    w[j + 16] = d * kTable[q >> 4];
  }
  if (mode == 1)
    for (int i = 0; i < kBlockWeights; ++i) w[i] = round_to_half(w[i]);
}

// Mode 2 dequantisation of one block of a row with exponent E.
void dequant_block_e4m3(const uint8_t* blk, int E, double* w) {
  dequant_block(blk, 0, w);
  for (int i = 0; i < kBlockWeights; ++i) w[i] = std::ldexp(round_to_e4m3(std::ldexp(w[i], -E)), E);
}

// Row r of a matrix with K inputs: blocks r*K/32 ... r*K/32 + K/32 - 1.
double row_dot(const uint8_t* mat, int r, int K, const double* v, int mode) {
  const int nb = K / kBlockWeights;
  const uint8_t* row = mat + static_cast<size_t>(r) * nb * kBlockBytes;
  double acc = 0.0;
  double w[kBlockWeights];
  const int E = mode == 2 ? row_exponent(row, nb) : 0;
  for (int b = 0; b < nb; ++b) {
    if (mode == 2)
      dequant_block_e4m3(row + static_cast<size_t>(b) * kBlockBytes, E, w);
    else
      dequant_block(row + static_cast<size_t>(b) * kBlockBytes, mode, w);
    for (int i = 0; i < kBlockWeights; ++i) acc += w[i] * v[b * kBlockWeights + i];
  }
  return acc;
}

double silu_times(double g, double u) { return g * u / (1.0 + std::exp(-g)); }

// One SwiGLU expert on one activation vector. gate, up: [F][H/32] blocks;
// down: [H][F/32] blocks. x has H entries, o receives H entries.
void expert_ffn(int H, int F, const uint8_t* gate, const uint8_t* up,
                const uint8_t* down, const double* x, int mode, double* o) {
  std::vector<double> h(F);
  for (int f = 0; f < F; ++f) {
    const double g = row_dot(gate, f, H, x, mode);
    const double u = row_dot(up, f, H, x, mode);
    double hv = silu_times(g, u);
    if (mode == 1) hv = round_to_half(hv);
    h[f] = hv;
  }
  if (mode == 2) round_vector_e4m3(h.data(), F);
  for (int n = 0; n < H; ++n) o[n] = row_dot(down, n, F, h.data(), mode);
}

}  // namespace

extern "C" {

int orc_table(int32_t* out16) {
  for (int i = 0; i < 16; ++i) out16[i] = kTable[i];
  return 0;
}

double orc_half_to_double(uint16_t h) { return half_to_double(h); }
double orc_e4m3_to_double(uint8_t c) { return e4m3_to_double(c); }
uint8_t orc_double_to_e4m3(double v) { return double_to_e4m3(v); }

// Mode-2 weights of `rows` rows of a K-input matrix, as doubles [rows][K], and
// each row's exponent E_m (row_exp may be NULL).
int orc_dequant_rows_e4m3(const uint8_t* mat, int64_t rows, int K, double* out,
                          int32_t* row_exp) {
  if (!mat || !out || rows < 0 || K <= 0 || K % 32) return -1;
  const int nb = K / 32;
  for (int64_t r = 0; r < rows; ++r) {
    const uint8_t* row = mat + static_cast<size_t>(r) * nb * kBlockBytes;
    const int E = row_exponent(row, nb);
    if (row_exp) row_exp[r] = E;
    for (int b = 0; b < nb; ++b)
      dequant_block_e4m3(row + static_cast<size_t>(b) * kBlockBytes, E,
                         out + static_cast<size_t>(r) * K + static_cast<size_t>(b) * 32);
  }
  return 0;
}
double orc_bf16_to_double(uint16_t b) { return bf16_to_double(b); }
uint16_t orc_double_to_half(double v) { return double_to_half(v); }

// Dequantise n_blocks consecutive blocks. mode 0: exact d*T[q];
// mode 1: each product rounded to fp16 (returned as its double value).
int orc_dequant_blocks(const uint8_t* blocks, int64_t n_blocks, int mode, double* out) {
  if (!blocks || !out || n_blocks < 0 || (mode != 0 && mode != 1)) return -1;
  for (int64_t b = 0; b < n_blocks; ++b)
    dequant_block(blocks + b * kBlockBytes, mode, out + b * kBlockWeights);
  return 0;
}

// Invalid-route rule of the vLLM article: an id outside [0, E) becomes expert
// 0 with weight 0; valid routes keep both. Returns the number of invalid routes.
int orc_sanitize(const int32_t* ids, const double* w, int64_t n, int E,
                 int32_t* ids_out, double* w_out) {
  int bad = 0;
  for (int64_t i = 0; i < n; ++i) {
    const bool ok = ids[i] >= 0 && ids[i] < E;
    ids_out[i] = ok ? ids[i] : 0;
    w_out[i] = ok ? w[i] : 0.0;
    bad += ok ? 0 : 1;
  }
  return bad;
}

// Router. Wr: bf16 [E][H]; bias: fp32 [E] or NULL; x: bf16 [T][H].
// Out: ids [T][k] in descending key order (ties to the lower index),
// w [T][k] renormalised sigmoids, gap [T] = key of the k-th choice minus the
// key of the best unchosen expert (+inf when k == E), scores [T][E] optional.
int orc_route(int H, int E, int k, const uint16_t* Wr, const float* bias,
              const uint16_t* x, int T, int32_t* ids, double* w, double* gap,
              double* scores) {
  if (H <= 0 || E <= 0 || k <= 0 || k > E || T < 0 || !Wr || !x || !ids || !w)
    return -1;
  std::vector<double> xv(H), p(E), key(E);
  std::vector<int> order(E);
  for (int t = 0; t < T; ++t) {
    for (int h = 0; h < H; ++h) xv[h] = bf16_to_double(x[static_cast<size_t>(t) * H + h]);
    for (int e = 0; e < E; ++e) {
      double s = 0.0;
      for (int h = 0; h < H; ++h)
        s += bf16_to_double(Wr[static_cast<size_t>(e) * H + h]) * xv[h];
      if (scores) scores[static_cast<size_t>(t) * E + e] = s;
      p[e] = 1.0 / (1.0 + std::exp(-s));
      key[e] = p[e] + (bias ? static_cast<double>(bias[e]) : 0.0);
    }
    for (int e = 0; e < E; ++e) order[e] = e;
    std::stable_sort(order.begin(), order.end(),
                     [&](int a, int b) { return key[a] > key[b]; });
    double sum = 0.0;
    for (int j = 0; j < k; ++j) sum += p[order[j]];
    for (int j = 0; j < k; ++j) {
      ids[static_cast<size_t>(t) * k + j] = order[j];
      w[static_cast<size_t>(t) * k + j] = p[order[j]] / sum;
    }
    if (gap)
      gap[t] = (k < E) ? key[order[k - 1]] - key[order[k]]
                       : std::numeric_limits<double>::infinity();
  }
  return 0;
}

// One expert on one bf16 activation row (for dense checks). Returns o [H].
int orc_expert_ffn(int H, int F, const uint8_t* gate, const uint8_t* up,
                   const uint8_t* down, const uint16_t* x, int mode, double* o) {
  if (H <= 0 || F <= 0 || H % 32 || F % 32 || !gate || !up || !down || !x || !o) return -1;
  if (mode != 0 && mode != 1 && mode != 2) return -1;
  std::vector<double> xv(H);
  for (int h = 0; h < H; ++h) {
    xv[h] = bf16_to_double(x[h]);
    if (mode == 1) xv[h] = round_to_half(xv[h]);
  }
  if (mode == 2) round_vector_e4m3(xv.data(), H);
  expert_ffn(H, F, gate, up, down, xv.data(), mode, o);
  return 0;
}

// The whole layer for T tokens, given routes (ids, w: [T][k]).
// gate/up/down: E pointers, each to one expert's blocks (NULL allowed for an
// expert no valid route uses). sh_*: the shared expert (ignored when
// n_shared == 0). y: [T][H] doubles. threads > 1 runs the (token, expert)
// pairs in parallel; the combine is always sequential in slot order.
// Returns 0, or -1 on bad arguments, -2 when a routed expert's pointer is NULL.
int orc_moe_layer(int H, int F, int Fs, int E, int k, int n_shared,
                  const uint8_t* const* gate, const uint8_t* const* up,
                  const uint8_t* const* down, const uint8_t* sh_gate,
                  const uint8_t* sh_up, const uint8_t* sh_down, const uint16_t* x,
                  int T, const int32_t* ids, const double* w, int mode, int threads,
                  double* y) {
  if (H <= 0 || F <= 0 || H % 32 || F % 32 || E <= 0 || k <= 0 || k > E || T < 0 ||
      (n_shared != 0 && n_shared != 1) || (mode != 0 && mode != 1 && mode != 2) || !x || !y ||
      (T > 0 && (!ids || !w)))
    return -1;
  if (n_shared && (Fs <= 0 || Fs % 32 || !sh_gate || !sh_up || !sh_down)) return -1;
  const int64_t n_pairs = static_cast<int64_t>(T) * (k + n_shared);
  std::vector<int32_t> sid(static_cast<size_t>(T) * k);
  std::vector<double> sw(static_cast<size_t>(T) * k);
  orc_sanitize(ids, w, static_cast<int64_t>(T) * k, E, sid.data(), sw.data());
  for (size_t i = 0; i < sid.size(); ++i)
    if (!gate[sid[i]] || !up[sid[i]] || !down[sid[i]]) return -2;
  // Activations, rounded to fp16 (mode mma16) or per token to E4M3 (mma8).
  std::vector<double> xv(static_cast<size_t>(T) * H);
  for (size_t i = 0; i < xv.size(); ++i) {
    xv[i] = bf16_to_double(x[i]);
    if (mode == 1) xv[i] = round_to_half(xv[i]);
  }
  if (mode == 2)
    for (int t = 0; t < T; ++t) round_vector_e4m3(xv.data() + static_cast<size_t>(t) * H, H);
  std::vector<double> o(static_cast<size_t>(n_pairs) * H);
  const int kk = k + n_shared;
  auto run_pair = [&](int64_t p) {
    const int t = static_cast<int>(p / kk);
    const int j = static_cast<int>(p % kk);
    const double* xt = xv.data() + static_cast<size_t>(t) * H;
    double* op = o.data() + static_cast<size_t>(p) * H;
    if (j < k) {
      const int e = sid[static_cast<size_t>(t) * k + j];
      expert_ffn(H, F, gate[e], up[e], down[e], xt, mode, op);
    } else {
      expert_ffn(H, Fs, sh_gate, sh_up, sh_down, xt, mode, op);
    }
  };
#ifdef _OPENMP
  if (threads > 1) {
#pragma omp parallel for num_threads(threads) schedule(dynamic, 1)
    for (int64_t p = 0; p < n_pairs; ++p) run_pair(p);
  } else {
    for (int64_t p = 0; p < n_pairs; ++p) run_pair(p);
  }
#else
  (void)threads;
  for (int64_t p = 0; p < n_pairs; ++p) run_pair(p);
#endif
  for (int t = 0; t < T; ++t) {
    for (int n = 0; n < H; ++n) {
      double acc = 0.0;
      for (int j = 0; j < k; ++j)
        acc += sw[static_cast<size_t>(t) * k + j] *
               o[(static_cast<size_t>(t) * kk + j) * H + n];
      if (n_shared) acc += o[(static_cast<size_t>(t) * kk + k) * H + n];
      y[static_cast<size_t>(t) * H + n] = acc;
    }
  }
  return 0;
}

int orc_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

}  // extern "C"
