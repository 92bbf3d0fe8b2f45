// bsgg_oracle.cpp -- plain, slow CPU reference for the grouped block-scaled GEMM
// with fused per-row epilogue and output quantization.
//
// TEST INFRASTRUCTURE ONLY.  This file is the parity oracle: nothing in the
// product library links, includes or calls it.  Only the test suite, the smoke
// check (__graft_entry__.smoke) and the CPU-baseline leg of bench.py load it.
// It shares no code, table, header or constant generator with the CUDA path.
//
// Every function follows one passage of the cuDNN-frontend documentation pages
// (cited by page title and section) and is written for a reader to check by
// eye: decode by table, dequantize, accumulate in fp64, apply the epilogue in
// fp64, then take the quantization decisions in fp32 (the pages evaluate the
// epilogue in FP32; "Grouped GEMM + sReLU", section "Tanh soft clamp").
//
// Parity pins: every function here is pinned by tests/test_oracle_*.py against
// closed forms, brute force, invariants and hand-worked examples, and
// tests/test_pin_mutants.py checks that those pins fail on copies of this file
// with one plausible mistake planted in each.  No function is "parity
// unpinned".  The one unpinned quantity is the *rate* of one-code
// flips caused by the device's approximate tanh; the tolerance covers it.
//
// Where the pages are silent this file takes a reading of them, marked
// "reading:" where it is implemented.

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <thread>
#include <vector>

namespace {

// ---------------------------------------------------------------------------
// Number formats.  Pages: "Grouped GEMM + Quant (SM100)", Data Types table
// (MXFP8 = float8_e4m3fn / float8_e5m2 data with float8_e8m0fnu scales per 32;
// NVF4 = float4_e2m1fn_x2 data with float8_e4m3fn scales per 16).  The values
// below are the OCP microscaling format definitions written out.
// ---------------------------------------------------------------------------

enum Fmt { F_E4M3 = 0, F_E5M2 = 1, F_E2M1 = 2, F_UE8M0 = 3 };

// E4M3 ("fn"): 1 sign, 4 exponent (bias 7), 3 mantissa; no infinity;
// S.1111.111 is NaN; largest finite 448.
double e4m3_value(uint8_t c) {
  int s = (c >> 7) & 1, e = (c >> 3) & 0xF, m = c & 7;
  double v;
  if (e == 0xF && m == 7) return NAN;
  if (e == 0) v = std::ldexp(m / 8.0, -6);          // subnormal: 0.m * 2^(1-7)
  else v = std::ldexp(1.0 + m / 8.0, e - 7);
  return s ? -v : v;
}

// E5M2: 1 sign, 5 exponent (bias 15), 2 mantissa; IEEE-style inf and NaN;
// largest finite 57344.
double e5m2_value(uint8_t c) {
  int s = (c >> 7) & 1, e = (c >> 2) & 0x1F, m = c & 3;
  double v;
  if (e == 0x1F) v = (m == 0) ? INFINITY : NAN;
  else if (e == 0) v = std::ldexp(m / 4.0, -14);
  else v = std::ldexp(1.0 + m / 4.0, e - 15);
  return s ? -v : v;
}

// E2M1: 1 sign, 2 exponent (bias 1), 1 mantissa; no inf/NaN; values
// {0, 0.5, 1, 1.5, 2, 3, 4, 6}.
double e2m1_value(uint8_t nib) {
  int s = (nib >> 3) & 1, e = (nib >> 1) & 3, m = nib & 1;
  double v = (e == 0) ? 0.5 * m : std::ldexp(1.0 + m / 2.0, e - 1);
  return s ? -v : v;
}

// UE8M0: unsigned power of two 2^(c-127); 0xFF is NaN.
double ue8m0_value(uint8_t c) { return c == 0xFF ? NAN : std::ldexp(1.0, int(c) - 127); }

struct Tables {
  double e4m3[256], e5m2[256], e2m1[16], ue8m0[256];
  Tables() {
    for (int c = 0; c < 256; ++c) {
      e4m3[c] = e4m3_value(uint8_t(c));
      e5m2[c] = e5m2_value(uint8_t(c));
      ue8m0[c] = ue8m0_value(uint8_t(c));
    }
    for (int c = 0; c < 16; ++c) e2m1[c] = e2m1_value(uint8_t(c));
  }
};
const Tables& tables() { static Tables t; return t; }

double decode(int fmt, uint32_t code) {
  const Tables& t = tables();
  switch (fmt) {
    case F_E4M3: return t.e4m3[code & 0xFF];
    case F_E5M2: return t.e5m2[code & 0xFF];
    case F_E2M1: return t.e2m1[code & 0xF];
    case F_UE8M0: return t.ue8m0[code & 0xFF];
  }
  return NAN;
}

// Largest finite positive code of each signed format.
uint32_t max_code(int fmt) { return fmt == F_E4M3 ? 0x7E : fmt == F_E5M2 ? 0x7B : 0x7; }
uint32_t sign_bit(int fmt) { return fmt == F_E2M1 ? 0x8 : 0x80; }

// Round-to-nearest-even with saturation to the largest finite value
// (reading: the pages do not name the output conversion's rounding; we take
// RNE, satfinite).  Positive codes 0..max_code are increasing in value, so the
// nearest code is found by bisection; on an exact tie the code whose last
// mantissa bit is 0 (the even code) wins.
uint32_t encode_rne_satfinite(int fmt, float x) {
  if (std::isnan(x)) return fmt == F_E2M1 ? 0x7 : 0x7F;   // E2M1 has no NaN
  const uint32_t sgn = std::signbit(x) ? sign_bit(fmt) : 0;
  const double ax = std::fabs(double(x));
  const uint32_t top = max_code(fmt);
  if (ax >= decode(fmt, top)) return sgn | top;
  uint32_t lo = 0, hi = top;              // invariant: value(lo) <= ax < value(hi)
  while (hi - lo > 1) {
    uint32_t mid = (lo + hi) / 2;
    if (decode(fmt, mid) <= ax) lo = mid; else hi = mid;
  }
  const double dlo = ax - decode(fmt, lo), dhi = decode(fmt, hi) - ax;
  uint32_t pick;
  if (dlo < dhi) pick = lo;
  else if (dhi < dlo) pick = hi;
  else pick = (lo % 2 == 0) ? lo : hi;
  return sgn | pick;
}

// Scale-factor encoding for UE8M0 (reading: round UP to a power of two, so that
// |D * norm / SFD| never exceeds q_max; the same rule the inputs use).
// sf <= 0 (an all-zero block) encodes as code 0.
uint32_t encode_ue8m0_ceil(float sf) {
  if (std::isnan(sf)) return 0xFF;
  if (!(sf > 0.0f)) return 0;
  int p;
  double m = std::frexp(double(sf), &p);     // sf = m * 2^p, m in [0.5, 1)
  int e = (m == 0.5) ? p - 1 : p;            // ceil(log2(sf))
  int code = e + 127;
  return uint32_t(std::min(254, std::max(0, code)));
}

// ---------------------------------------------------------------------------
// Scale-factor layout.  Pages: "Grouped GEMM + Quant (SM100)", Shapes (SFA is
// (32, 4, ceil(rows/128), 4, ceil(ceil(K/sf_vec)/4), L)) and "Grouped GEMM +
// SwiGLU (SM100)", Canonical layouts (physical C-contiguous order
// (L, ceil(rows/128), ceil(kblocks/4), 32, 4, 4)).  Logical index
// (i0, i1, i2, i3, i4, l) names row = 128*i2 + 32*i1 + i0 and
// k-block = 4*i4 + i3.
// ---------------------------------------------------------------------------
int64_t sf_offset(int64_t row, int64_t kblk, int64_t l, int64_t rows, int64_t kblocks) {
  const int64_t R = (rows + 127) / 128, KQ = (kblocks + 3) / 4;
  const int64_t i0 = row % 32, i1 = (row / 32) % 4, i2 = row / 128;
  const int64_t i3 = kblk % 4, i4 = kblk / 4;
  return ((((l * R + i2) * KQ + i4) * 32 + i0) * 4 + i1) * 4 + i3;
}
int64_t sf_bytes(int64_t rows, int64_t kblocks, int64_t L) {
  return L * ((rows + 127) / 128) * ((kblocks + 3) / 4) * 512;
}

// ---------------------------------------------------------------------------
// Problem description (the oracle's own; the library's header is not used).
// ---------------------------------------------------------------------------
// "Grouped GEMM + Quant (SM100)", Data Types: FP4 data takes E4M3 scales per 16
// (NVFP4) or UE8M0 scales per 16 or 32 (E4M3 is incompatible with 32).
// IN_BF16: the BF16 backend of "Grouped GEMM + dGLU (SM100)" (BF16 contract):
// bfloat16 A and B, no scale factors.
enum InFmt { IN_MXFP8_E4M3 = 0, IN_MXFP8_E5M2 = 1, IN_NVFP4 = 2, IN_FP4_UE8M0_16 = 3, IN_MXFP4 = 4, IN_BF16 = 5 };
enum OutFmt { OUT_BF16 = 0, OUT_F16 = 1, OUT_F32 = 2, OUT_E4M3 = 3, OUT_E5M2 = 4, OUT_E2M1 = 5 };
// EPI_DSWIGLU, EPI_DGEGLU, EPI_DSITUGLU: the backward epilogues of "Grouped GEMM +
// dGLU (SM100)".
enum Epi {
  EPI_GATE = 0, EPI_SWIGLU = 1, EPI_SRELU = 2, EPI_GEGLU = 3, EPI_DSWIGLU = 4, EPI_DGEGLU = 5,
  EPI_DSITUGLU = 6
};

}  // namespace

extern "C" {

typedef struct {
  int64_t m_pad, n, k, num_groups;
  // rht: the Hadamard output of "Grouped GEMM + GLU + Hadamard + Quant (SM100)"
  // (0 = none, 1 = rowwise bf16, 2 = rowwise NVFP4 with E4M3 scales per 16,
  // 3 = colwise NVFP4: 16-token blocks per column, per-expert transposed)
  int32_t in_fmt, out_fmt, epi, gate_first, want_col, rht;
  double tanh_clamp_s;   // 0 = no clamp
  // "Grouped GEMM + GLU + Hadamard + Quant (SM100)", Equations: both GLU
  // halves clamped to [-glu_limit, glu_limit] (0 = no clamp) and the GLU
  // output scaled by gamma = glu_alpha (1 = none); SwiGLU and GeGLU only.
  double glu_limit;
  double glu_alpha;
  double rht_norm;       // global encode scale of an NVFP4 RHT output (rht_norm_const)
  // dGeGLU ("Grouped GEMM + dGLU (SM100)", Block-scaled contract, Step 2):
  // sigmoid slope, clamp bounds and the offset added to the clamped up value
  double geglu_alpha, glu_clamp_min, glu_clamp_max, linear_offset;
  // dSiTU-GLU (same page, Equations): the tanh scales beta1 (gate) and beta2 (up)
  double situ_beta1, situ_beta2;
} orc_desc;

// ---- exported helpers (pinned individually by the tests) ----
double orc_decode(int fmt, uint32_t code) { return decode(fmt, code); }
uint32_t orc_encode_rne_satfinite(int fmt, float x) { return encode_rne_satfinite(fmt, x); }
uint32_t orc_encode_ue8m0_ceil(float sf) { return encode_ue8m0_ceil(sf); }
int64_t orc_sf_offset(int64_t row, int64_t kblk, int64_t l, int64_t rows, int64_t kblocks) {
  return sf_offset(row, kblk, l, rows, kblocks);
}
int64_t orc_sf_bytes(int64_t rows, int64_t kblocks, int64_t L) { return sf_bytes(rows, kblocks, L); }

// Pack row-major logical scale factors (L, rows, kblocks) into the swizzled
// physical layout; padding bytes are written as zero (the pages' convention
// for untouched padding: "Grouped GEMM + SwiGLU (SM100)", JAX execution).
void orc_pack_sf(const uint8_t* logical, uint8_t* swz, int64_t rows, int64_t kblocks, int64_t L) {
  std::memset(swz, 0, size_t(sf_bytes(rows, kblocks, L)));
  for (int64_t l = 0; l < L; ++l)
    for (int64_t r = 0; r < rows; ++r)
      for (int64_t kb = 0; kb < kblocks; ++kb)
        swz[sf_offset(r, kb, l, rows, kblocks)] = logical[(l * rows + r) * kblocks + kb];
}

// The activation of "Grouped GEMM + SwiGLU (SM100)" Step 2 (swish(x) = x*sigmoid(x))
// and of "Grouped GEMM + sReLU (SM100)", Equations and Tanh soft clamp.
double orc_sigmoid(double x) { return 1.0 / (1.0 + std::exp(-x)); }
// "Grouped GEMM + GLU + Hadamard + Quant (SM100)", Equations: GeGLU of an up
// value u and a gate value g is (u + 1) * g * sigmoid(1.702 * g).
double orc_geglu(double u, double g) { return (u + 1.0) * g * orc_sigmoid(1.702 * g); }
double orc_srelu(double c, double s) {
  double r = c > 0.0 ? c : 0.0;                 // relu
  if (s > 0.0) r = s * std::min(std::tanh(r / s), 1.0);   // soft clamp, t capped at 1
  return r * r;
}

// Round to the nearest bfloat16 value, ties to even (1 sign, 8 exponent, 7
// stored mantissa bits: 8 significant bits for normal values, a fixed quantum
// of 2^-133 below 2^-126).  "Grouped GEMM + GLU + Hadamard + Quant (SM100)",
// Equations: the RHT transforms bf16-rounded D.
double orc_round_bf16(double x) {
  if (x == 0.0 || !std::isfinite(x)) return x;
  int p;
  std::frexp(x, &p);                          // |x| in [2^(p-1), 2^p)
  const int q = std::max(p - 8, -133);        // exponent of the last kept bit
  const double r = std::nearbyint(std::ldexp(x, -q));   // default rounding: to nearest, ties even
  const double y = std::ldexp(r, q);
  return std::fabs(y) > 3.3895313892515355e38 ? std::copysign(INFINITY, y) : y;
}
// Entry (i, j) of the 16 x 16 Sylvester Hadamard matrix, (-1)^popcount(i & j);
// the pages' "fixed 16-wide orthonormal Hadamard transform" is this matrix / 4
// (reading: Sylvester order, no random signs).
double orc_hadamard16(int i, int j) {
  int c = i & j, bits = 0;
  while (c) { bits += c & 1; c >>= 1; }
  return (bits % 2) ? -1.0 : 1.0;
}

// Which group owns row m: the g with padded_offsets[g-1] <= m < padded_offsets[g]
// ("Grouped GEMM + Quant (SM100)", Equations, Step 1).  -1 if none.
int64_t orc_group_of_row(const int32_t* off, int64_t L, int64_t m) {
  int64_t start = 0;
  for (int64_t g = 0; g < L; ++g) {
    if (m >= start && m < off[g]) return g;
    start = off[g];
  }
  return -1;
}

// Reference computation for the 32-row blocks listed in `blocks` (rows
// 32*b .. 32*b+31 of the padded M extent).  Writes, for those rows only:
//   d_ref    [nblocks*32, n_d]  fp64 D before any output conversion
//   d_q, d_col_q, sfd_row, sfd_col   (quantized outputs; full-size buffers in
//            the device layout; NULL when not wanted)
//   amax     [L]: max |D| (fp32) over the computed rows of each group
//            (reading: amax covers all rows of the group's padded range).
// Returns 0, or a negative value for an invalid description.
//   c_ref    [nblocks*32, n] fp64 C (GEMM plus bias, before any clamp or
//            activation) when not NULL
// `bias` (L x n, bias[g*n + col]) is added to C when not NULL.
// The rowwise RHT (P->rht != 0; "Grouped GEMM + GLU + Hadamard + Quant
// (SM100)", Equations): every 16-column block x of bf16-rounded D becomes
// y = (H16 / 4) x, written to rht_ref [nblocks*32, n_d] (fp64) and, for NVFP4,
// quantized into rht_q (packed E2M1, full size) with E4M3 scales per 16 in
// sfrht (swizzled SF(m_pad, n_d)) under rht_norm.
// The dSwiGLU backward (epi = EPI_DSWIGLU, "Grouped GEMM + dGLU (SM100)",
// Block-scaled contract, Steps 1-3) also takes
//   saved_c  [m_pad, 2n] fp64 values of the saved forward C (its input and gate
//            32-column blocks interleaved; the caller decodes its storage type)
//   beta     [L] scale of C per group
// and writes dprob_ref [nblocks*32] fp64 (the listed rows' dprob), dbias
// [L, 2n] fp64 when not NULL (the sum of D over the listed rows of each group:
// "dbias is the per-expert row reduction of interleaved D_row"; reading: of D
// before any output conversion) and, for
// 16/32-bit D, amax [2L]: index 2g for the input-gradient blocks, 2g+1 for the
// gate-gradient blocks (reading of the pages' amax shape (L, 2, 1)).  D is
// (m_pad, 2n).
int orc_run(const orc_desc* P, const uint8_t* A, const uint8_t* SFA, const uint8_t* B,
            const uint8_t* SFB, const int32_t* padded_offsets, const float* alpha,
            const float* prob, const float* bias, const double* saved_c, const float* beta,
            float norm_const, const int64_t* blocks, int64_t nblocks, double* d_ref, double* c_ref,
            double* dprob_ref, uint8_t* d_q, uint8_t* d_col_q, uint8_t* sfd_row, uint8_t* sfd_col,
            float* amax, double* rht_ref, uint8_t* rht_q, uint8_t* sfrht, double* dbias, int threads);

}  // extern "C"

namespace {

struct Job {
  const orc_desc* P;
  const float* bias;
  double* c_ref;
  const double* saved_c;
  const float* beta;
  double* dprob_ref;
  double* rht_ref;
  uint8_t *rht_q, *sfrht;
  double* dbias;          // backward: [L, n_d] row sums of D per group, or null
  const uint8_t *A, *SFA, *B, *SFB;
  const int32_t* off;
  const float *alpha, *prob;
  float norm;
  const int64_t* blocks;
  int64_t nblocks;
  double* d_ref;
  uint8_t *d_q, *d_col_q, *sfd_row, *sfd_col;
  std::vector<float> amax;     // merged under the mutex
  std::mutex mu;
};

bool is_fp4_in(const orc_desc* P) {
  return P->in_fmt == IN_NVFP4 || P->in_fmt == IN_FP4_UE8M0_16 || P->in_fmt == IN_MXFP4;
}
int sf_vec(const orc_desc* P) { return (P->in_fmt == IN_NVFP4 || P->in_fmt == IN_FP4_UE8M0_16) ? 16 : 32; }
int sf_fmt(const orc_desc* P) { return P->in_fmt == IN_NVFP4 ? F_E4M3 : F_UE8M0; }
int data_fmt(const orc_desc* P) {
  return P->in_fmt == IN_MXFP8_E4M3 ? F_E4M3 : P->in_fmt == IN_MXFP8_E5M2 ? F_E5M2 : F_E2M1;
}
bool out_quantized(const orc_desc* P) { return P->out_fmt >= OUT_E4M3; }
int out_code_fmt(const orc_desc* P) {
  return P->out_fmt == OUT_E4M3 ? F_E4M3 : P->out_fmt == OUT_E5M2 ? F_E5M2 : F_E2M1;
}
// q_max: "Grouped GEMM + Quant (SM100)", Step 3 (448 for E4M3, 57344 for E5M2);
// 6 for E2M1, the format's largest value.
double q_max(const orc_desc* P) {
  return P->out_fmt == OUT_E4M3 ? 448.0 : P->out_fmt == OUT_E5M2 ? 57344.0 : 6.0;
}
bool is_glu(const orc_desc* P) { return P->epi == EPI_SWIGLU || P->epi == EPI_GEGLU; }
bool is_bwd(const orc_desc* P) {
  return P->epi == EPI_DSWIGLU || P->epi == EPI_DGEGLU || P->epi == EPI_DSITUGLU;
}
// D width: N/2 for the forward GLUs (two C blocks per D block), 2N for the
// backward (two gradient blocks per GEMM block), else N.
int64_t n_out(const orc_desc* P) { return is_glu(P) ? P->n / 2 : is_bwd(P) ? 2 * P->n : P->n; }

// A bfloat16 value is the upper half of the binary32 value with the same bits;
// its two bytes are stored little-endian.
double bf16_value(const uint8_t* two_bytes) {
  const uint32_t bits = (uint32_t(two_bytes[0]) | (uint32_t(two_bytes[1]) << 8)) << 16;
  float f;
  std::memcpy(&f, &bits, 4);
  return double(f);
}

// Bytes of one K-major operand row: one per FP8 value, half for FP4, two per
// bfloat16 value.
int64_t row_bytes(const orc_desc* P) {
  return P->in_fmt == IN_BF16 ? 2 * P->k : is_fp4_in(P) ? P->k / 2 : P->k;
}

// Element (r, k) of a K-major low-precision operand: one byte per FP8 value,
// two FP4 values per byte with element 2i in the low nibble (reading).
uint32_t element_code(const orc_desc* P, const uint8_t* base, int64_t row, int64_t k) {
  if (is_fp4_in(P)) {
    uint8_t byte = base[row * (P->k / 2) + k / 2];
    return (k % 2 == 0) ? (byte & 0xF) : (byte >> 4);
  }
  return base[row * P->k + k];
}

// Dequantized operand row: value(code) * value(scale of its k-block); a
// bfloat16 row is its values (no scales on the BF16 backend).
void dequant_row(const orc_desc* P, const uint8_t* data, const uint8_t* sf, int64_t row,
                 int64_t rows, int64_t l, double* out) {
  if (P->in_fmt == IN_BF16) {
    for (int64_t k = 0; k < P->k; ++k) out[k] = bf16_value(data + row * 2 * P->k + 2 * k);
    return;
  }
  const int64_t v = sf_vec(P), kblocks = (P->k + v - 1) / v;
  for (int64_t k = 0; k < P->k; ++k) {
    double s = decode(sf_fmt(P), sf[sf_offset(row, k / v, l, rows, kblocks)]);
    out[k] = decode(data_fmt(P), element_code(P, data, row, k)) * s;
  }
}

// Step 3 of "Grouped GEMM + Quant (SM100)": for one block of values of D (a row
// block or a column block), compute the scale factor code and the scale that
// multiplies D before the output conversion.  Decisions in fp32:
//   SFD = norm_const * max|D| * rcp_max,  Dq = D * (norm_const / SFD).
struct BlockScale { uint32_t code; float scale; };
BlockScale block_scale(const orc_desc* P, float norm, float amax_blk) {
  const float rcp_max = float(1.0 / q_max(P));
  const float sf = (norm * amax_blk) * rcp_max;
  BlockScale b;
  b.code = (sf_fmt(P) == F_UE8M0) ? encode_ue8m0_ceil(sf) : encode_rne_satfinite(F_E4M3, sf);
  const float sfd = float(decode(sf_fmt(P), b.code));
  // reading: a block whose max is zero (or whose scale decodes to zero) is
  // written with scale 0, so its values stay (signed) zero.
  b.scale = (amax_blk == 0.0f || sfd == 0.0f) ? 0.0f : norm / sfd;
  return b;
}

void store_code(const orc_desc* P, uint8_t* buf, int64_t m, int64_t j, uint32_t code) {
  const int64_t nd = n_out(P);
  if (P->out_fmt == OUT_E2M1) {
    uint8_t& byte = buf[m * (nd / 2) + j / 2];
    if (j % 2 == 0) byte = uint8_t((byte & 0xF0) | (code & 0xF));
    else byte = uint8_t((byte & 0x0F) | ((code & 0xF) << 4));
  } else {
    buf[m * nd + j] = uint8_t(code);
  }
}

// One work item: 32-row block `bi` (index into the block list) and output
// columns [j0, j1) of D.
void run_item(Job& J, int64_t bi, int64_t j0, int64_t j1) {
  const orc_desc* P = J.P;
  const int64_t K = P->k, L = P->num_groups, nd = n_out(P);
  const int64_t m0 = J.blocks[bi] * 32;
  const int64_t v = sf_vec(P);
  const int64_t w = j1 - j0;
  const int64_t b_group_bytes = P->n * row_bytes(P);

  // C columns needed for D column j; `gate` picks the gate half for SwiGLU.
  auto c_col_of = [&](int64_t j, bool gate) -> int64_t {
    if (!is_glu(P)) return j;
    // "Grouped GEMM + SwiGLU (SM100)", Step 2: block b = j/32 pairs C columns
    // [64b, 64b+32) (input X_b) and [64b+32, 64b+64) (gate G_b).  gate_first
    // swaps the two, which is the order of "Grouped GEMM + GLU + Hadamard +
    // Quant (SM100)", Equations.
    const int64_t b = j / 32, r = j % 32;
    const bool second = (gate != bool(P->gate_first));
    return 64 * b + (second ? 32 : 0) + r;
  };
  // GEMM columns behind D columns [j0, j1): twice as many for the GLUs, half as
  // many for the backward (D columns 64b..64b+63 come from GEMM columns
  // 32b..32b+31)
  const int64_t c0 = is_glu(P) ? 2 * j0 : is_bwd(P) ? j0 / 2 : j0;
  const int64_t c1 = is_glu(P) ? 2 * j1 : is_bwd(P) ? j1 / 2 : j1;

  // Group of each row ("Grouped GEMM + Quant (SM100)", Equations, Step 1).
  std::vector<int64_t> grp(32);
  for (int64_t i = 0; i < 32; ++i) grp[size_t(i)] = orc_group_of_row(J.off, L, m0 + i);

  // Step 1: C[m,n] = alpha_g * sum_k dequant(A[m,k], SFA) * dequant(B[n,k,g], SFB).
  std::vector<double> arows(size_t(32 * K), 0.0);
  std::vector<double> brow(static_cast<size_t>(K), 0.0);
  for (int64_t i = 0; i < 32; ++i)
    if (grp[size_t(i)] >= 0) dequant_row(P, J.A, J.SFA, m0 + i, P->m_pad, 0, &arows[size_t(i * K)]);
  std::vector<double> C(size_t(32 * (c1 - c0)), 0.0);
  for (int64_t n = c0; n < c1; ++n) {
    for (int64_t g = 0; g < L; ++g) {
      bool used = false;
      for (int64_t i = 0; i < 32; ++i) used = used || grp[size_t(i)] == g;
      if (!used) continue;
      dequant_row(P, J.B + g * b_group_bytes, J.SFB, n, P->n, g, brow.data());
      for (int64_t i = 0; i < 32; ++i) {
        if (grp[size_t(i)] != g) continue;
        double acc = 0.0;
        for (int64_t k = 0; k < K; ++k) acc += arows[size_t(i * K + k)] * brow[size_t(k)];
        // the backward's GEMM is scaled by alpha_g^2 ("Grouped GEMM + dGLU
        // (SM100)", Block-scaled contract, Step 1)
        const double a = double(J.alpha[g]);
        C[size_t(i * (c1 - c0) + (n - c0))] = (is_bwd(P) ? a * a : a) * acc;
      }
    }
  }
  // "Grouped GEMM + GLU + Hadamard + Quant (SM100)", Equations: + bias_g[n].
  // C (stored when asked for) is this value, before any clamp or activation.
  for (int64_t i = 0; i < 32; ++i) {
    const int64_t g = grp[size_t(i)];
    if (g < 0) continue;
    for (int64_t n = c0; n < c1; ++n) {
      double& c = C[size_t(i * (c1 - c0) + (n - c0))];
      if (J.bias) c += double(J.bias[g * P->n + n]);
      if (J.c_ref) J.c_ref[size_t((bi * 32 + i) * P->n + n)] = c;
    }
  }

  // Step 2: the epilogue, in fp64.
  std::vector<double> D(size_t(32 * w), 0.0);
  std::vector<float> amax_local(size_t(is_bwd(P) ? 2 * L : L), 0.0f);
  std::vector<double> dprob_local(32, 0.0);
  for (int64_t i = 0; i < 32; ++i) {
    const int64_t g = grp[size_t(i)];
    if (g < 0) continue;
    const int64_t m = m0 + i;
    const double p = J.prob[m];
    auto Cv = [&](int64_t n) { return C[size_t(i * (c1 - c0) + (n - c0))]; };
    // Backward ("Grouped GEMM + dGLU (SM100)", Block-scaled contract, Step 2):
    // the saved C split into the input (up) X and gate G 32-column blocks of
    // pair b (the forward's block order); dSwiGLU scales it by beta_g, dGeGLU
    // uses it as saved.  The BF16 contract scales C by beta_g for both
    // (X_g = beta_g C_g, then the gate and input of X).
    const bool scale_c = P->epi == EPI_DSWIGLU || (P->in_fmt == IN_BF16 && P->epi == EPI_DGEGLU);
    auto saved = [&](int64_t jr, bool gate) {
      const int64_t b = jr / 32, r = jr % 32;
      const bool second = (gate != bool(P->gate_first));
      const double c = J.saved_c[m * 2 * P->n + 64 * b + (second ? 32 : 0) + r];
      return scale_c ? double(J.beta[g]) * c : c;   // (reading: dSiTU-GLU unscaled too)
    };
    // dGeGLU: the gate has only an upper clamp, the up value both; the masks
    // test the values before clamping and keep the gradient at either bound
    auto dgeglu = [&](double up, double gate, double ref, double& d_up, double& d_gate, double& dprob_term) {
      const double gc = std::min(gate, P->glu_clamp_max);
      const double uc = std::min(std::max(up, P->glu_clamp_min), P->glu_clamp_max);
      const double s = orc_sigmoid(P->geglu_alpha * gc);
      const double gate_mask = gate <= P->glu_clamp_max ? 1.0 : 0.0;
      const double up_mask = (P->glu_clamp_min <= up && up <= P->glu_clamp_max) ? 1.0 : 0.0;
      d_gate = ref * p * (uc + P->linear_offset) * s * (1.0 + P->geglu_alpha * gc * (1.0 - s)) * gate_mask;
      d_up = ref * p * gc * s * up_mask;
      dprob_term = ref * gc * s * (uc + P->linear_offset);
    };
    // dSiTU-GLU: T_g = b1 tanh(G/b1) sigmoid(G), T_u = b2 tanh(U/b2); the
    // gate gradient is ref prob T_u dT_g/dG, the up gradient ref prob T_g dT_u/dU
    auto dsitu = [&](double up, double gate, double ref, double& d_up, double& d_gate, double& dprob_term) {
      const double b1 = P->situ_beta1, b2 = P->situ_beta2;
      const double th_g = std::tanh(gate / b1), th_u = std::tanh(up / b2), sg = orc_sigmoid(gate);
      const double t_g = b1 * th_g * sg, t_u = b2 * th_u;
      const double dtg = (1.0 - th_g * th_g) * sg + b1 * th_g * sg * (1.0 - sg);
      const double dtu = 1.0 - th_u * th_u;
      d_gate = ref * p * t_u * dtg;
      d_up = ref * p * t_g * dtu;
      dprob_term = ref * t_g * t_u;
    };
    if (is_bwd(P)) {
      // dprob += sum over the GEMM columns of ref times the activation
      for (int64_t jr = c0; jr < c1; ++jr) {
        const double x = saved(jr, false), gt = saved(jr, true);
        if (P->epi == EPI_DSWIGLU) {
          dprob_local[size_t(i)] += x * (gt * orc_sigmoid(gt)) * Cv(jr);
        } else if (P->epi == EPI_DSITUGLU) {
          double du, dg, t;
          dsitu(x, gt, Cv(jr), du, dg, t);
          dprob_local[size_t(i)] += t;
        } else {
          double du, dg, t;
          dgeglu(x, gt, Cv(jr), du, dg, t);
          dprob_local[size_t(i)] += t;
        }
      }
    }
    for (int64_t j = j0; j < j1; ++j) {
      double d;
      int64_t amax_idx = g;
      if (is_bwd(P)) {
        // D column j: pair b = j/64; its first or second 32-column block holds
        // the gradient of the C block at the same place (X or G)
        const int64_t b = j / 64, r = j % 32;
        const bool second = (j % 64) >= 32;
        const bool is_input = (second == bool(P->gate_first));
        const int64_t jr = 32 * b + r;
        const double x = saved(jr, false), gt = saved(jr, true), ref = Cv(jr);
        if (P->epi == EPI_DSWIGLU) {
          const double sg = orc_sigmoid(gt);
          if (is_input) d = ref * p * (gt * sg);                        // d input = ref prob swish(G)
          else d = ref * p * x * sg * (1.0 + gt * (1.0 - sg));          // d gate
        } else {
          double du, dg, t;
          if (P->epi == EPI_DSITUGLU) dsitu(x, gt, ref, du, dg, t);
          else dgeglu(x, gt, ref, du, dg, t);
          d = is_input ? du : dg;
        }
        amax_idx = 2 * g + (is_input ? 0 : 1);
      } else if (P->epi == EPI_GATE) {
        d = p * Cv(j);                                    // D = prob * ref
      } else if (is_glu(P)) {
        double x = Cv(c_col_of(j, false)), gt = Cv(c_col_of(j, true));
        if (P->glu_limit > 0.0) {                         // both halves clamped first
          x = std::min(std::max(x, -P->glu_limit), P->glu_limit);
          gt = std::min(std::max(gt, -P->glu_limit), P->glu_limit);
        }
        if (P->epi == EPI_SWIGLU) d = p * x * (gt * orc_sigmoid(gt));   // prob * X * swish(G)
        else d = p * orc_geglu(x, gt);                                  // prob * (U+1) * G * sig(1.702 G)
        d *= P->glu_alpha;                                              // gamma
      } else {
        d = p * orc_srelu(Cv(j), P->tanh_clamp_s);        // prob * relu(C)^2, clamped
      }
      D[size_t(i * w + (j - j0))] = d;
      J.d_ref[size_t((bi * 32 + i) * nd + j)] = d;
      amax_local[size_t(amax_idx)] = std::max(amax_local[size_t(amax_idx)], std::fabs(float(d)));
    }
  }

  // Colwise RHT ("Grouped GEMM + GLU + Hadamard + Quant (SM100)", Outputs and
  // Equations): for every column n and every block of 16 consecutive tokens of
  // an expert (rows of its padded range, counted from the group's start), the
  // transform of bf16-rounded D along the tokens, quantized to NVFP4 with one
  // E4M3 scale per block under rht_norm.  Expert g's data is the logical
  // (n_d, expert_m) matrix, tokens contiguous, at flat element n_d * start_g;
  // its scales the swizzled SF(n_d, expert_m) at byte n_d * start_g / 16.
  if (P->rht == 3) {
    for (int64_t ib = 0; ib < 32; ib += 16) {
      const int64_t g = grp[size_t(ib)];
      if (g < 0) continue;
      const int64_t start = g ? J.off[g - 1] : 0, em = J.off[g] - start;
      const int64_t t0 = m0 + ib - start;            // first token of the block within the expert
      for (int64_t j = j0; j < j1; ++j) {
        double x[16], y[16];
        for (int t = 0; t < 16; ++t) x[t] = orc_round_bf16(D[size_t((ib + t) * w + (j - j0))]);
        for (int r = 0; r < 16; ++r) {
          double acc = 0.0;
          for (int t = 0; t < 16; ++t) acc += orc_hadamard16(r, t) * x[t];
          y[r] = acc / 4.0;
        }
        for (int t = 0; t < 16; ++t) J.rht_ref[size_t((bi * 32 + ib + t) * nd + j)] = y[t];
        float am = 0.0f;
        for (int t = 0; t < 16; ++t) am = std::max(am, std::fabs(float(y[t])));
        const float norm = float(P->rht_norm);
        const float sf = (norm * am) * float(1.0 / 6.0);
        const uint32_t code = encode_rne_satfinite(F_E4M3, sf);
        const float sfd = float(decode(F_E4M3, code));
        const float scale = (am == 0.0f || sfd == 0.0f) ? 0.0f : norm / sfd;
        J.sfrht[nd * start / 16 + sf_offset(j, t0 / 16, 0, nd, (em + 15) / 16)] = uint8_t(code);
        for (int t = 0; t < 16; ++t) {
          const uint32_t c = encode_rne_satfinite(F_E2M1, float(y[t]) * scale);
          const int64_t e = nd * start + j * em + t0 + t;            // flat element index
          uint8_t& byte = J.rht_q[e / 2];
          if (e % 2 == 0) byte = uint8_t((byte & 0xF0) | (c & 0xF));
          else byte = uint8_t((byte & 0x0F) | ((c & 0xF) << 4));
        }
      }
    }
  }
  // Rowwise RHT of the bf16-rounded D, block by block of 16 columns.
  if (P->rht == 1 || P->rht == 2) {
    const int64_t kb16 = (nd + 15) / 16;
    for (int64_t i = 0; i < 32; ++i) {
      if (grp[size_t(i)] < 0) continue;
      const int64_t m = m0 + i;
      for (int64_t jb = j0; jb < j1; jb += 16) {
        double x[16], y[16];
        for (int t = 0; t < 16; ++t) x[t] = orc_round_bf16(D[size_t(i * w + (jb - j0) + t)]);
        for (int r = 0; r < 16; ++r) {
          double acc = 0.0;
          for (int t = 0; t < 16; ++t) acc += orc_hadamard16(r, t) * x[t];
          y[r] = acc / 4.0;
        }
        for (int t = 0; t < 16; ++t) J.rht_ref[size_t((bi * 32 + i) * nd + jb + t)] = y[t];
        if (P->rht == 2 && J.rht_q) {
          // the Step-3 quantization with E4M3 scales per 16 and q_max 6 under
          // rht_norm (SFRHT is E4M3 whatever the input scale type)
          float am = 0.0f;
          for (int t = 0; t < 16; ++t) am = std::max(am, std::fabs(float(y[t])));
          const float norm = float(P->rht_norm);
          const float sf = (norm * am) * float(1.0 / 6.0);
          const uint32_t code = encode_rne_satfinite(F_E4M3, sf);
          const float sfd = float(decode(F_E4M3, code));
          const float scale = (am == 0.0f || sfd == 0.0f) ? 0.0f : norm / sfd;
          J.sfrht[sf_offset(m, jb / 16, 0, P->m_pad, kb16)] = uint8_t(code);
          for (int t = 0; t < 16; ++t) {
            const uint32_t c = encode_rne_satfinite(F_E2M1, float(y[t]) * scale);
            uint8_t& byte = J.rht_q[m * (nd / 2) + (jb + t) / 2];
            if ((jb + t) % 2 == 0) byte = uint8_t((byte & 0xF0) | (c & 0xF));
            else byte = uint8_t((byte & 0x0F) | ((c & 0xF) << 4));
          }
        }
      }
    }
  }

  // Step 3: output quantization (row blocks and column blocks of v values).
  if (out_quantized(P)) {
    const int fmt = out_code_fmt(P);
    const int64_t kb_row = (nd + v - 1) / v;          // SFD_row is SF(m_pad, n_d)
    const int64_t kb_col = (P->m_pad + v - 1) / v;    // SFD_col is SF(n_d, m_pad)
    auto Dv = [&](int64_t i, int64_t j) { return float(D[size_t(i * w + (j - j0))]); };
    if (J.d_q) {
      for (int64_t i = 0; i < 32; ++i) {
        if (grp[size_t(i)] < 0) continue;
        const int64_t m = m0 + i;
        for (int64_t jb = j0; jb < j1; jb += v) {
          const int64_t je = std::min(jb + v, j1);
          float am = 0.0f;
          for (int64_t j = jb; j < je; ++j) am = std::max(am, std::fabs(Dv(i, j)));
          const BlockScale bs = block_scale(P, J.norm, am);
          J.sfd_row[sf_offset(m, jb / v, 0, P->m_pad, kb_row)] = uint8_t(bs.code);
          for (int64_t j = jb; j < je; ++j)
            store_code(P, J.d_q, m, j, encode_rne_satfinite(fmt, Dv(i, j) * bs.scale));
        }
      }
    }
    if (J.d_col_q && P->want_col) {
      for (int64_t ib = 0; ib < 32; ib += v) {
        bool any = false;
        for (int64_t i = ib; i < ib + v; ++i) any = any || grp[size_t(i)] >= 0;
        if (!any) continue;
        for (int64_t j = j0; j < j1; ++j) {
          float am = 0.0f;
          for (int64_t i = ib; i < ib + v; ++i)
            if (grp[size_t(i)] >= 0) am = std::max(am, std::fabs(Dv(i, j)));
          const BlockScale bs = block_scale(P, J.norm, am);
          J.sfd_col[sf_offset(j, (m0 + ib) / v, 0, nd, kb_col)] = uint8_t(bs.code);
          for (int64_t i = ib; i < ib + v; ++i)
            if (grp[size_t(i)] >= 0)
              store_code(P, J.d_col_q, m0 + i, j, encode_rne_satfinite(fmt, Dv(i, j) * bs.scale));
        }
      }
    }
  }

  std::lock_guard<std::mutex> lk(J.mu);
  for (size_t g = 0; g < amax_local.size(); ++g) J.amax[g] = std::max(J.amax[g], amax_local[g]);
  if (is_bwd(P) && J.dbias)
    for (int64_t i = 0; i < 32; ++i) {
      const int64_t g = grp[size_t(i)];
      if (g < 0) continue;
      for (int64_t j = j0; j < j1; ++j) J.dbias[g * nd + j] += D[size_t(i * w + (j - j0))];
    }
  if (is_bwd(P) && J.dprob_ref)
    for (int64_t i = 0; i < 32; ++i) J.dprob_ref[size_t(bi * 32 + i)] += dprob_local[size_t(i)];
}

}  // namespace

extern "C" int orc_run(const orc_desc* P, const uint8_t* A, const uint8_t* SFA, const uint8_t* B,
                       const uint8_t* SFB, const int32_t* padded_offsets, const float* alpha,
                       const float* prob, const float* bias, const double* saved_c, const float* beta,
                       float norm_const, const int64_t* blocks, int64_t nblocks, double* d_ref, double* c_ref,
                       double* dprob_ref, uint8_t* d_q, uint8_t* d_col_q, uint8_t* sfd_row, uint8_t* sfd_col,
                       float* amax, double* rht_ref, uint8_t* rht_q, uint8_t* sfrht, double* dbias,
                       int threads) {
  if (!P || P->m_pad <= 0 || P->m_pad % 32 || P->n <= 0 || P->k <= 0 || P->num_groups <= 0)
    return -1;
  if (is_glu(P) && P->n % 64) return -2;
  if (is_bwd(P) && (P->n % 32 || !saved_c || (P->epi == EPI_DSWIGLU && !beta) || bias)) return -4;
  if (P->in_fmt == IN_BF16 && P->epi == EPI_DGEGLU && !beta) return -4;
  if (P->rht && (is_bwd(P) || !rht_ref || (P->rht >= 2 && (!rht_q || !sfrht)))) return -5;
  // colwise: a segment's swizzled scales SF(n_d, expert_m) occupy exactly
  // n_d * expert_m / 16 bytes (the page's flat segment length) only when n_d is
  // a multiple of 128 and expert_m of 64
  if (P->rht == 3) {
    if (n_out(P) % 128) return -6;
    for (int64_t g = 0; g < P->num_groups; ++g)
      if ((padded_offsets[g] - (g ? padded_offsets[g - 1] : 0)) % 64) return -6;
  }
  if (is_fp4_in(P) && P->k % 2) return -3;
  const int64_t nd = n_out(P);
  // One work item per (block, 128-column slice of D); slices are multiples of
  // the scale-factor vector so that row blocks never straddle two items.
  const int64_t slice = 128;
  Job J;
  J.P = P; J.bias = bias; J.c_ref = c_ref; J.A = A; J.SFA = SFA; J.B = B; J.SFB = SFB; J.off = padded_offsets;
  J.saved_c = saved_c; J.beta = beta; J.dprob_ref = dprob_ref;
  J.rht_ref = rht_ref; J.rht_q = rht_q; J.sfrht = sfrht; J.dbias = dbias;
  J.alpha = alpha; J.prob = prob; J.norm = norm_const; J.blocks = blocks; J.nblocks = nblocks;
  J.d_ref = d_ref; J.d_q = d_q; J.d_col_q = d_col_q; J.sfd_row = sfd_row; J.sfd_col = sfd_col;
  J.amax.assign(size_t(is_bwd(P) ? 2 * P->num_groups : P->num_groups), 0.0f);
  const int64_t nslices = (nd + slice - 1) / slice;
  const int64_t nitems = nblocks * nslices;
  std::atomic<int64_t> next{0};
  auto worker = [&]() {
    for (;;) {
      const int64_t it = next.fetch_add(1);
      if (it >= nitems) break;
      const int64_t bi = it / nslices, s = it % nslices;
      run_item(J, bi, s * slice, std::min(nd, (s + 1) * slice));
    }
  };
  const int nt = std::max(1, threads);
  std::vector<std::thread> pool;
  for (int t = 1; t < nt; ++t) pool.emplace_back(worker);
  worker();
  for (auto& th : pool) th.join();
  if (amax)
    for (size_t g = 0; g < J.amax.size(); ++g) amax[g] = J.amax[g];
  return 0;
}
