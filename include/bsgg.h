/*
 * bsgg.h -- C ABI of the GB300 grouped block-scaled GEMM with fused epilogue.
 *
 * The operation (cuDNN-frontend documentation, "Grouped GEMM + Quant (SM100)",
 * Equations, Steps 1-3; "Grouped GEMM + SwiGLU (SM100)", Step 2; "Grouped GEMM
 * + sReLU (SM100)", Equations and Tanh soft clamp):
 *
 *   for every expert group g and every row m in [padded_offsets[g-1], padded_offsets[g]):
 *     C[m, n] = alpha[g] * sum_k dequant(A[m, k], SFA) * dequant(B[n, k, g], SFB)
 *             (+ bias_g[n] when a bias is given; C itself can be stored, before any
 *              clamp or activation: "Grouped GEMM + GLU + Hadamard + Quant (SM100)",
 *              Equations)
 *     D[m, j] = prob[m] * C[m, j]                                   (GATE)
 *             = gamma * prob[m] * X_b * swish(G_b)  over paired 32-col blocks (SWIGLU,
 *               N/2 outputs)
 *             = gamma * prob[m] * (X_b + 1) * G_b * sigmoid(1.702 G_b)  (GEGLU, N/2 outputs)
 *               with X_b, G_b first clamped to [-glu_limit, glu_limit] when a limit is set
 *             = prob[m] * relu(C)^2, or (s * min(tanh(relu(C)/s), 1))^2  (SRELU)
 *   and, for FP8/FP4 outputs, per block of v values of D along a row (SFD_row)
 *   and along a column (SFD_col, blocks of v rows):
 *     SFD = norm_const * max|D| / q_max  (rounded up to a power of two for UE8M0,
 *                                         to nearest for E4M3 scales)
 *     Dq  = convert_rne_satfinite(D * (norm_const / SFD))
 *   For 16/32-bit outputs, amax[g] = max |D| over the rows of group g.
 *
 * Everything runs in hand-written CUDA kernels for sm_103a (tcgen05 block-scaled
 * MMAs accumulating in tensor memory, TMA operand pipelines).  There is no CPU
 * path: every entry point that computes needs a CUDA device.
 *
 * Conventions shared by all entry points
 *  - Pointers in bsgg_args are DEVICE pointers (except in bsgg_run_host), owned
 *    by the caller, and must stay valid until the stream work completes.
 *  - All tensors are dense and C-contiguous, 16-byte aligned:
 *      A        (m_pad, K)      K-major, 1 byte per FP8 value, FP4 packed 2 per
 *                               byte (element 2i in the low nibble)
 *      B        (L, N, K)       K-major, same element encoding as A
 *      SFA      swizzled SF(m_pad, K)          (bsgg_sf_bytes(m_pad, K, v, 1) bytes)
 *      SFB      swizzled SF(N, K) per expert   (bsgg_sf_bytes(N, K, v, L) bytes)
 *      padded_offsets int32 (L), alpha float (L), prob float (m_pad),
 *      norm_const float (1)
 *      D, D_col (m_pad, N_out)  N-major; N_out = N/2 for SWIGLU/GEGLU, 2N for
 *                               the backward epilogues, else N;
 *                               bf16/f16/f32, or 1-byte FP8 codes, or packed FP4
 *      C        (m_pad, N)      N-major, bf16/f16, with MXFP8 inputs also f32 or
 *                               unscaled FP8/FP4 codes (optional pre-activation output)
 *      bias     (L, N)          N contiguous, bf16/f16/f32 (optional)
 *      SFD_row  swizzled SF(m_pad, N_out); SFD_col swizzled SF(N_out, m_pad)
 *      amax     float (L), 2L for the backward epilogues
 *    where SF(rows, cols) is the pages' (32, 4, ceil(rows/128), 4,
 *    ceil(ceil(cols/v)/4), L) layout in physical order (L, ceil(rows/128),
 *    ceil(ceil(cols/v)/4), 32, 4, 4) ("Grouped GEMM + SwiGLU (SM100)",
 *    Canonical layouts) and v is the scale-factor vector size (32 for MXFP8
 *    with UE8M0 scales, 16 for NVFP4 with E4M3 scales).  Output scale factors
 *    use the input's scale format and v ("Grouped GEMM + Quant (SM100)",
 *    Additional Type Constraints: SFA, SFB, SFD_row, SFD_col share a dtype).
 *  - Streams are passed as `void*` holding a cudaStream_t (NULL = legacy
 *    default stream).  bsgg_run and bsgg_pack_sf are asynchronous.
 *  - Errors are returned as bsgg_status; no entry point throws or aborts.
 *    Host-side validation mirrors the pages' "Support Surface and Constraints".
 *    Device-side values (padded_offsets) are checked by the kernel itself; a
 *    violation is reported through bsgg_query_device_status, and the kernel
 *    then writes no output.
 */
#ifndef BSGG_H
#define BSGG_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Every entry point below is exported with default visibility; the library is
 * compiled with hidden visibility otherwise, so that two builds of it (the
 * release and the range-checking one) can live in one process without sharing
 * any internal symbol. */
#if defined(__GNUC__)
#define BSGG_API __attribute__((visibility("default")))
#else
#define BSGG_API
#endif

typedef enum {
  BSGG_OK = 0,
  BSGG_ERR_INVALID_ARG = 1,     /* null/misaligned pointer, bad shape or enum */
  BSGG_ERR_UNSUPPORTED = 2,     /* valid on the pages but not built here */
  BSGG_ERR_CUDA = 3,            /* a CUDA runtime call failed */
  BSGG_ERR_DEVICE_TIMEOUT = 4,  /* a kernel wait ran out; the kernel returned early */
  BSGG_ERR_BAD_OFFSETS = 5,     /* padded_offsets not non-decreasing multiples of 128
                                   ending at m_pad; the kernel wrote nothing */
  BSGG_ERR_BAD_POINTERS = 6,    /* discrete weight mode: a b_ptrs / sfb_ptrs entry of a
                                   non-empty group is null or not 16-byte aligned; the
                                   kernel wrote nothing */
  BSGG_ERR_DEVICE_BOUNDS = 7    /* range-checking build only (libbsgg_debug.so): an index
                                   failed its range check; that access was skipped (see
                                   bsgg_debug_bounds_violation) */
} bsgg_status;

/* Input formats ("Grouped GEMM + Quant (SM100)", Data Types table). */
typedef enum {
  BSGG_IN_MXFP8_E4M3 = 0,  /* float8_e4m3fn data, float8_e8m0fnu scales, v = 32 */
  BSGG_IN_MXFP8_E5M2 = 1,  /* float8_e5m2 data,   float8_e8m0fnu scales, v = 32 */
  BSGG_IN_NVFP4 = 2,       /* float4_e2m1fn_x2 data, float8_e4m3fn scales, v = 16 */
  BSGG_IN_FP4_UE8M0_16 = 3,/* float4_e2m1fn_x2 data, float8_e8m0fnu scales, v = 16 */
  BSGG_IN_MXFP4 = 4,       /* float4_e2m1fn_x2 data, float8_e8m0fnu scales, v = 32 */
  BSGG_IN_BF16 = 5         /* bfloat16 A and B, no scale factors: the BF16 backend of
                              "Grouped GEMM + dGLU (SM100)" (Backend dispatch, BF16
                              contract).  Backward DSWIGLU / DGEGLU only (dGeGLU with
                              its fixed constants: dgeglu_custom = 0), BF16/F16/F32 D,
                              no D_col; K % 8 == 0; single CTAs and CTA pairs.  The
                              dGeGLU saved C is scaled by beta as well (X = beta C). */
} bsgg_in_format;

/* Output formats of D (and D_col). */
typedef enum {
  BSGG_OUT_BF16 = 0, BSGG_OUT_F16 = 1, BSGG_OUT_F32 = 2,
  BSGG_OUT_E4M3 = 3, BSGG_OUT_E5M2 = 4, BSGG_OUT_E2M1 = 5
} bsgg_out_format;

/* Epilogues: gating ("Grouped GEMM + Quant (SM100)", Step 2), SwiGLU ("Grouped GEMM +
 * SwiGLU (SM100)", Step 2), squared ReLU with optional tanh soft clamp ("Grouped GEMM +
 * sReLU (SM100)"), GeGLU ("Grouped GEMM + GLU + Hadamard + Quant (SM100)", Equations),
 * and the dSwiGLU backward ("Grouped GEMM + dGLU (SM100)", Block-scaled contract):
 *   ref = alpha_g^2 * sum_k A B;  X, G = beta_g * the saved forward C's input and gate
 *   32-column blocks;  D = [ref*prob*swish(G) | ref*prob*X*sigmoid(G)*(1 + G*(1 - sigmoid(G)))]
 *   in C's block order (width 2N);  dprob[m] += sum_n X*swish(G)*ref. */
typedef enum {
  BSGG_EPI_GATE = 0, BSGG_EPI_SWIGLU = 1, BSGG_EPI_SRELU = 2, BSGG_EPI_GEGLU = 3, BSGG_EPI_DSWIGLU = 4,
  BSGG_EPI_DGEGLU = 5,  /* dGeGLU backward (same page): the saved C unscaled (beta not read),
                           gate G clamped above at clamp_max, up U clamped to [clamp_min,
                           clamp_max]; s = sigmoid(a * Gc);
                           d gate = ref*prob*(Uc + offset)*s*(1 + a*Gc*(1 - s)) if G <= clamp_max,
                           d up = ref*prob*Gc*s if clamp_min <= U <= clamp_max, else 0;
                           dprob[m] += sum_n ref*Gc*s*(Uc + offset) */
  BSGG_EPI_DSITUGLU = 6 /* dSiTU-GLU backward (same page, Equations): the saved C unscaled;
                           T_g = b1*tanh(G/b1)*sigmoid(G), T_u = b2*tanh(U/b2);
                           d gate = ref*prob*T_u*dT_g/dG, d up = ref*prob*T_g*dT_u/dU;
                           dprob[m] += sum_n ref*T_g*T_u */
} bsgg_epilogue;

/* Problem description, fixed at plan creation (the pages' constructor +
 * check_support + compile, "Grouped GEMM + Quant (SM100)", Class API). */
typedef struct {
  int64_t m_pad;          /* rows of A/D/prob = padded_offsets[L-1]; a positive multiple
                             of 128 (a batch whose groups are all empty, m_pad = 0, is
                             refused with BSGG_ERR_INVALID_ARG: the caller skips the call,
                             and every amax of such a batch is 0) */
  int64_t n;              /* GEMM N (rows of each expert's B); multiple of 32 (64 for SWIGLU
                             and GEGLU); for DSWIGLU the compact gradient width (D is 2N wide) */
  int64_t k;              /* reduction length in elements; multiple of 16 (FP8) / 32 (FP4) */
  int32_t num_groups;     /* L, 1..1024 */
  int32_t in_format;      /* bsgg_in_format */
  int32_t out_format;     /* bsgg_out_format */
  int32_t epilogue;       /* bsgg_epilogue */
  int32_t want_col;       /* 1: also write D_col and SFD_col (quantized outputs only) */
  int32_t gate_first;     /* SWIGLU/GEGLU block order: 0 = [X_b | G_b] ("Grouped GEMM +
                             SwiGLU (SM100)", Step 2), 1 = [G_b | U_b] ("Grouped GEMM + GLU +
                             Hadamard + Quant (SM100)", Equations) */
  float tanh_clamp_s;     /* SRELU soft clamp s > 0, or 0 for none */
  int32_t tile_m;         /* rows per MMA tile: 128 (one CTA) or 256 (a pair of CTAs with
                             2-CTA instructions); 0 = library choice.  The pages' mma_tiler_mn[0]
                             ("Grouped GEMM + Quant (SM100)", Common Parameters) */
  int32_t tile_n;         /* columns per MMA tile: 128 or 256 (256 when tile_m = 256); 0 = library
                             choice.  The pages' mma_tiler_mn[1] */
  /* Thread-block cluster shape (cluster_m, cluster_n): the pages' cluster_shape_mn
     ("Grouped GEMM + Quant (SM100)", Common Parameters; Support Surface and Constraints,
     Tiling and Cluster).  Built: (1, 1) with tile_m = 128; (2, 1) with tile 256 x 256 (the
     CTA pair; tile (0, 0) with cluster (2, 1) selects it).  (0, 0) = the library's choice.
     A (2, 1) cluster of 128-row or 128-column tiles would share an operand tile between two
     CTAs by TMA multicast, which this library never issues: it returns
     BSGG_ERR_UNSUPPORTED, as do the other powers of two up to 4 that the pages allow; any
     other value returns BSGG_ERR_INVALID_ARG. */
  int32_t cluster_m;
  int32_t cluster_n;
  /* Forward epilogue options of "Grouped GEMM + GLU + Hadamard + Quant (SM100)"
     (Equations; Configuration).  All zero = none of them. */
  float glu_limit;        /* SWIGLU/GEGLU: both halves clamped to [-glu_limit, glu_limit]
                             before the activation; 0 = no clamp; must be finite, >= 0 */
  float glu_alpha;        /* SWIGLU/GEGLU: output scale gamma; 0 (unset) or 1 = none; finite */
  int32_t want_c;         /* 1: also store C = alpha_g * acc (+ bias), before any clamp or
                             activation, (m_pad, N) N-major, in c_format */
  int32_t c_format;       /* BSGG_OUT_BF16 or BSGG_OUT_F16 (when want_c); with MXFP8 inputs
                             also BSGG_OUT_F32, or BSGG_OUT_E4M3 / E5M2 / E2M1: C converted
                             with round-to-nearest-even and saturation, no scale factor */
  int32_t want_bias;      /* 1: add bias_g[n] to C; bias is (L, N), N contiguous per expert
                             (the pages' (N, L) tensor with stride (1, N)) */
  int32_t bias_format;    /* BSGG_OUT_BF16, BSGG_OUT_F16 or BSGG_OUT_F32 (when want_bias) */
  /* Discrete weight mode ("Grouped GEMM + GLU + Hadamard + Quant (SM100)", Discrete weight
     mode): 1 = each expert's B and SFB are separate allocations named by the device
     pointer arrays b_ptrs / sfb_ptrs instead of the dense b / sfb tensors (the two
     modes are mutually exclusive).  B_g is (N, K) K-major, SFB_g is SF(N, K) with one
     slice (bsgg_sf_bytes(N, K, v, 1) bytes).  The plan then owns 256 * L + 256 bytes
     of device memory for one TMA descriptor pair per expert, written by a small
     kernel on the stream before every launch. */
  int32_t discrete_b;
  /* DSWIGLU: storage type of the saved forward C, BSGG_OUT_BF16, BSGG_OUT_F16 or
     BSGG_OUT_F32 ("Grouped GEMM + dGLU (SM100)", BF16 contract: C in BF16/FP16/FP32). */
  int32_t saved_c_format;
  /* Hadamard output ("Grouped GEMM + GLU + Hadamard + Quant (SM100)", Outputs and
     Equations), forward epilogues only; H16 is the 16 x 16 Sylvester Hadamard matrix.
     1 = rowwise: RHT = (H16 / 4) x for every 16-column block x of bf16-rounded D;
         (m_pad, N_out) N-major in rht_format: BSGG_OUT_BF16, or BSGG_OUT_E2M1 (packed
         NVFP4 with E4M3 scales per 16 in SFRHT = swizzled SF(m_pad, N_out) under
         rht_norm_const, whatever the input's scale type).
     2 = colwise (rht_format BSGG_OUT_E2M1, N_out % 128 == 0): (H16 / 4) x for every
         column and every block x of 16 consecutive tokens of an expert (rows of its
         padded range, counted from its start), NVFP4 with one E4M3 scale per block;
         expert g (padded rows [start_g, end_g), expert_m = end_g - start_g) is the
         logical (N_out, expert_m) matrix, tokens contiguous, from flat element
         N_out * start_g of RHT (m_pad * N_out / 2 bytes in all), its scales the
         swizzled SF(N_out, expert_m) from byte N_out * start_g / 16 of SFRHT
         (m_pad * N_out / 16 bytes in all). */
  int32_t want_rht;
  int32_t rht_format;
  /* DGEGLU: 0 = the page's defaults (geglu_alpha 1.702, clamp [-7, 7], linear_offset 1),
     1 = the four values below (finite, clamp_min <= clamp_max). */
  int32_t dgeglu_custom;
  float dgeglu_alpha;
  float dgeglu_clamp_min;
  float dgeglu_clamp_max;
  float dgeglu_linear_offset;
  /* DSITUGLU: the tanh scales b1 (gate) and b2 (up), finite and > 0; 0 = 1. */
  float situ_beta1;
  float situ_beta2;
} bsgg_desc;

/* Tensors of one call.  Unused outputs may be NULL: d_col/sfd_col unless
 * want_col; sfd_row/sfd_col/norm_const for 16/32-bit outputs; amax for
 * quantized outputs; bias unless want_bias; c unless want_c.  amax is
 * required for BF16/F16 outputs and optional for F32 ("Grouped GEMM + Quant
 * (SM100)", Scale Factor Output Requirements); with BSGG_IN_BF16 inputs it is
 * optional, and sfa, sfb and sfb_ptrs are not read (NULL). */
typedef struct {
  const void* a;
  const void* sfa;
  const void* b;
  const void* sfb;
  const int32_t* padded_offsets;
  const float* alpha;
  const float* prob;         /* required: pass ones for no gating */
  const float* norm_const;   /* required for quantized outputs */
  void* d;
  void* d_col;
  void* sfd_row;
  void* sfd_col;
  float* amax;               /* zeroed by bsgg_run on the stream before the kernel */
  const void* bias;          /* (L, N) in bias_format; required iff want_bias */
  void* c;                   /* (m_pad, N) in c_format; required iff want_c */
  /* discrete_b only (b and sfb then NULL): device arrays of L int64 device
     addresses.  Entries of empty groups are not read by the GEMM and may be 0;
     the others must be 16-byte aligned (checked on the device: a violation is
     BSGG_ERR_BAD_POINTERS from bsgg_query_device_status, and nothing is written). */
  const int64_t* b_ptrs;
  const int64_t* sfb_ptrs;
  /* DSWIGLU, DGEGLU and DSITUGLU: the saved forward C (m_pad, 2N) N-major in saved_c_format,
     its per-group scale beta (L; DSWIGLU, and DGEGLU with BSGG_IN_BF16), and dprob
     (m_pad), which the kernel
     ACCUMULATES into:
     zero it before the call ("Grouped GEMM + dGLU (SM100)": dprob must be
     zero-initialized).  amax then holds 2L floats: [2g] over the input-gradient
     blocks, [2g + 1] over the gate-gradient blocks of group g. */
  const void* saved_c;
  const float* beta;
  float* dprob;
  /* want_rht only: the RHT output; SFRHT and rht_norm_const (1 float) for an
     NVFP4 RHT. */
  void* rht;
  void* sfrht;
  const float* rht_norm_const;
  /* Backward epilogues, optional: dbias (L, 2N) float, ACCUMULATED like dprob
     (zero it before the call): dbias[g][n] += sum over the rows of group g of
     D[m][n] before any output conversion ("Grouped GEMM + dGLU (SM100)": the
     per-expert row reduction of the interleaved D).  NULL = not computed. */
  float* dbias;
} bsgg_args;

typedef struct bsgg_plan bsgg_plan;

/* Validate `desc` and build a plan (kernel choice, launch shape, a 16-byte
 * device status word).  The plan belongs to the device that is current at
 * creation.  Returns BSGG_ERR_INVALID_ARG / BSGG_ERR_UNSUPPORTED for
 * descriptions the pages or this library reject; *plan is NULL then. */
BSGG_API bsgg_status bsgg_create(const bsgg_desc* desc, bsgg_plan** plan);

/* Enqueue one grouped GEMM on `stream` (asynchronous, no host sync, graph
 * capturable).  Checks pointers for presence and 16-byte alignment. */
BSGG_API bsgg_status bsgg_run(bsgg_plan* plan, const bsgg_args* args, void* stream);

/* End-to-end call with HOST buffers: `host` holds host pointers (pinned for
 * speed) for every input and output to move; `dev` holds device buffers of the
 * same shapes.  Inputs present in `host` are copied into `dev`, the kernel runs
 * on the `dev` buffers, outputs present in `host` are copied back, and the
 * stream is synchronized.  An input left NULL in `host` is taken as already
 * resident in `dev`.  Bytes moved are returned in *h2d_bytes / *d2h_bytes
 * (either may be NULL).  Allocates nothing.  In discrete weight mode the
 * experts' weights are taken as resident (dev->b_ptrs / dev->sfb_ptrs; host->b
 * and host->sfb must be NULL). */
BSGG_API bsgg_status bsgg_run_host(bsgg_plan* plan, const bsgg_args* host, const bsgg_args* dev,
                          void* stream, uint64_t* h2d_bytes, uint64_t* d2h_bytes);

/* bsgg_run_host without the final synchronization (the pages have no
 * counterpart): the copies in, the kernel and the copies out are enqueued on
 * `stream` and the call returns.  The host buffers (pinned, or the copies are
 * synchronous on the host side) and the device buffers must stay valid, and
 * the outputs in `host` are complete only once the stream's work has
 * finished.  Lets a caller keep several batches in flight on several streams,
 * so that one batch's outputs travel to the host while the next batch's
 * inputs travel to the device and its kernel runs; each stream in flight
 * needs its own `dev` buffers, its own output buffers in `host` and its own
 * plan (the status word is per plan).  Same arguments, byte counts and errors
 * as bsgg_run_host. */
BSGG_API bsgg_status bsgg_run_host_async(bsgg_plan* plan, const bsgg_args* host, const bsgg_args* dev,
                                void* stream, uint64_t* h2d_bytes, uint64_t* d2h_bytes);

/* Number of kernel launches one bsgg_run of this plan enqueues (the pages have
 * no counterpart): 1, or 2 in discrete weight mode (the per-expert descriptor
 * kernel, then the GEMM).  -1 for a null plan. */
BSGG_API int32_t bsgg_launches_per_run(const bsgg_plan* plan);

/* Synchronize `stream`, then read and clear the plan's device status word:
 * BSGG_OK, BSGG_ERR_DEVICE_TIMEOUT, BSGG_ERR_BAD_OFFSETS or BSGG_ERR_BAD_POINTERS
 * (a status bit the library does not define reads as BSGG_ERR_CUDA). */
BSGG_API bsgg_status bsgg_query_device_status(bsgg_plan* plan, void* stream);

/* Test hook for the failure path; the pages have no counterpart.  With enable =
 * 1, every later bsgg_run / bsgg_run_host of this plan launches a kernel whose
 * MMA thread first waits on a barrier that nothing completes, with every
 * barrier wait bounded by 50 ms instead of 2 s: each role gives up, drains its
 * in-flight work and returns, no output is complete, and the status word reads
 * BSGG_ERR_DEVICE_TIMEOUT; the CUDA context stays usable.  enable = 0 restores
 * normal launches.  Errors: BSGG_ERR_INVALID_ARG (null plan, enable not 0/1). */
BSGG_API bsgg_status bsgg_debug_force_timeout(bsgg_plan* plan, int32_t enable);

BSGG_API void bsgg_destroy(bsgg_plan* plan);
BSGG_API const char* bsgg_status_string(bsgg_status status);

/* Bytes of the swizzled SF(rows, cols) layout with L slices and vector v:
 * 512 * L * ceil(rows/128) * ceil(ceil(cols/v)/4). */
BSGG_API uint64_t bsgg_sf_bytes(int64_t rows, int64_t cols, int32_t sf_vec, int32_t num_slices);

/* Byte offset of the scale of (row, k-block, slice l) in that layout, where
 * kblocks = ceil(cols/v).  Pure host function. */
BSGG_API int64_t bsgg_sf_offset(int64_t row, int64_t kblk, int64_t l, int64_t rows, int64_t kblocks);

/* Pack row-major scale codes (L, rows, kblocks) into the swizzled layout,
 * writing every byte (padding = 0, "Grouped GEMM + SwiGLU (SM100)", JAX
 * execution: untouched SF padding is zero).  Device pointers; asynchronous. */
BSGG_API bsgg_status bsgg_pack_sf(const uint8_t* rowmajor, uint8_t* swizzled, int64_t rows,
                         int64_t kblocks, int32_t num_slices, void* stream);

/* Size of the library-owned device scratch used by bsgg_run_noalloc. */
#define BSGG_NOALLOC_SCRATCH_BYTES 256

/* Allocation-free run (the pages have no counterpart; this is a library
 * convenience).  Same computation, arguments and validation as bsgg_create +
 * bsgg_run + bsgg_destroy, but it creates no plan and never calls cudaMalloc
 * or cudaFree.  It is for callers that cannot allocate device memory at the
 * point of the call: a framework whose own pool has already reserved the
 * device memory (a raw cudaMalloc would fail or fragment it), a serving loop
 * that must not let cudaMalloc/cudaFree synchronize the device, or a plug-in
 * inside a host application that owns memory management.
 *
 * The kernel's only scratch, its device status word (16 bytes with the record a
 * range-checking build keeps behind it), lives in a file-scope static device
 * array of BSGG_NOALLOC_SCRATCH_BYTES bytes that every GPU which loads the
 * library holds until the process exits.  A call whose scratch need exceeds
 * that array is rejected with BSGG_ERR_UNSUPPORTED: the need is those 16 bytes,
 * except in discrete weight mode, whose per-expert descriptors (256 * L + 256
 * bytes) never fit, so discrete_b = 1 is rejected.
 *
 * The first call on a device looks up the array's device address with that
 * device current (cudaGetSymbolAddress) and remembers it with the id of the
 * device's context; a call that finds a different context (after
 * cudaDeviceReset, say) looks it up again.  Make the first call on a device,
 * and the first after a reset, before any stream capture.  Every call clears
 * the 16 status bytes on `stream` before its kernel.  All calls share the array, which keeps the last call's contents:
 * calls whose kernels overlap on the GPU (several streams, several host
 * threads) race on it, so run them on one stream when the status matters.
 * With wait_status != 0 the call synchronizes `stream` after the launch and
 * returns the device status as bsgg_query_device_status would (BSGG_OK,
 * BSGG_ERR_DEVICE_TIMEOUT or BSGG_ERR_BAD_OFFSETS; a status bit the library
 * does not define reads as BSGG_ERR_CUDA); with 0 it returns once the kernel
 * is enqueued. */
BSGG_API bsgg_status bsgg_run_noalloc(const bsgg_desc* desc, const bsgg_args* args, void* stream,
                             int32_t wait_status);

/* Range-checking build; the pages have no counterpart.  The library is also
 * built as libbsgg_debug.so with every TMA box origin (A rows, K offset, B row
 * and slice, scale-factor atoms), every output index (D and D_col rows and
 * columns, SFD_row / SFD_col offsets, C, the Hadamard output, dbias) and every
 * per-row / per-group read (prob, alpha) checked against the problem's extents
 * before use.  A failed check skips the access, records the first failure and
 * raises a status bit that bsgg_query_device_status returns as
 * BSGG_ERR_DEVICE_BOUNDS; a failure in the operand loads also makes every role
 * of the CTA give up and drain as after a timeout.  No trap, no fault.  The
 * release build compiles the checks away.
 *
 * bsgg_debug_bounds_checked: 1 in the range-checking build, 0 otherwise.
 * bsgg_debug_bounds_margin: test hook: later launches of the plan check rows
 *   against m_pad - rows instead of m_pad (rows: a multiple of 128 below m_pad),
 *   so that in-range accesses fail their checks without any out-of-range access
 *   being made; barrier waits are then bounded by 50 ms.  0 restores the checks.
 *   BSGG_ERR_UNSUPPORTED in the release build; BSGG_ERR_INVALID_ARG for other rows.
 * bsgg_debug_bounds_violation: the failure recorded by the last
 *   bsgg_query_device_status that returned BSGG_ERR_DEVICE_BOUNDS (site code,
 *   value, limit; all 0 if none).  Site codes: 1 A rows, 2 B n-tile, 3 B slice,
 *   4 SFA atom, 5 SFB row block, 6 K offset, 10 D row, 11 D column, 12 SFD_row,
 *   13 SFD_col, 15 C column, 16 Hadamard output, 18 dbias column, 19 group. */
BSGG_API int32_t bsgg_debug_bounds_checked(void);
BSGG_API bsgg_status bsgg_debug_bounds_margin(bsgg_plan* plan, int32_t rows);
BSGG_API bsgg_status bsgg_debug_bounds_violation(const bsgg_plan* plan, uint32_t* site, uint32_t* value, uint32_t* limit);

/* Measurement utility; the pages have no counterpart.  Measures the dense
 * block-scaled tensor-core throughput of the current device, the denominator of
 * the kernel's roofline: one CTA per SM issues `mmas_per_sm` tcgen05.mma
 * block_scale instructions (M = 128, N = tile_n, K = 32 for MXFP8 or 64 for
 * NVFP4) on operands and unit scales resident in shared memory, with no loads and
 * no epilogue, timed with CUDA events on `stream`.  Synchronizes the stream.
 * in_format: a bsgg_in_format; tile_n: 128 or 256; mmas_per_sm: 4 .. 2^22.
 * Writes TFLOP/s (2*M*N*K per instruction) to *tflops.  Allocates and frees a
 * 4-byte status word.  Errors: BSGG_ERR_INVALID_ARG for other arguments,
 * BSGG_ERR_CUDA for a failed CUDA call, BSGG_ERR_DEVICE_TIMEOUT if the final
 * wait ran out (2 s). */
BSGG_API bsgg_status bsgg_measure_mma_peak(int32_t in_format, int32_t tile_n, int64_t mmas_per_sm, double* tflops,
                                  void* stream);

/* Measurement utility; the pages have no counterpart.  The same measurement for
 * either instruction form the GEMM issues: tile_m = 128 is bsgg_measure_mma_peak
 * (cta_group::1, M = 128, one issuing CTA per SM, tile_n 128 or 256); tile_m = 256
 * is cta_group::2 with M = 256, N = 256 (tile_n must be 256): clusters of two
 * CTAs, each holding its 128 rows of A and half of B's rows, the even CTA issuing
 * `mmas` instructions for the pair, on floor(SMs / 2) pairs.  Each CTA reserves
 * 120 KB of shared memory so that every SM holds one.  TFLOP/s counts 2*M*N*K per
 * instruction.  Synchronizes the stream; allocates and frees a 4-byte status
 * word.  Errors: BSGG_ERR_INVALID_ARG for tile_m not 128 or 256 and the
 * arguments bsgg_measure_mma_peak refuses (mmas: 4 .. 2^22 per issuing thread),
 * BSGG_ERR_UNSUPPORTED for tile_m = 256 with tile_n = 128, BSGG_ERR_CUDA for a
 * failed CUDA call, BSGG_ERR_DEVICE_TIMEOUT if the final wait ran out (2 s). */
BSGG_API bsgg_status bsgg_measure_mma_peak_tile(int32_t in_format, int32_t tile_m, int32_t tile_n, int64_t mmas,
                                       double* tflops, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* BSGG_H */
