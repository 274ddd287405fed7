/*
 * fsa.h -- C ABI of libfsa: MX block-scaled attention forward with a
 * reformulated softmax, for NVIDIA GB300 (sm_103a).
 *
 * Sources (by page title and section):
 *   "Fused-Softmax for efficient quantized attention" (The Singularity Report),
 *       abstract: QK^T and PV as MXFP8/MXFP6/MXFP4 GEMMs; softmax reformulated
 *       and approximated so its dominant work folds into the GEMMs; BF16
 *       attention as the comparison point.
 *   "Moving softmax to matrix operations speeds up AI inference by over 2x"
 *       (zot.news), summary, "Read it as" and the "How it works" figure: max
 *       subtraction and exponentiation folded into the score GEMM; the row
 *       maximum frozen speculatively with a fallback; a fast exponential;
 *       "Exp + MX Quant" fused; probabilities summed on the matrix unit.
 *   "EFQ-Softmax: Exp-Free Quantization for Softmax" (paper-with-me),
 *       abstract: per 32-element block an exponent-only scale from the local
 *       maximum and nonnegative E2M1 probability codes from one affine rule;
 *       the same operand feeds the P~V numerator and the P~1 denominator;
 *       final normalisation in high precision.
 *
 * Conventions for every entry point:
 *   - All tensor pointers are DEVICE pointers, allocated and owned by the
 *     caller; the library keeps no reference after the call returns.  The
 *     library allocates no device memory on any entry point below.
 *   - `stream` is a cudaStream_t passed as void*; NULL means the legacy
 *     default stream.  Work is enqueued asynchronously; no entry point
 *     synchronises.
 *   - Return value: FSA_OK (0) or a negative FSA_ERR_* code.  Argument errors
 *     are detected on the host before any launch; nothing is enqueued then.
 *   - Shapes: B batch, H query heads, Hkv key/value heads (H % Hkv == 0; query
 *     head h reads kv head h / (H/Hkv)), Sq queries, Sk keys, head dim D in
 *     {64, 128}; the attention calls also need B*H <= 65535, Sq <= 65535*128
 *     and Sk <= 2^20 (else INVALID_ARG).  The key limit is one of accuracy: the
 *     fp32 accumulator in tensor memory, to which every key tile adds its
 *     products, drifts by a per-row factor that grows with the number of key
 *     tiles, as adds that drop low-order bits would (measured at 2^20 keys:
 *     below 5e-4 of the output, within the 2e-3 parity bound; at 2^22 keys up
 *     to 7e-3 with 8-bit P~).
 *     Causal masking is bottom-right aligned: key j is visible to
 *     query i iff j <= i + Sk - Sq.  A query with no visible key gets a zero
 *     output row.
 */
#ifndef FSA_H
#define FSA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---------------------------------------------------------------- status */
#define FSA_OK                   0
#define FSA_ERR_INVALID_ARG     -1  /* null pointer, bad shape, misaligned pointer */
#define FSA_ERR_UNSUPPORTED_FMT -2  /* e.g. E2M1_EFQ as a QK^T operand format */
#define FSA_ERR_LAUNCH          -3  /* CUDA runtime/driver error at launch */
#define FSA_ERR_TIMEOUT         -4  /* a bounded on-chip wait gave up (reported via fsa_stats) */
#define FSA_ERR_NO_DEVICE       -5  /* no sm_100-family device with tcgen05 */

/* ------------------------------------------------------- element formats */
/* OCP MX element types; E2M1_EFQ is the E2M1 operand produced by the EFQ
 * direct-code rule and is valid only as the PV format. */
typedef enum {
  FSA_FMT_E4M3 = 0,      /* MXFP8 */
  FSA_FMT_E2M3 = 1,      /* MXFP6 */
  FSA_FMT_E2M1 = 2,      /* MXFP4, P by exp then round-to-nearest-even */
  FSA_FMT_E2M1_EFQ = 3,  /* MXFP4, P by the EFQ affine rule (fmt_pv only) */
  FSA_FMT_E3M2 = 4,      /* MXFP6, the OCP MX E3M2 element type (bias 3, max 28) */
  FSA_FMT_NVFP4 = 5      /* NVFP4: E2M1 codes with one E4M3 scale per 16 elements
                          * (FSA_MX_ROWS only, i.e. Q and K, fmt_qk only); an
                          * operand format adjacent to the MX ones the
                          * Fused-Softmax brief names (abstract), from NVIDIA's
                          * public FP4 definition without its per-tensor scale */
} fsa_fmt;

/* ------------------------------------------------------------ MX tensors */
/* An MX tensor holds element codes plus one E8M0 scale byte (2^(byte-127))
 * per 32 consecutive elements along the contraction dimension.
 *
 * FSA_MX_ROWS (Q and K; blocks along D).  Source x[B][H][S][D] bf16.
 *   codes : [B*H][S][row_bytes], row_bytes = D (E4M3, E2M3, E3M2) or D/2
 *           (E2M1).  E4M3: one byte per element.  E2M3 and E3M2: each group of
 *           16 elements is 12 bytes of 6-bit codes packed least-significant-bit
 *           first, followed by 4 zero bytes.  E2M1: two elements per byte, the
 *           even element in the low nibble.
 *   scales: [B*H][ceil(S/128)][512] bytes: for row r of a 128-row tile and
 *           block b (b < D/32), byte (r%32)*16 + (r/32)*4 + b.  Slots with no
 *           data (rows >= S, blocks >= D/32) hold 0x7F.
 * FSA_MX_COLS_T (V; blocks along S, stored transposed, K-major for PV).
 *   codes : [B*H][D][Sp] elements, Sp = S rounded up to 128, packed as above
 *           along the key axis; codes of keys >= S are 0.
 *   scales: [B*H][Sp/128][512] bytes: for d (row of V^T) and key block b of
 *           a 128-key tile, byte (d%32)*16 + (d/32)*4 + b.  Rows d >= D hold
 *           0x7F; blocks of keys wholly >= S hold 0x7F.
 * The block scale is E = clamp(floor(log2 amax) - emax, -127, 127) (emax 8
 * for E4M3, 4 for E3M2, 2 for E2M3/E2M1), codes = round-to-nearest-even, saturating, of
 * x * 2^-E; a block with a non-finite element gets scale 0xFF.
 * FSA_FMT_NVFP4 (FSA_MX_ROWS only): codes as E2M1 above; one E4M3 scale byte
 *   per 16 elements along D: the E4M3 value nearest amax/6 (ties to even,
 *   saturating at 448), codes the E2M1 values nearest x/scale (saturating at 6;
 *   a zero scale gives zero codes; a non-finite block gets scale 0x7F, the
 *   E4M3 NaN, and zero codes).  scales: [B*H][ceil(S/128)][D/64][512] bytes:
 *   for row r of a 128-row tile and 16-element block b (b < D/16), byte
 *   (b/4)*512 + (r%32)*16 + (r/32)*4 + b%4; rows >= S hold 0x38 (1.0).   */
typedef enum { FSA_MX_ROWS = 0, FSA_MX_COLS_T = 1 } fsa_mx_layout;

typedef struct {
  void*    codes;    /* device, 16-byte aligned */
  uint8_t* scales;   /* device, 16-byte aligned */
  int32_t  fmt;      /* fsa_fmt of the codes (E4M3, E2M3, E2M1, E3M2 or NVFP4) */
  int32_t  layout;   /* fsa_mx_layout */
  int32_t  B, H, S, D;
} fsa_mx_tensor;

/* Bytes of the codes and scales buffers for an MX tensor. */
int fsa_mx_sizes(int B, int H, int S, int D, int layout, int fmt, size_t* codes_bytes, size_t* scales_bytes);

/* Quantise x_bf16 [B][H][S][D] (device, 16-byte aligned) into out->codes /
 * out->scales with the given layout and element format.  The shape, layout
 * and format fields of *out are written by the call.  One kernel launch on
 * `stream`, which writes every byte of both buffers; nothing is allocated and
 * nothing synchronises, so the call may be captured in a CUDA graph.  Cited:
 * MXFP8/6/4 GEMM operands ("Fused-Softmax for efficient quantized
 * attention", abstract). */
int fsa_mx_quantize(const void* x_bf16, int B, int H, int S, int D, int layout, int fmt,
                    fsa_mx_tensor* out, void* stream);

/* The operands of one attention call in one kernel launch: q [B][H][Sq][D]
 * and k [B][Hkv][Sk][D] into FSA_MX_ROWS tensors of format fmt_qk, v
 * [B][Hkv][Sk][D] into an FSA_MX_COLS_T tensor of format fmt_v (E2M1 for an
 * EFQ P~ V product).  Codes and scales are identical to three
 * fsa_mx_quantize calls; argument checks, field writes and launch behaviour
 * are the same as there.  Errors: FSA_ERR_INVALID_ARG (null or misaligned
 * pointer, bad shape), FSA_ERR_UNSUPPORTED_FMT (E2M1_EFQ as a storage
 * format), FSA_ERR_LAUNCH. */
int fsa_mx_quantize_qkv(const void* q_bf16, const void* k_bf16, const void* v_bf16, int B, int H, int Hkv,
                        int Sq, int Sk, int D, int fmt_qk, int fmt_v, fsa_mx_tensor* q_out,
                        fsa_mx_tensor* k_out, fsa_mx_tensor* v_out, void* stream);

/* ------------------------------------------------------ options and stats */
typedef enum {
  FSA_EXP_POLY = 0,   /* cubic interpolant of 2^f on the FMA pipe for every element */
  FSA_EXP_MUFU = 1,   /* hardware ex2.approx for every element */
  FSA_EXP_SPLIT = 2   /* key positions 4k+3 (of each 32-key block) the cubic, the others ex2.approx */
} fsa_exp_mode;

typedef enum {
  FSA_OUT_F32 = 0,    /* O as fp32 */
  FSA_OUT_BF16 = 1    /* O as bf16: the fp32 result rounded to nearest even */
} fsa_out_dtype;

/* Debug dumps of every key tile the kernel processes (a test instrument: the
 * P~ codes are the method's product, and the EFQ-Softmax page, abstract, defines
 * them as nonnegative E2M1 codes under exponent-only block scales).  All
 * pointers are device memory of the caller.  Query row r (r = (b*H + h)*Sq + i)
 * is dumped to slot row_slot[r] (row_slot NULL: slot r; a negative slot: not
 * dumped); N is the number of slots, NKT = ceil(Sk/128) key tiles.  Entries of
 * tiles a query tile does not process are left untouched (callers initialise
 * them).  The debug instance computes the same outputs as the production kernel,
 * bit for bit.
 *   s        : float    [N][NKT*128]  raw fp32 scores of the MMA (masked keys -inf)
 *   m        : float    [N][NKT]      frozen maximum M used for the tile's P~
 *   p        : uint32_t [N][NKT][32]  P~ code words as written to tensor memory:
 *                                     one byte per code (E4M3; E2M3 in the low 6
 *                                     bits) in words 0..31, or two E2M1 codes per
 *                                     byte (even key in the low nibble) in words 0..15
 *   p_scales : uint32_t [N][NKT]      byte b = E8M0 scale of the tile's 32-key block b
 *   row_slot : int32_t  [B*H*Sq]      optional slot of each query row */
typedef struct {
  float*    s;
  float*    m;
  uint32_t* p;
  uint32_t* p_scales;
  const int32_t* row_slot;
} fsa_debug_dump;

/* The EFQ direct-code rule (EFQ-Softmax page, abstract: an exponent-only block
 * scale from the local maximum, shifted scores in a normalised residual domain,
 * codes by a single affine rule; the page prints no constants).  Per 32-key block
 * with maximum shifted score tmax (log2 units):
 *     E    = clamp(floor(tmax + efq_phi) - 2, -127, 127)
 *     code = clamp(rne(efq_a * (t - E) + efq_b), 0, 7)
 * computed as one fused multiply-add per raw score s (t - E = s*c - (M + E)).
 * The defaults come from a scan of the rule family against fp64 exact attention
 * on the long-context workload (the error-floor criterion of the Fused-Softmax
 * brief, abstract). */
#define FSA_EFQ_A_DEFAULT   1.6875f
#define FSA_EFQ_B_DEFAULT   3.4375f
#define FSA_EFQ_PHI_DEFAULT 0.625f

typedef struct {
  float    delta;        /* fallback margin in log2 units, >= 0 (default 8): a later tile falls
                            back only when its maximum exceeds the frozen one by more than
                            delta; per-block scales make a stale maximum cost no precision.
                            0 is the literal test "any score exceeds the frozen maximum" */
  int32_t  exp_mode;     /* fsa_exp_mode (default FSA_EXP_MUFU: on sm_103a the hardware exp2
                            issues at twice the rate of earlier parts, and the cubic's
                            extra FMA-pipe instructions cost more than they save) */
  float    efq_a;        /* EFQ slope a (default FSA_EFQ_A_DEFAULT), finite, 0 < a <= 16 */
  float    efq_b;        /* EFQ offset b (default FSA_EFQ_B_DEFAULT), finite, |b| <= 64 */
  float    efq_phi;      /* EFQ block-scale reference point (default FSA_EFQ_PHI_DEFAULT), 0 <= phi < 1 */
  uint32_t timeout_ms;   /* limit of each on-chip wait (0: 4000 ms) */
  int32_t* row_fallbacks;/* optional device int32 [B][H][Sq]: fallback count per row */
  int32_t  inject_stall; /* test hook: 1 makes the MMA warp wait on a barrier nobody
                            arrives on, so the bounded wait expires (status TIMEOUT) */
  int32_t  schedule;     /* fsa_schedule (default FSA_SCHED_AUTO); the result does not
                            depend on it: both schedules compute bit-identical outputs */
  int32_t  out_dtype;    /* fsa_out_dtype of `out` (default FSA_OUT_F32) */
  int32_t  reserved;
  const fsa_debug_dump* debug;  /* optional (NULL: none): run the debug instance, which
                            also writes the per-tile dumps; per-query-tile schedule,
                            exp modes POLY and MUFU (else FSA_ERR_UNSUPPORTED_FMT) */
} fsa_opts;

typedef enum {
  FSA_SCHED_AUTO = 0,        /* persistent when query tiles average at most 32 key tiles
                                (short causal prefill), else one CTA per query tile; the
                                BF16 entry point always takes one CTA per query tile */
  FSA_SCHED_PER_TILE = 1,    /* one CTA per 128-row query tile */
  FSA_SCHED_PERSISTENT = 2   /* one CTA per SM, each walking a list of query tiles: a CTA's
                                setup, first loads, pipeline fill and drain are paid once
                                per SM instead of once per query tile */
} fsa_schedule;

typedef struct {                      /* device memory, zeroed by the caller */
  unsigned long long fallback_events; /* (row, tile) pairs whose score beat the frozen max */
  unsigned long long row_tiles;       /* (row, tile) pairs with at least one visible key */
  int32_t status;                     /* FSA_OK or FSA_ERR_TIMEOUT; after TIMEOUT the output
                                         is undefined */
  int32_t reserved;
} fsa_stats;

void fsa_default_opts(fsa_opts* opts);

/* ------------------------------------------------------------- attention */
/* O[B][H][Sq][D] fp32 = softmax(scale * Q K^T) V computed by the fused MX
 * algorithm: QK^T as a block-scaled MMA into tensor memory; the row maximum
 * frozen from the first key tile of 128, with a fallback that rescales the
 * accumulator when a later tile's maximum exceeds it by more than delta; per
 * 32-key block an exponent-only scale from the block maximum and codes by
 * exp-then-round (fmt_pv E4M3/E2M3/E2M1) or the EFQ rule (E2M1_EFQ);
 * P~ [V^|1] as a block-scaled MMA whose extra ones column accumulates the
 * denominator; O = O_acc / l in fp32.
 * q, k: FSA_MX_ROWS tensors in fmt_qk; v: FSA_MX_COLS_T tensor in the
 * element format of fmt_pv (E2M1 for E2M1_EFQ).  out: device fp32, 16-byte
 * aligned.  scale: softmax scale (e.g. 1/sqrt(D)). */
int fsa_attention_fwd(const fsa_mx_tensor* q, const fsa_mx_tensor* k, const fsa_mx_tensor* v, float* out,
                      int B, int H, int Hkv, int Sq, int Sk, int D, int causal, float scale,
                      int fmt_qk, int fmt_pv, void* stream);

/* As fsa_attention_fwd with options and statistics: the frozen-maximum margin
 * (the fallback of "Moving softmax to matrix operations...", "Read it as"), the
 * exp2 path of the exp-then-round formats (its "fast method"), the EFQ rule's
 * constants (EFQ-Softmax page, abstract), the output dtype (`out` is fp32 or
 * bf16 [B][H][Sq][D] per opts->out_dtype, 16-byte aligned), the schedule, the
 * wait limit and the debug dumps.  opts NULL: defaults.  stats: device
 * fsa_stats (NULL: none; without stats a wait that times out is not reported).
 * Errors as fsa_attention_fwd, plus FSA_ERR_INVALID_ARG for options out of
 * range (negative or non-finite delta, exp_mode, EFQ constants, schedule,
 * out_dtype) and FSA_ERR_UNSUPPORTED_FMT for a debug run of a format pair or
 * exp mode without a debug instance. */
int fsa_attention_fwd_ex(const fsa_mx_tensor* q, const fsa_mx_tensor* k, const fsa_mx_tensor* v, void* out,
                         int B, int H, int Hkv, int Sq, int Sk, int D, int causal, float scale,
                         int fmt_qk, int fmt_pv, const fsa_opts* opts, fsa_stats* stats, void* stream);

/* As fsa_attention_fwd_ex, with Q given as bf16 [B][H][Sq][D] (device, 16-byte
 * aligned) and quantised to fmt_qk inside the attention kernel's prologue, so Q
 * makes no round trip through HBM as MX codes (the Fused-Softmax brief, abstract:
 * MX operands of the attention GEMMs; the codes and scales are those of
 * fsa_mx_quantize, so the output is bit-identical to quantising Q first).  Runs
 * one CTA per query tile with the hardware exp2 (or EFQ P codes): a request for
 * the persistent schedule, another exp mode or a debug dump returns
 * FSA_ERR_UNSUPPORTED_FMT.  Other errors as fsa_attention_fwd_ex. */
int fsa_attention_fwd_qbf16(const void* q_bf16, const fsa_mx_tensor* k, const fsa_mx_tensor* v, void* out,
                            int B, int H, int Hkv, int Sq, int Sk, int D, int causal, float scale,
                            int fmt_qk, int fmt_pv, const fsa_opts* opts, fsa_stats* stats, void* stream);

/* Rearrange V [B][Hkv][S][D] bf16 into V^T [B][Hkv][D][Sp] bf16 (Sp = S
 * rounded up to 128, zero padded) for the BF16 kernel. */
int fsa_bf16_transpose_v(const void* v, void* vt, int B, int Hkv, int S, int D, void* stream);

/* In-house baseline: the same kernel skeleton with BF16 operands and exact
 * online softmax (standard attention of the "How it works" figure, tiled with
 * the running maximum and historical rescaling that the EFQ page keeps
 * unchanged; rescale only when the maximum grows by more than 8 in log2
 * units).  q [B][H][Sq][D], vt from fsa_bf16_transpose_v, k [B][Hkv][Sk][D],
 * all bf16 device, 16-byte aligned; out fp32. */
int fsa_attention_fwd_bf16(const void* q, const void* k, const void* vt, float* out,
                           int B, int H, int Hkv, int Sq, int Sk, int D, int causal, float scale,
                           fsa_stats* stats, void* stream);

/* ------------------------------------------------- hybrid-format layer schedule */
/* One attention layer of a model that picks its MX formats per layer (the
 * Fused-Softmax brief, abstract: a hybrid MXFP6/MXFP4 schedule on a video
 * model).  Fields as the arguments of fsa_attention_fwd_ex; `out` is fp32 or
 * bf16 per the call's opts->out_dtype; `delta` is this layer's frozen-maximum
 * margin (>= 0); `stats` optional device fsa_stats of this layer. */
typedef struct {
  const fsa_mx_tensor* q;
  const fsa_mx_tensor* k;
  const fsa_mx_tensor* v;
  void*   out;
  int32_t B, H, Hkv, Sq, Sk, D, causal;
  float   scale;
  int32_t fmt_qk, fmt_pv;
  float   delta;
  fsa_stats* stats;
} fsa_layer;

/* Run n_layers layers back to back on `stream`, each with its own formats and
 * margin and the remaining options of `opts` (NULL: defaults; a debug dump is
 * refused, the per-row fallback buffer is not used).  Every layer's arguments
 * are checked before the first launch: on an argument error nothing is
 * enqueued.  Errors as fsa_attention_fwd_ex. */
int fsa_attention_fwd_layers(const fsa_layer* layers, int n_layers, const fsa_opts* opts, void* stream);

/* Host-side margin update driven by the fallback counts of a previous run (the
 * speculative maximum of "Moving softmax to matrix operations...", "Read it
 * as", falls back when the guess is wrong; a larger margin trades fallbacks for
 * accumulator headroom).  stats: HOST copies of each layer's fsa_stats; delta:
 * host array of the layers' margins, updated in place: a layer whose fallback
 * rate (events / row-tiles) is above target_rate gets delta + step, at most
 * max_delta; layers without evidence (status not FSA_OK, no row-tiles) keep
 * theirs.  FSA_ERR_INVALID_ARG for null arrays, step <= 0, a negative target or
 * maximum, or a delta outside [0, max_delta]. */
int fsa_tune_delta(const fsa_stats* stats, int n_layers, float target_rate, float step, float max_delta,
                   float* delta);

/* ------------------------------------------------------- from host memory */
/* Inputs and output of one attention call in HOST memory (page-locked memory lets
 * the copies run asynchronously and overlap; pageable memory works, without the
 * overlap).  q [B][H][Sq][D], k and v [B][Hkv][Sk][D] bf16; out [B][H][Sq][D] fp32
 * or bf16 per opts->out_dtype. */
typedef struct {
  const void* q;
  const void* k;
  const void* v;
  void*       out;
} fsa_host_io;

/* The caller's device buffers for the same call: q, k, v bf16 of the host shapes,
 * out of the output's shape and dtype, and the three MX tensors (codes and scales
 * of fsa_mx_sizes bytes for q and k in FSA_MX_ROWS / fmt_qk and v in
 * FSA_MX_COLS_T / the storage format of fmt_pv).  All 16-byte aligned. */
typedef struct {
  void*          q;
  void*          k;
  void*          v;
  fsa_mx_tensor* q_mx;
  fsa_mx_tensor* k_mx;
  fsa_mx_tensor* v_mx;
  void*          out;
} fsa_device_io;

/* The attention of fsa_attention_fwd_ex (the Fused-Softmax brief, abstract; the
 * pages say nothing of where the operands live) on operands in host memory.  The
 * call is split into n_chunks groups of whole kv heads (a kv head with its H/Hkv
 * query heads; n_chunks <= 0: min(B*Hkv, 8), fewer when a group would hold under two
 * query tiles per SM), and for each group: Q, K and V are
 * copied host to device on a stream of the library's own, quantised
 * (fsa_mx_quantize_qkv) and attended on `stream` once they have landed, and O
 * copied back on a second stream of its own while the next group computes.  The
 * output is bit-identical to quantising and attending the whole call at once (every
 * head is computed by the same kernels on the same data).  Nothing is allocated on
 * the device; the two streams and the events are created by the call and released
 * when their work completes.  On return the work is enqueued: `stream` completes
 * after the last copy back, so synchronising it makes host->out valid.  The MX
 * tensors' shape, layout and format fields are written as fsa_mx_quantize_qkv
 * would.  opts as fsa_attention_fwd_ex (row_fallbacks: device [B][H][Sq]; a debug
 * dump is refused); stats accumulates over the groups.  Not for CUDA graph capture.
 * Errors: FSA_ERR_INVALID_ARG (null or misaligned pointer, bad shape or option),
 * FSA_ERR_UNSUPPORTED_FMT, FSA_ERR_LAUNCH (a stream, event, copy or launch failed;
 * what was enqueued before the failure still completes before `stream` does). */
int fsa_attention_fwd_host(const fsa_host_io* host, const fsa_device_io* dev, int B, int H, int Hkv, int Sq,
                           int Sk, int D, int causal, float scale, int fmt_qk, int fmt_pv, const fsa_opts* opts,
                           fsa_stats* stats, int n_chunks, void* stream);

/* ------------------------------------------------------ tensor-core peak probe */
/* Measurement instrument (the roofline denominator of the attention kernels; the
 * Fused-Softmax brief, abstract, quotes its kernels' throughput on the block-
 * scaled matrix cores).  Launches n_ctas CTAs (one per SM) that each issue
 * `iters` iterations of dense M=128, N=n (128 or 256), K=128 products from
 * shared-memory operand tiles into tensor memory, as 8 kind::f16 bf16 MMAs
 * (kind 0), 4 kind::mxf8f6f4 E4M3 block-scaled MMAs (kind 1), 2 kind::mxf4
 * E2M1 block-scaled MMAs (kind 2) or 2 kind::mxf4nvf4 MMAs on the same MXFP4
 * operands (E2M1, E8M0 scales, scale_vec::2X; kind 3).  *flops (host, optional) receives the
 * launch's 2*M*N*K*iters*n_ctas; time the launch with events on `stream`.
 * status: optional device int32, set to FSA_ERR_TIMEOUT if the final wait
 * (2 s) expires.  Errors: FSA_ERR_INVALID_ARG, FSA_ERR_LAUNCH. */
int fsa_mma_peak(int kind, int n, int n_ctas, long long iters, int32_t* status, double* flops, void* stream);

const char* fsa_status_string(int status);
int fsa_version(void);

#ifdef __cplusplus
}
#endif
#endif /* FSA_H */
