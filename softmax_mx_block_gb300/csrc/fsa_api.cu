// fsa_api.cu -- the C ABI of libfsa (declared in include/fsa.h): argument
// checks, TMA tensor-map construction and kernel dispatch.  No entry point
// allocates device memory; all buffers belong to the caller.
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <cuda.h>
#include <cuda_runtime.h>
#include "fsa.h"
#include "fsa_launch.h"

namespace {

using fsa::AttnLaunch;

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// 3-D byte tensor {inner bytes, rows, planes}, box {width, box_rows, 1}, swizzle by width.
bool make_tmap(CUtensorMap* m, const void* base, uint64_t inner, uint64_t rows, uint64_t planes, uint32_t width,
               uint32_t box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[3] = {inner, rows, planes};
  const cuuint64_t strides[2] = {inner, inner * rows};
  const cuuint32_t box[3] = {width, box_rows, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUtensorMapSwizzle sw = width == 128 ? CU_TENSOR_MAP_SWIZZLE_128B
                                : width == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                                              : CU_TENSOR_MAP_SWIZZLE_32B;
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Tensor map of the fp32 output O [planes][rows][D]: boxes of 32 rows x 32 floats
// (128 bytes), 128B swizzle, written by TMA stores from the kernel's epilogue.
// fp32 output [planes][rows][D]: 32x32 boxes with 128B swizzle (one CTA per query
// tile), or 16x32 boxes with 64B swizzle (the persistent schedule's staging box)
bool make_tmap_out(CUtensorMap* m, float* base, uint64_t D, uint64_t rows, uint64_t planes, bool persistent) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[3] = {D, rows, planes};
  const cuuint64_t strides[2] = {D * 4, D * 4 * rows};
  const cuuint32_t box[3] = {persistent ? 16u : 32u, 32, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            persistent ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// storage bits per element * 2, as the kernels store them
int bits2_of(int fmt) { return fmt == FSA_FMT_E2M1 || fmt == FSA_FMT_E2M1_EFQ ? 8 : 16; }

int row_bytes(int D, int fmt) { return D * bits2_of(fmt) / 16; }

bool valid_fmt(int f) { return f >= FSA_FMT_E4M3 && f <= FSA_FMT_E2M1; }

int storage_fmt(int f) { return f == FSA_FMT_E2M1_EFQ ? FSA_FMT_E2M1 : f; }

bool shape_ok(int B, int H, int Hkv, int Sq, int Sk, int D) {
  return B > 0 && H > 0 && Hkv > 0 && H % Hkv == 0 && Sq > 0 && Sk > 0 && (D == 64 || D == 128) &&
         (int64_t)B * H <= 65535 && (int64_t)Sq <= 65535 * 128 && (int64_t)Sk <= (1 << 24);
}

using ImplFn = cudaError_t (*)(const AttnLaunch&);

ImplFn impl_for(int fqk, int fpv) {
  using namespace fsa;
  static const ImplFn table[3][4] = {
      {launch_attn_impl<0, 0>, launch_attn_impl<0, 1>, launch_attn_impl<0, 2>, launch_attn_impl<0, 3>},
      {launch_attn_impl<1, 0>, launch_attn_impl<1, 1>, launch_attn_impl<1, 2>, launch_attn_impl<1, 3>},
      {launch_attn_impl<2, 0>, launch_attn_impl<2, 1>, launch_attn_impl<2, 2>, launch_attn_impl<2, 3>}};
  return table[fqk][fpv];
}

int launch_status(cudaError_t e) { return e == cudaSuccess ? FSA_OK : FSA_ERR_LAUNCH; }

// The schedule: FSA_SCHED_AUTO takes the persistent one when the query tiles average
// at most 32 key tiles, where a CTA's fixed cost (setup, first loads, pipeline fill
// and drain, output) is a large share of its work; measured on GB300 it gains 8% on
// causal 4K prefill and loses a few percent on long sequences.
bool persistent_schedule(int schedule, int Sq, int Sk, int causal) {
  if (schedule == FSA_SCHED_PER_TILE) return false;
  if (schedule == FSA_SCHED_PERSISTENT) return true;
  const int64_t nq = (Sq + 127) / 128, nk = (Sk + 127) / 128;
  int64_t tiles = 0;
  for (int64_t qt = 0; qt < nq; ++qt) {
    int64_t n = nk;
    if (causal) {
      const int64_t lim = qt * 128 + 127 + Sk - Sq;
      n = lim < 0 ? 0 : std::min<int64_t>(nk, lim / 128 + 1);
    }
    tiles += n;
  }
  return tiles <= 32 * nq;
}

void fill_common(fsa::KParams& p, int B, int H, int Hkv, int Sq, int Sk, int causal, float scale,
                 const fsa_opts* o, fsa_stats* stats) {
  p.B = B; p.H = H; p.Hkv = Hkv; p.Sq = Sq; p.Sk = Sk;
  p.n_qtiles = (Sq + 127) / 128;
  p.n_items = B * H * p.n_qtiles;
  p.causal = causal ? 1 : 0;
  p.c = (float)((double)scale * 1.4426950408889634073599246810018921);   // log2(e)
  p.delta = o->delta;
  p.efq_beta = o->efq_beta;
  p.efq_fast = (o->efq_beta <= 2 && o->delta <= 120.0f) ? 1 : 0;
  p.timeout_ns = (uint64_t)(o->timeout_ms ? o->timeout_ms : 4000u) * 1000000ull;
  p.row_fallbacks = o->row_fallbacks;
  p.stat_fallbacks = stats ? &stats->fallback_events : nullptr;
  p.stat_row_tiles = stats ? &stats->row_tiles : nullptr;
  p.status = stats ? &stats->status : nullptr;
  p.inject_stall = o->inject_stall;
}

}  // namespace

extern "C" {

void fsa_default_opts(fsa_opts* o) {
  if (!o) return;
  std::memset(o, 0, sizeof(*o));
  o->delta = 8.0f;
  o->exp_mode = FSA_EXP_MUFU;
  o->efq_beta = 2;
  o->timeout_ms = 4000;
}

int fsa_version(void) { return 100; }

const char* fsa_status_string(int s) {
  switch (s) {
    case FSA_OK: return "ok";
    case FSA_ERR_INVALID_ARG: return "invalid argument";
    case FSA_ERR_UNSUPPORTED_FMT: return "unsupported format";
    case FSA_ERR_LAUNCH: return "CUDA launch error";
    case FSA_ERR_TIMEOUT: return "on-chip wait timed out";
    case FSA_ERR_NO_DEVICE: return "no tcgen05-capable device";
    default: return "unknown status";
  }
}

int fsa_mx_sizes(int B, int H, int S, int D, int layout, int fmt, size_t* codes_bytes, size_t* scales_bytes) {
  if (B <= 0 || H <= 0 || S <= 0 || (D != 64 && D != 128) || !valid_fmt(storage_fmt(fmt)) ||
      (layout != FSA_MX_ROWS && layout != FSA_MX_COLS_T) || !codes_bytes || !scales_bytes)
    return FSA_ERR_INVALID_ARG;
  const size_t bh = (size_t)B * H;
  const int sf = storage_fmt(fmt);
  if (layout == FSA_MX_ROWS) {
    *codes_bytes = bh * (size_t)S * row_bytes(D, sf);
    *scales_bytes = bh * (size_t)((S + 127) / 128) * 512;
  } else {
    const size_t Sp = (size_t)(S + 127) / 128 * 128;
    *codes_bytes = bh * (size_t)D * Sp * bits2_of(sf) / 16;
    *scales_bytes = bh * (Sp / 128) * 512;
  }
  return FSA_OK;
}

int fsa_mx_quantize(const void* x, int B, int H, int S, int D, int layout, int fmt, fsa_mx_tensor* out,
                    void* stream) {
  size_t cb, sb;
  if (!x || !out || !out->codes || !out->scales) return FSA_ERR_INVALID_ARG;
  if (fmt == FSA_FMT_E2M1_EFQ) return FSA_ERR_UNSUPPORTED_FMT;
  int st = fsa_mx_sizes(B, H, S, D, layout, fmt, &cb, &sb);
  if (st != FSA_OK) return st;
  if (!aligned16(x) || !aligned16(out->codes) || !aligned16(out->scales)) return FSA_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  out->fmt = fmt; out->layout = layout; out->B = B; out->H = H; out->S = S; out->D = D;
  // the kernels write every byte of codes and scales (unused scale slots: 2^0, 0x7F)
  cudaError_t e;
  if (layout == FSA_MX_ROWS) e = fsa::launch_mx_quant_rows(x, B * H, S, D, fmt, out->codes, out->scales, s);
  else e = fsa::launch_mx_quant_cols(x, B * H, S, D, fmt, out->codes, out->scales, s);
  return launch_status(e);
}

int fsa_mx_quantize_qkv(const void* q, const void* k, const void* v, int B, int H, int Hkv, int Sq, int Sk, int D,
                        int fmt_qk, int fmt_v, fsa_mx_tensor* q_out, fsa_mx_tensor* k_out, fsa_mx_tensor* v_out,
                        void* stream) {
  size_t cb, sb;
  if (!q || !k || !v || !q_out || !k_out || !v_out) return FSA_ERR_INVALID_ARG;
  if (fmt_qk == FSA_FMT_E2M1_EFQ || fmt_v == FSA_FMT_E2M1_EFQ) return FSA_ERR_UNSUPPORTED_FMT;
  int st;
  if ((st = fsa_mx_sizes(B, H, Sq, D, FSA_MX_ROWS, fmt_qk, &cb, &sb)) != FSA_OK) return st;
  if ((st = fsa_mx_sizes(B, Hkv, Sk, D, FSA_MX_ROWS, fmt_qk, &cb, &sb)) != FSA_OK) return st;
  if ((st = fsa_mx_sizes(B, Hkv, Sk, D, FSA_MX_COLS_T, fmt_v, &cb, &sb)) != FSA_OK) return st;
  const fsa_mx_tensor* outs[3] = {q_out, k_out, v_out};
  for (const fsa_mx_tensor* o : outs)
    if (!o->codes || !o->scales || !aligned16(o->codes) || !aligned16(o->scales)) return FSA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v)) return FSA_ERR_INVALID_ARG;
  auto set = [&](fsa_mx_tensor* o, int fmt, int layout, int h, int S) {
    o->fmt = fmt; o->layout = layout; o->B = B; o->H = h; o->S = S; o->D = D;
  };
  set(q_out, fmt_qk, FSA_MX_ROWS, H, Sq);
  set(k_out, fmt_qk, FSA_MX_ROWS, Hkv, Sk);
  set(v_out, fmt_v, FSA_MX_COLS_T, Hkv, Sk);
  return launch_status(fsa::launch_mx_quant_qkv(q, k, v, B * H, B * Hkv, Sq, Sk, D, fmt_qk, fmt_v, q_out->codes,
                                                q_out->scales, k_out->codes, k_out->scales, v_out->codes,
                                                v_out->scales, static_cast<cudaStream_t>(stream)));
}

int fsa_bf16_transpose_v(const void* v, void* vt, int B, int Hkv, int S, int D, void* stream) {
  if (!v || !vt || B <= 0 || Hkv <= 0 || S <= 0 || (D != 64 && D != 128) || !aligned16(v) || !aligned16(vt))
    return FSA_ERR_INVALID_ARG;
  return launch_status(fsa::launch_transpose_v(v, vt, B * Hkv, S, D, static_cast<cudaStream_t>(stream)));
}

int fsa_attention_fwd_ex(const fsa_mx_tensor* q, const fsa_mx_tensor* k, const fsa_mx_tensor* v, float* out,
                         int B, int H, int Hkv, int Sq, int Sk, int D, int causal, float scale, int fmt_qk,
                         int fmt_pv, const fsa_opts* opts, fsa_stats* stats, void* stream) {
  if (!q || !k || !v || !out) return FSA_ERR_INVALID_ARG;
  if (!shape_ok(B, H, Hkv, Sq, Sk, D) || !(scale > 0.0f) || !std::isfinite(scale)) return FSA_ERR_INVALID_ARG;
  if (!valid_fmt(fmt_qk) || fmt_pv < FSA_FMT_E4M3 || fmt_pv > FSA_FMT_E2M1_EFQ) return FSA_ERR_UNSUPPORTED_FMT;
  const int fv = storage_fmt(fmt_pv);
  // operand descriptors must match the call
  if (q->layout != FSA_MX_ROWS || k->layout != FSA_MX_ROWS || v->layout != FSA_MX_COLS_T) return FSA_ERR_INVALID_ARG;
  if (q->fmt != fmt_qk || k->fmt != fmt_qk || v->fmt != fv) return FSA_ERR_UNSUPPORTED_FMT;
  if (q->B != B || q->H != H || q->S != Sq || q->D != D || k->B != B || k->H != Hkv || k->S != Sk || k->D != D ||
      v->B != B || v->H != Hkv || v->S != Sk || v->D != D)
    return FSA_ERR_INVALID_ARG;
  if (!aligned16(q->codes) || !aligned16(k->codes) || !aligned16(v->codes) || !aligned16(q->scales) ||
      !aligned16(k->scales) || !aligned16(v->scales) || !aligned16(out))
    return FSA_ERR_INVALID_ARG;
  fsa_opts o;
  fsa_default_opts(&o);
  if (opts) o = *opts;
  if (o.exp_mode < 0 || o.exp_mode > 2 || o.efq_beta < -16 || o.efq_beta > 16 || !std::isfinite(o.delta) ||
      o.schedule < FSA_SCHED_AUTO || o.schedule > FSA_SCHED_PERSISTENT)
    return FSA_ERR_INVALID_ARG;
  const bool persistent = persistent_schedule(o.schedule, Sq, Sk, causal);

  AttnLaunch a;
  std::memset(&a, 0, sizeof(a));
  const int rbq = row_bytes(D, fmt_qk);
  const uint32_t wq = rbq < 128 ? rbq : 128;
  const uint64_t Sp = (uint64_t)(Sk + 127) / 128 * 128;
  const uint64_t rbv_total = Sp * bits2_of(fv) / 16;
  const int rbv_tile = 128 * bits2_of(fv) / 16;
  const uint32_t wv = rbv_tile < 128 ? rbv_tile : 128;
  if (!make_tmap(&a.tq, q->codes, rbq, Sq, (uint64_t)B * H, wq, 128) ||
      !make_tmap(&a.tk, k->codes, rbq, Sk, (uint64_t)B * Hkv, wq, 128) ||
      !make_tmap(&a.tv, v->codes, rbv_total, D, (uint64_t)B * Hkv, wv, D) ||
      !make_tmap_out(&a.to, out, D, Sq, (uint64_t)B * H, persistent))
    return FSA_ERR_LAUNCH;
  fill_common(a.p, B, H, Hkv, Sq, Sk, causal, scale, &o, stats);
  a.p.sf_q = q->scales; a.p.sf_k = k->scales; a.p.sf_v = v->scales;
  a.p.out = out;
  a.D = D;
  a.exp_mode = o.exp_mode;
  a.persistent = persistent ? 1 : 0;
  a.stream = static_cast<cudaStream_t>(stream);
  return launch_status(impl_for(fmt_qk, fmt_pv)(a));
}

int fsa_attention_fwd(const fsa_mx_tensor* q, const fsa_mx_tensor* k, const fsa_mx_tensor* v, float* out, int B,
                      int H, int Hkv, int Sq, int Sk, int D, int causal, float scale, int fmt_qk, int fmt_pv,
                      void* stream) {
  return fsa_attention_fwd_ex(q, k, v, out, B, H, Hkv, Sq, Sk, D, causal, scale, fmt_qk, fmt_pv, nullptr, nullptr,
                              stream);
}

int fsa_attention_fwd_bf16(const void* q, const void* k, const void* vt, float* out, int B, int H, int Hkv, int Sq,
                           int Sk, int D, int causal, float scale, fsa_stats* stats, void* stream) {
  if (!q || !k || !vt || !out) return FSA_ERR_INVALID_ARG;
  if (!shape_ok(B, H, Hkv, Sq, Sk, D) || !(scale > 0.0f) || !std::isfinite(scale)) return FSA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(vt) || !aligned16(out)) return FSA_ERR_INVALID_ARG;
  fsa_opts o;
  fsa_default_opts(&o);
  // one CTA per query tile: on GB300 the persistent schedule measured slower for the
  // BF16 kernel (its K/V ring has two stages), even on short causal prefill
  const bool persistent = false;
  AttnLaunch a;
  std::memset(&a, 0, sizeof(a));
  const uint64_t Sp = (uint64_t)(Sk + 127) / 128 * 128;
  if (!make_tmap(&a.tq, q, 2 * D, Sq, (uint64_t)B * H, 128, 128) ||
      !make_tmap(&a.tk, k, 2 * D, Sk, (uint64_t)B * Hkv, 128, 128) ||
      !make_tmap(&a.tv, vt, 2 * Sp, D, (uint64_t)B * Hkv, 128, D) ||
      !make_tmap_out(&a.to, out, D, Sq, (uint64_t)B * H, persistent))
    return FSA_ERR_LAUNCH;
  fill_common(a.p, B, H, Hkv, Sq, Sk, causal, scale, &o, stats);
  a.p.out = out;
  a.D = D;
  a.persistent = persistent ? 1 : 0;
  a.stream = static_cast<cudaStream_t>(stream);
  return launch_status(fsa::launch_attn_impl<fsa::F_BF16, fsa::F_BF16>(a));
}

}  // extern "C"
