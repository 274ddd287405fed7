// fsa_api.cu -- the C ABI of libfsa (declared in include/fsa.h): argument
// checks, TMA tensor-map construction and kernel dispatch.  No entry point
// allocates device memory; all buffers belong to the caller (the host-memory entry
// point creates two streams and some events, released when their work completes).
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <climits>
#include <mutex>
#include <unordered_map>
#include <vector>
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

// Tensor maps are a pure function of (base, type, dims, strides, box, swizzle):
// encoded once per distinct key and reused, so repeated calls on the same buffers
// skip the driver's encode.  The cache is bounded (cleared when full).
struct TmapKey {
  uintptr_t base;
  uint64_t dims[3], strides[2];
  uint32_t box[3];
  int dtype, swizzle, promo;
  bool operator==(const TmapKey& o) const { return std::memcmp(this, &o, sizeof(*this)) == 0; }
};
struct TmapKeyHash {
  size_t operator()(const TmapKey& k) const {
    const unsigned char* b = reinterpret_cast<const unsigned char*>(&k);
    uint64_t h = 1469598103934665603ull;                     // FNV-1a over the key bytes
    for (size_t i = 0; i < sizeof(k); ++i) h = (h ^ b[i]) * 1099511628211ull;
    return (size_t)h;
  }
};

bool encode_cached(CUtensorMap* m, CUtensorMapDataType dtype, const void* base, const uint64_t dims[3],
                   const uint64_t strides[2], const uint32_t box[3], CUtensorMapSwizzle sw,
                   CUtensorMapL2promotion promo) {
  static std::mutex mu;
  static std::unordered_map<TmapKey, CUtensorMap, TmapKeyHash> cache;
  TmapKey key;
  std::memset(&key, 0, sizeof(key));
  key.base = reinterpret_cast<uintptr_t>(base);
  for (int i = 0; i < 3; ++i) { key.dims[i] = dims[i]; key.box[i] = box[i]; }
  key.strides[0] = strides[0]; key.strides[1] = strides[1];
  key.dtype = (int)dtype; key.swizzle = (int)sw; key.promo = (int)promo;
  {
    std::lock_guard<std::mutex> g(mu);
    auto it = cache.find(key);
    if (it != cache.end()) { *m = it->second; return true; }
  }
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t d[3] = {dims[0], dims[1], dims[2]};
  const cuuint64_t st[2] = {strides[0], strides[1]};
  const cuuint32_t bx[3] = {box[0], box[1], box[2]};
  const cuuint32_t estr[3] = {1, 1, 1};
  if (fn(m, dtype, 3, const_cast<void*>(base), d, st, bx, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw, promo,
         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return false;
  std::lock_guard<std::mutex> g(mu);
  if (cache.size() >= 512) cache.clear();
  cache.emplace(key, *m);
  return true;
}

// 3-D byte tensor {inner bytes, rows, planes}, box {width, box_rows, 1}, swizzle by width.
bool make_tmap(CUtensorMap* m, const void* base, uint64_t inner, uint64_t rows, uint64_t planes, uint32_t width,
               uint32_t box_rows) {
  const uint64_t dims[3] = {inner, rows, planes};
  const uint64_t strides[2] = {inner, inner * rows};
  const uint32_t box[3] = {width, box_rows, 1};
  const CUtensorMapSwizzle sw = width == 128 ? CU_TENSOR_MAP_SWIZZLE_128B
                                : width == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                                              : CU_TENSOR_MAP_SWIZZLE_32B;
  return encode_cached(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, base, dims, strides, box, sw,
                       CU_TENSOR_MAP_L2_PROMOTION_L2_256B);
}

// 3-D byte tensor loaded unswizzled: box {inner bytes (<= 256), box_rows, 1}.
bool make_tmap_plain(CUtensorMap* m, const void* base, uint64_t inner, uint64_t rows, uint64_t planes,
                     uint32_t box_rows) {
  const uint64_t dims[3] = {inner, rows, planes};
  const uint64_t strides[2] = {inner, inner * rows};
  const uint32_t box[3] = {(uint32_t)inner, box_rows, 1};
  return encode_cached(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, base, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_NONE,
                       CU_TENSOR_MAP_L2_PROMOTION_L2_256B);
}

// Output O [planes][rows][D], written by TMA stores from the epilogue.
//   one CTA per query tile: fp32 boxes of 32 rows x 32 floats (128B swizzle); bf16
//     boxes of 32 rows x D/2 values (128B swizzle for D = 128, 64B for D = 64)
//   persistent schedule: boxes of 32 rows x 16 values, fp32 (64B swizzle) or bf16
//     (32B swizzle)
bool make_tmap_out(CUtensorMap* m, void* base, uint64_t D, uint64_t rows, uint64_t planes, bool persistent,
                   bool bf16) {
  const uint64_t esz = bf16 ? 2 : 4;
  const uint64_t dims[3] = {D, rows, planes};
  const uint64_t strides[2] = {D * esz, D * esz * rows};
  uint32_t bw;
  CUtensorMapSwizzle sw;
  if (!bf16) {
    bw = persistent ? 16u : 32u;
    sw = persistent ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B;
  } else if (persistent) {
    bw = 16u;
    sw = CU_TENSOR_MAP_SWIZZLE_32B;
  } else {
    bw = (uint32_t)(D / 2);
    sw = D == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
  }
  const uint32_t box[3] = {bw, 32, 1};
  return encode_cached(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, base, dims,
                       strides, box, sw, CU_TENSOR_MAP_L2_PROMOTION_NONE);
}

// storage bits per element * 2, as the kernels store them
int bits2_of(int fmt) { return fmt == FSA_FMT_E2M1 || fmt == FSA_FMT_E2M1_EFQ || fmt == FSA_FMT_NVFP4 ? 8 : 16; }

int row_bytes(int D, int fmt) { return D * bits2_of(fmt) / 16; }

// storage formats of MX tensors (E2M1_EFQ is a P format only; NVFP4 a Q/K format only)
bool valid_fmt(int f) {
  return (f >= FSA_FMT_E4M3 && f <= FSA_FMT_E2M1) || f == FSA_FMT_E3M2 || f == FSA_FMT_NVFP4;
}
bool valid_pv(int f) { return f >= FSA_FMT_E4M3 && f <= FSA_FMT_E3M2; }

int storage_fmt(int f) { return f == FSA_FMT_E2M1_EFQ ? FSA_FMT_E2M1 : f; }

// The query-tile count B*H*ceil(Sq/128) must fit an int (the persistent schedule
// indexes its work list with it).  Sk is limited by accuracy, not indexing: the fp32
// accumulator in tensor memory drifts by a per-row factor that grows with the key
// tiles added into it, as adds that drop low-order bits would (below 5e-4 of the
// output at 2^20 keys, up to 7e-3 at 2^22 with 8-bit P~).
bool shape_ok(int B, int H, int Hkv, int Sq, int Sk, int D) {
  return B > 0 && H > 0 && Hkv > 0 && H % Hkv == 0 && Sq > 0 && Sk > 0 && (D == 64 || D == 128) &&
         (int64_t)B * H <= 65535 && (int64_t)Sq <= 65535 * 128 && (int64_t)Sk <= (1 << 20) &&
         (int64_t)B * H * ((Sq + 127) / 128) <= INT_MAX;
}

using ImplFn = cudaError_t (*)(const AttnLaunch&);

// fsa.h format numbers are the kernels' template arguments (fsa_attn.cuh)
ImplFn impl_for(int fqk, int fpv) {
  using namespace fsa;
  static const ImplFn table[6][5] = {
      {launch_attn_impl<0, 0>, launch_attn_impl<0, 1>, launch_attn_impl<0, 2>, launch_attn_impl<0, 3>,
       launch_attn_impl<0, 4>},
      {launch_attn_impl<1, 0>, launch_attn_impl<1, 1>, launch_attn_impl<1, 2>, launch_attn_impl<1, 3>,
       launch_attn_impl<1, 4>},
      {launch_attn_impl<2, 0>, launch_attn_impl<2, 1>, launch_attn_impl<2, 2>, launch_attn_impl<2, 3>,
       launch_attn_impl<2, 4>},
      {nullptr, nullptr, nullptr, nullptr, nullptr},
      {launch_attn_impl<4, 0>, launch_attn_impl<4, 1>, launch_attn_impl<4, 2>, launch_attn_impl<4, 3>,
       launch_attn_impl<4, 4>},
      {launch_attn_impl<6, 0>, launch_attn_impl<6, 1>, launch_attn_impl<6, 2>, launch_attn_impl<6, 3>,
       launch_attn_impl<6, 4>}};   // NVFP4 (fsa.h 5) is the kernels' format 6
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

// a negative margin would make nearly every tile fall back; the EFQ constants keep
// the code domain finite and the block exponent's reference point within one binade
bool opts_ok(const fsa_opts& o) {
  return !(o.exp_mode < 0 || o.exp_mode > 2 || !std::isfinite(o.delta) || o.delta < 0.0f ||
           !(o.efq_a > 0.0f && o.efq_a <= 16.0f) || !(std::fabs(o.efq_b) <= 64.0f) ||
           !(o.efq_phi >= 0.0f && o.efq_phi < 1.0f) || o.schedule < FSA_SCHED_AUTO ||
           o.schedule > FSA_SCHED_PERSISTENT || (o.out_dtype != FSA_OUT_F32 && o.out_dtype != FSA_OUT_BF16));
}

void fill_common(fsa::KParams& p, int B, int H, int Hkv, int Sq, int Sk, int causal, float scale,
                 const fsa_opts* o, fsa_stats* stats) {
  p.B = B; p.H = H; p.Hkv = Hkv; p.Sq = Sq; p.Sk = Sk;
  p.n_qtiles = (Sq + 127) / 128;
  p.n_items = B * H * p.n_qtiles;
  p.causal = causal ? 1 : 0;
  p.c = (float)((double)scale * 1.4426950408889634073599246810018921);   // log2(e)
  p.delta = o->delta;
  // EFQ constants scaled by 1/8 (exact): A = fp32(a c), a, b; phi as given
  const float A = o->efq_a * p.c;
  p.efq_A8 = A * 0.125f;
  p.efq_a8 = o->efq_a * 0.125f;
  p.efq_b8 = o->efq_b * 0.125f;
  p.efq_phi = o->efq_phi;
  p.out_bf16 = o->out_dtype == FSA_OUT_BF16 ? 1 : 0;
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
  o->efq_a = FSA_EFQ_A_DEFAULT;
  o->efq_b = FSA_EFQ_B_DEFAULT;
  o->efq_phi = FSA_EFQ_PHI_DEFAULT;
  o->timeout_ms = 4000;
  o->out_dtype = FSA_OUT_F32;
}

int fsa_version(void) { return 200; }

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
      (layout != FSA_MX_ROWS && layout != FSA_MX_COLS_T) || !codes_bytes || !scales_bytes ||
      (fmt == FSA_FMT_NVFP4 && layout != FSA_MX_ROWS))
    return FSA_ERR_INVALID_ARG;
  const size_t bh = (size_t)B * H;
  const int sf = storage_fmt(fmt);
  if (layout == FSA_MX_ROWS) {
    *codes_bytes = bh * (size_t)S * row_bytes(D, sf);
    *scales_bytes = bh * (size_t)((S + 127) / 128) * 512 * (sf == FSA_FMT_NVFP4 ? D / 64 : 1);
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

}  // extern "C"

namespace {

// Both attention entry points: q (MX) or q_bf16 (bf16 [B][H][Sq][D], quantised in the
// kernel's prologue into fmt_qk) -- exactly one of them is non-null.
int attention_impl(const fsa_mx_tensor* q, const void* q_bf16, const fsa_mx_tensor* k, const fsa_mx_tensor* v,
                   void* out, int B, int H, int Hkv, int Sq, int Sk, int D, int causal, float scale, int fmt_qk,
                   int fmt_pv, const fsa_opts* opts, fsa_stats* stats, void* stream) {
  if (!(q || q_bf16) || !k || !v || !out) return FSA_ERR_INVALID_ARG;
  if (!shape_ok(B, H, Hkv, Sq, Sk, D) || !(scale > 0.0f) || !std::isfinite(scale)) return FSA_ERR_INVALID_ARG;
  if (!valid_fmt(fmt_qk) || !valid_pv(fmt_pv)) return FSA_ERR_UNSUPPORTED_FMT;
  const int fv = storage_fmt(fmt_pv);
  // operand descriptors must match the call
  if (q && q->layout != FSA_MX_ROWS) return FSA_ERR_INVALID_ARG;
  if (k->layout != FSA_MX_ROWS || v->layout != FSA_MX_COLS_T) return FSA_ERR_INVALID_ARG;
  if ((q && q->fmt != fmt_qk) || k->fmt != fmt_qk || v->fmt != fv) return FSA_ERR_UNSUPPORTED_FMT;
  if ((q && (q->B != B || q->H != H || q->S != Sq || q->D != D)) || k->B != B || k->H != Hkv || k->S != Sk ||
      k->D != D || v->B != B || v->H != Hkv || v->S != Sk || v->D != D)
    return FSA_ERR_INVALID_ARG;
  if ((q && (!aligned16(q->codes) || !aligned16(q->scales))) || (q_bf16 && !aligned16(q_bf16)) ||
      !aligned16(k->codes) || !aligned16(v->codes) || !aligned16(k->scales) || !aligned16(v->scales) ||
      !aligned16(out))
    return FSA_ERR_INVALID_ARG;
  fsa_opts o;
  fsa_default_opts(&o);
  if (opts) o = *opts;
  if (!opts_ok(o)) return FSA_ERR_INVALID_ARG;
  const fsa_debug_dump* dbg = o.debug;
  if (dbg && (!dbg->s || !dbg->m || !dbg->p || !dbg->p_scales)) return FSA_ERR_INVALID_ARG;
  if (dbg && fmt_pv != FSA_FMT_E2M1_EFQ && o.exp_mode == FSA_EXP_SPLIT) return FSA_ERR_UNSUPPORTED_FMT;
  // Q quantised in the prologue: one CTA per query tile, the hardware exp2 (or EFQ)
  if (q_bf16 && (dbg || o.schedule == FSA_SCHED_PERSISTENT || fmt_qk == FSA_FMT_NVFP4 ||
                 (fmt_pv != FSA_FMT_E2M1_EFQ && o.exp_mode != FSA_EXP_MUFU)))
    return FSA_ERR_UNSUPPORTED_FMT;
  // NVFP4 Q/K run one CTA per query tile
  if (fmt_qk == FSA_FMT_NVFP4 && o.schedule == FSA_SCHED_PERSISTENT) return FSA_ERR_UNSUPPORTED_FMT;
  const bool persistent =
      !dbg && !q_bf16 && fmt_qk != FSA_FMT_NVFP4 && persistent_schedule(o.schedule, Sq, Sk, causal);
  const bool bf16 = o.out_dtype == FSA_OUT_BF16;

  AttnLaunch a;
  std::memset(&a, 0, sizeof(a));
  const int rbq = row_bytes(D, fmt_qk);
  const uint32_t wq = rbq < 128 ? rbq : 128;
  const uint64_t Sp = (uint64_t)(Sk + 127) / 128 * 128;
  const uint64_t rbv_total = Sp * bits2_of(fv) / 16;
  const int rbv_tile = 128 * bits2_of(fv) / 16;
  const uint32_t wv = rbv_tile < 128 ? rbv_tile : 128;
  const bool tq_ok = q ? make_tmap(&a.tq, q->codes, rbq, Sq, (uint64_t)B * H, wq, 128)
                      : make_tmap_plain(&a.tq, q_bf16, (uint64_t)2 * D, Sq, (uint64_t)B * H, 128);
  if (!tq_ok || !make_tmap(&a.tk, k->codes, rbq, Sk, (uint64_t)B * Hkv, wq, 128) ||
      !make_tmap(&a.tv, v->codes, rbv_total, D, (uint64_t)B * Hkv, wv, D) ||
      !make_tmap_out(&a.to, out, D, Sq, (uint64_t)B * H, persistent, bf16))
    return FSA_ERR_LAUNCH;
  fill_common(a.p, B, H, Hkv, Sq, Sk, causal, scale, &o, stats);
  a.p.sf_q = q ? q->scales : nullptr; a.p.sf_k = k->scales; a.p.sf_v = v->scales;
  a.q_fused = q ? 0 : 1;
  if (dbg) {
    a.dbg.s = dbg->s; a.dbg.m = dbg->m; a.dbg.p = dbg->p; a.dbg.sf = dbg->p_scales; a.dbg.row_slot = dbg->row_slot;
    a.debug = 1;
  }
  a.D = D;
  a.exp_mode = o.exp_mode;
  if (fmt_pv == FSA_FMT_E2M1_EFQ) {
    // EFQ codes need no fix when they cannot exceed 7: every block's largest residual
    // is below 3 - phi unless its exponent is clamped from above (margin <= 120 rules
    // that out), so a (3 - phi) + b < 7.49 keeps every rounded code at 7 or below
    const double top = (double)o.efq_a * (3.0 - (double)o.efq_phi) + (double)o.efq_b;
    a.exp_mode = (o.delta <= 120.0f && top < 7.49) ? 1 : 0;
  }
  a.persistent = persistent ? 1 : 0;
  a.stream = static_cast<cudaStream_t>(stream);
  const cudaError_t e = impl_for(fmt_qk, fmt_pv)(a);
  if (e == cudaErrorNotSupported) return FSA_ERR_UNSUPPORTED_FMT;
  return launch_status(e);
}

}  // namespace

extern "C" {

int fsa_attention_fwd_ex(const fsa_mx_tensor* q, const fsa_mx_tensor* k, const fsa_mx_tensor* v, void* out,
                         int B, int H, int Hkv, int Sq, int Sk, int D, int causal, float scale, int fmt_qk,
                         int fmt_pv, const fsa_opts* opts, fsa_stats* stats, void* stream) {
  if (!q) return FSA_ERR_INVALID_ARG;
  return attention_impl(q, nullptr, k, v, out, B, H, Hkv, Sq, Sk, D, causal, scale, fmt_qk, fmt_pv, opts, stats,
                        stream);
}

int fsa_attention_fwd_qbf16(const void* q_bf16, const fsa_mx_tensor* k, const fsa_mx_tensor* v, void* out, int B,
                            int H, int Hkv, int Sq, int Sk, int D, int causal, float scale, int fmt_qk, int fmt_pv,
                            const fsa_opts* opts, fsa_stats* stats, void* stream) {
  if (!q_bf16) return FSA_ERR_INVALID_ARG;
  return attention_impl(nullptr, q_bf16, k, v, out, B, H, Hkv, Sq, Sk, D, causal, scale, fmt_qk, fmt_pv, opts, stats,
                        stream);
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
      !make_tmap_out(&a.to, out, D, Sq, (uint64_t)B * H, persistent, false))
    return FSA_ERR_LAUNCH;
  fill_common(a.p, B, H, Hkv, Sq, Sk, causal, scale, &o, stats);
  a.D = D;
  a.persistent = persistent ? 1 : 0;
  a.stream = static_cast<cudaStream_t>(stream);
  return launch_status(fsa::launch_attn_impl<fsa::F_BF16, fsa::F_BF16>(a));
}

int fsa_attention_fwd_layers(const fsa_layer* layers, int n_layers, const fsa_opts* opts, void* stream) {
  if (n_layers < 0 || (n_layers > 0 && !layers)) return FSA_ERR_INVALID_ARG;
  // every layer is checked before the first launch, so an argument error enqueues nothing
  for (int l = 0; l < n_layers; ++l) {
    const fsa_layer& L = layers[l];
    if (!L.q || !L.k || !L.v || !L.out || !std::isfinite(L.delta) || L.delta < 0.0f) return FSA_ERR_INVALID_ARG;
    if (!shape_ok(L.B, L.H, L.Hkv, L.Sq, L.Sk, L.D) || !(L.scale > 0.0f) || !std::isfinite(L.scale))
      return FSA_ERR_INVALID_ARG;
    if (!valid_fmt(L.fmt_qk) || !valid_pv(L.fmt_pv)) return FSA_ERR_UNSUPPORTED_FMT;
    if (L.q->fmt != L.fmt_qk || L.k->fmt != L.fmt_qk || L.v->fmt != storage_fmt(L.fmt_pv))
      return FSA_ERR_UNSUPPORTED_FMT;
  }
  fsa_opts o;
  fsa_default_opts(&o);
  if (opts) o = *opts;
  if (o.debug) return FSA_ERR_INVALID_ARG;
  for (int l = 0; l < n_layers; ++l) {
    const fsa_layer& L = layers[l];
    o.delta = L.delta;
    o.row_fallbacks = nullptr;
    const int st = fsa_attention_fwd_ex(L.q, L.k, L.v, L.out, L.B, L.H, L.Hkv, L.Sq, L.Sk, L.D, L.causal, L.scale,
                                        L.fmt_qk, L.fmt_pv, &o, L.stats, stream);
    if (st != FSA_OK) return st;
  }
  return FSA_OK;
}

int fsa_attention_fwd_host(const fsa_host_io* host, const fsa_device_io* dev, int B, int H, int Hkv, int Sq,
                           int Sk, int D, int causal, float scale, int fmt_qk, int fmt_pv, const fsa_opts* opts,
                           fsa_stats* stats, int n_chunks, void* stream) {
  if (!host || !dev || !host->q || !host->k || !host->v || !host->out || !dev->q || !dev->k || !dev->v ||
      !dev->q_mx || !dev->k_mx || !dev->v_mx || !dev->out)
    return FSA_ERR_INVALID_ARG;
  if (!shape_ok(B, H, Hkv, Sq, Sk, D) || !(scale > 0.0f) || !std::isfinite(scale)) return FSA_ERR_INVALID_ARG;
  if (!valid_fmt(fmt_qk) || !valid_pv(fmt_pv)) return FSA_ERR_UNSUPPORTED_FMT;
  fsa_opts o;
  fsa_default_opts(&o);
  if (opts) o = *opts;
  if (!opts_ok(o) || o.debug) return FSA_ERR_INVALID_ARG;
  if (fmt_qk == FSA_FMT_NVFP4 && o.schedule == FSA_SCHED_PERSISTENT) return FSA_ERR_UNSUPPORTED_FMT;
  const int fv = storage_fmt(fmt_pv);
  const fsa_mx_tensor* mx[3] = {dev->q_mx, dev->k_mx, dev->v_mx};
  for (const fsa_mx_tensor* m : mx)
    if (!m->codes || !m->scales || !aligned16(m->codes) || !aligned16(m->scales)) return FSA_ERR_INVALID_ARG;
  if (!aligned16(dev->q) || !aligned16(dev->k) || !aligned16(dev->v) || !aligned16(dev->out))
    return FSA_ERR_INVALID_ARG;
  // bytes of one head of each MX tensor (the layouts keep every head contiguous)
  size_t qc, qs, kc, ks, vc, vs;
  int st;
  if ((st = fsa_mx_sizes(1, 1, Sq, D, FSA_MX_ROWS, fmt_qk, &qc, &qs)) != FSA_OK) return st;
  if ((st = fsa_mx_sizes(1, 1, Sk, D, FSA_MX_ROWS, fmt_qk, &kc, &ks)) != FSA_OK) return st;
  if ((st = fsa_mx_sizes(1, 1, Sk, D, FSA_MX_COLS_T, fv, &vc, &vs)) != FSA_OK) return st;
  const int G = H / Hkv, U = B * Hkv;               // kv-head units: a kv head and its G query heads
  // default: up to 8 groups, but each group's launch keeps at least two query tiles
  // per SM (a short call split 8 ways would leave SMs idle in every group)
  int n = n_chunks <= 0 ? std::min(U, 8) : std::min(n_chunks, U);
  if (n_chunks <= 0) {
    int dev = 0, n_sm = 152;
    if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev);
    const int64_t qtiles = (int64_t)B * H * ((Sq + 127) / 128);
    n = (int)std::max<int64_t>(1, std::min<int64_t>(n, qtiles / (2 * (int64_t)std::max(n_sm, 1))));
  }
  const size_t qe = (size_t)Sq * D, ke = (size_t)Sk * D;   // elements of one head
  const size_t oes = o.out_dtype == FSA_OUT_BF16 ? 2 : 4;

  cudaStream_t s = static_cast<cudaStream_t>(stream), in_s = nullptr, out_s = nullptr;
  std::vector<cudaEvent_t> ev;                      // every event made here, destroyed at the end
  auto event = [&](cudaEvent_t* e) -> bool {
    if (cudaEventCreateWithFlags(e, cudaEventDisableTiming) != cudaSuccess) return false;
    ev.push_back(*e);
    return true;
  };
  int rc = FSA_OK;
  cudaEvent_t e0;
  if (cudaStreamCreateWithFlags(&in_s, cudaStreamNonBlocking) != cudaSuccess ||
      cudaStreamCreateWithFlags(&out_s, cudaStreamNonBlocking) != cudaSuccess || !event(&e0) ||
      cudaEventRecord(e0, s) != cudaSuccess || cudaStreamWaitEvent(in_s, e0, 0) != cudaSuccess ||
      cudaStreamWaitEvent(out_s, e0, 0) != cudaSuccess)
    rc = FSA_ERR_LAUNCH;
  // copies in, chunk by chunk, on their own stream: they run ahead of the compute
  std::vector<cudaEvent_t> landed(n, nullptr);
  for (int c = 0; rc == FSA_OK && c < n; ++c) {
    const size_t u0 = (size_t)U * c / n, u1 = (size_t)U * (c + 1) / n;
    const size_t nq = (u1 - u0) * G * qe, nk = (u1 - u0) * ke;
    const size_t oq = u0 * G * qe, ok = u0 * ke;
    if (cudaMemcpyAsync(static_cast<uint16_t*>(dev->q) + oq, static_cast<const uint16_t*>(host->q) + oq, 2 * nq,
                        cudaMemcpyDefault, in_s) != cudaSuccess ||
        cudaMemcpyAsync(static_cast<uint16_t*>(dev->k) + ok, static_cast<const uint16_t*>(host->k) + ok, 2 * nk,
                        cudaMemcpyDefault, in_s) != cudaSuccess ||
        cudaMemcpyAsync(static_cast<uint16_t*>(dev->v) + ok, static_cast<const uint16_t*>(host->v) + ok, 2 * nk,
                        cudaMemcpyDefault, in_s) != cudaSuccess ||
        !event(&landed[c]) || cudaEventRecord(landed[c], in_s) != cudaSuccess)
      rc = FSA_ERR_LAUNCH;
  }
  // compute on the caller's stream as each chunk lands; its output goes back on the
  // third stream while the next chunk computes
  for (int c = 0; rc == FSA_OK && c < n; ++c) {
    const size_t u0 = (size_t)U * c / n, u1 = (size_t)U * (c + 1) / n;
    const int nu = (int)(u1 - u0);
    const size_t oq = u0 * G * qe, ok = u0 * ke;
    fsa_mx_tensor cq = *dev->q_mx, ck = *dev->k_mx, cv = *dev->v_mx;
    cq.codes = static_cast<uint8_t*>(cq.codes) + u0 * G * qc; cq.scales += u0 * G * qs;
    ck.codes = static_cast<uint8_t*>(ck.codes) + u0 * kc;     ck.scales += u0 * ks;
    cv.codes = static_cast<uint8_t*>(cv.codes) + u0 * vc;     cv.scales += u0 * vs;
    fsa_opts oc = o;
    if (o.row_fallbacks) oc.row_fallbacks = o.row_fallbacks + u0 * G * Sq;
    void* out_c = static_cast<uint8_t*>(dev->out) + oq * oes;
    cudaEvent_t done;
    if (cudaStreamWaitEvent(s, landed[c], 0) != cudaSuccess) { rc = FSA_ERR_LAUNCH; break; }
    // the chunk's kv-head units as one batch of nu kv heads and nu * G query heads
    if ((rc = fsa_mx_quantize_qkv(static_cast<uint16_t*>(dev->q) + oq, static_cast<uint16_t*>(dev->k) + ok,
                                  static_cast<uint16_t*>(dev->v) + ok, 1, nu * G, nu, Sq, Sk, D, fmt_qk, fv, &cq, &ck,
                                  &cv, s)) != FSA_OK)
      break;
    if ((rc = fsa_attention_fwd_ex(&cq, &ck, &cv, out_c, 1, nu * G, nu, Sq, Sk, D, causal, scale, fmt_qk, fmt_pv, &oc,
                                   stats, s)) != FSA_OK)
      break;
    if (!event(&done) || cudaEventRecord(done, s) != cudaSuccess || cudaStreamWaitEvent(out_s, done, 0) != cudaSuccess ||
        cudaMemcpyAsync(static_cast<uint8_t*>(host->out) + oq * oes, out_c, nu * G * qe * oes, cudaMemcpyDefault,
                        out_s) != cudaSuccess) {
      rc = FSA_ERR_LAUNCH;
      break;
    }
  }
  // the caller's stream completes after everything enqueued here, whatever failed
  cudaEvent_t fin_in, fin_out;
  if (in_s && event(&fin_in) && cudaEventRecord(fin_in, in_s) == cudaSuccess) cudaStreamWaitEvent(s, fin_in, 0);
  else if (in_s) rc = FSA_ERR_LAUNCH;
  if (out_s && event(&fin_out) && cudaEventRecord(fin_out, out_s) == cudaSuccess) cudaStreamWaitEvent(s, fin_out, 0);
  else if (out_s) rc = FSA_ERR_LAUNCH;
  // streams and events are released once their work completes
  for (cudaEvent_t e : ev) cudaEventDestroy(e);
  if (in_s) cudaStreamDestroy(in_s);
  if (out_s) cudaStreamDestroy(out_s);
  if (rc == FSA_OK) {
    auto set = [&](fsa_mx_tensor* m, int fmt, int layout, int h, int S) {
      m->fmt = fmt; m->layout = layout; m->B = B; m->H = h; m->S = S; m->D = D;
    };
    set(dev->q_mx, fmt_qk, FSA_MX_ROWS, H, Sq);
    set(dev->k_mx, fmt_qk, FSA_MX_ROWS, Hkv, Sk);
    set(dev->v_mx, fv, FSA_MX_COLS_T, Hkv, Sk);
  }
  return rc;
}

int fsa_tune_delta(const fsa_stats* stats, int n_layers, float target_rate, float step, float max_delta,
                   float* delta) {
  if (n_layers < 0 || (n_layers > 0 && (!stats || !delta)) || !(target_rate >= 0.0f) || !(step > 0.0f) ||
      !std::isfinite(step) || !(max_delta >= 0.0f) || !std::isfinite(max_delta))
    return FSA_ERR_INVALID_ARG;
  for (int l = 0; l < n_layers; ++l)
    if (!std::isfinite(delta[l]) || delta[l] < 0.0f || delta[l] > max_delta) return FSA_ERR_INVALID_ARG;
  for (int l = 0; l < n_layers; ++l) {
    if (stats[l].status != FSA_OK || stats[l].row_tiles == 0) continue;   // no evidence from this layer
    const double rate = (double)stats[l].fallback_events / (double)stats[l].row_tiles;
    if (rate > (double)target_rate) delta[l] = std::min(max_delta, delta[l] + step);
  }
  return FSA_OK;
}

int fsa_mma_peak(int kind, int n, int n_ctas, long long iters, int32_t* status, double* flops, void* stream) {
  if (kind < 0 || kind > 3 || (n != 128 && n != 256) || n_ctas <= 0 || n_ctas > 65535 || iters <= 0 ||
      iters > (1ll << 40))
    return FSA_ERR_INVALID_ARG;
  if (flops) *flops = fsa::mma_peak_flops_per_iter(kind, n) * (double)iters * (double)n_ctas;
  return launch_status(fsa::launch_mma_peak(kind, n, n_ctas, iters, status, 2000000000ull,
                                            static_cast<cudaStream_t>(stream)));
}

}  // extern "C"
