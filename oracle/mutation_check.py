"""Mutation check of the oracle's CPU pins.

Plants one plausible mistake at a time (a wrong bias, rounding mode, clamp,
index, block size, sign, missing term...) in a copy of fsa_oracle.c and runs the
oracle tests (tests/test_oracle_*.py) against that copy.  A mistake the pins
miss is reported as SURVIVED.  One entry is an equivalent mutant on purpose: the
final saturation line of orc_encode cannot be reached (below the format maximum,
round-to-nearest never rounds past it), so that mutant survives by design.

    python oracle/mutation_check.py [index ...]

Copies go to oracle/_mutants/ (ignored by git) and are removed after each run.
Developer tool: nothing in the product or the tests runs it.
"""
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
WORK = os.path.join(HERE, "_mutants")
EQUIVALENT = {"no final saturation"}

# (name, fragment of fsa_oracle.c, replacement); each fragment occurs exactly once
M = [
 ("e4m3 bias", "f.bias = 7;", "f.bias = 8;"),
 ("e2m3 max", "f.maxv = 7.5;", "f.maxv = 7.0;"),
 ("e3m2 bias", "f.ebits = 3; f.mbits = 2; f.bias = 3;", "f.ebits = 3; f.mbits = 2; f.bias = 2;"),
 ("e3m2 emax", "return fmt == 0 ? 8 : (fmt == 4 ? 4 : 2);", "return fmt == 0 ? 8 : 2;"),
 ("subnormal decode", "ldexp((double)m, 1 - f.bias - f.mbits)", "ldexp((double)m, -f.bias - f.mbits)"),
 ("ties away", "nearbyint(a / q) * q", "round(a / q) * q"),
 ("no final saturation", "    if (v > f.maxv) v = f.maxv;\n", ""),
 ("zero loses sign", "  if (v == 0.0) return sbit;", "  if (v == 0.0) return 0;"),
 ("mx E off by one", "        E = (ex - 1) - emax;\n        if (E < -127) E = -127;\n        if (E > 127) E = 127;\n      }\n      scales", "        E = ex - emax;\n        if (E < -127) E = -127;\n        if (E > 127) E = 127;\n      }\n      scales"),
 ("mx clamp -126", "        if (E < -127) E = -127;\n        if (E > 127) E = 127;\n      }\n      scales", "        if (E < -126) E = -126;\n        if (E > 127) E = 127;\n      }\n      scales"),
 ("mx zero block E=0", "      if (amax == 0.0) {\n        E = -127;", "      if (amax == 0.0) {\n        E = 0;"),
 ("nonfinite scale", "scales[r * scales_stride + b] = 0xFF;", "scales[r * scales_stride + b] = 0x7F;"),
 ("gqa mapping", "*kvh = *h / (g->H / g->Hkv);", "*kvh = *h % g->Hkv;"),
 ("causal offset", "int lim = i + g->Sk - g->Sq;", "int lim = i;"),
 ("exact no scale", "s[j] = scale * acc;", "s[j] = acc;"),
 ("exact no normalise", "o[d] = acc / l;", "o[d] = acc;"),
 ("floor exp2 for exp", "for (int j = 0; j < nk; ++j) p[j] = exp(p[j] - m);", "for (int j = 0; j < nk; ++j) p[j] = exp2(p[j] - m);"),
 ("floor blocks of 16", "for (int jb = 0; jb < nk; jb += 32) {\n          int je = jb + 32 < nk ? jb + 32 : nk;", "for (int jb = 0; jb < nk; jb += 16) {\n          int je = jb + 16 < nk ? jb + 16 : nk;"),
 ("floor P emax+1", "            E = (ex - 1) - emax;\n            if (E < -127) E = -127;\n            if (E > 127) E = 127;\n          }\n          for (int j = jb", "            E = ex - emax;\n            if (E < -127) E = -127;\n            if (E > 127) E = 127;\n          }\n          for (int j = jb"),
 ("poly nodes", "double x[4] = {0.0, 1.0 / 3.0, 2.0 / 3.0, 1.0};", "double x[4] = {0.0, 0.3, 0.7, 1.0};"),
 ("poly no 2^n", "  return ldexpf(p, (int)n);\n}\n\n/* ---", "  return p;\n}\n\n/* ---"),
 ("emu c without log2e", "const float c = (float)((double)scale * 1.4426950408889634073599246810018921);  /* log2(e) */", "const float c = scale;"),
 ("emu M = x + delta", "          if (!M_set) {\n            M = x;", "          if (!M_set) {\n            M = x + opt->delta;"),
 ("emu no margin", "            if (x > M + opt->delta) {", "            if (x > M) {"),
 ("emu fallback keeps l", "              l *= alpha;\n              if (A) {", "              if (A) {"),
 ("emu alpha sign", "double alpha = exp2((double)(M - Mn));", "double alpha = exp2((double)(Mn - M));"),
 ("emu E +1", "            int E = (int)floorf(tmax + phi) - emax;", "            int E = (int)floorf(tmax + phi) - emax + 1;"),
 ("emu r without E", "              float r = fmaf(s[j - j0], c, -bE);", "              float r = fmaf(s[j - j0], c, -M);"),
 ("efq slope from c only", "  const float a_c = opt->efq_a * c;               /* EFQ: fp32(a c) */", "  const float a_c = c;"),
 ("efq clamp 6", "                if (kk > 7.0) kk = 7.0;\n                code", "                if (kk > 6.0) kk = 6.0;\n                code"),
 ("efq floor", "double kk = nearbyint((double)y);                 /* ties to even */", "double kk = floor((double)y);"),
 ("emu pt scale", "              pt[j - j0] = orc_decode(efmt, used) * sc;", "              pt[j - j0] = orc_decode(efmt, used) * sc * 2.0;"),
 ("emu mask inverted", "int hw = (opt->mufu_mask >> (j % 32)) & 1;", "int hw = !((opt->mufu_mask >> (j % 32)) & 1);"),
 ("emu tiles of 64", "  const int D = g->D, BN = 128;\n  const int64_t Skp", "  const int D = g->D, BN = 64;\n  const int64_t Skp"),
 ("bf16 tau 0", "else if (x - M > tau) {", "else if (x - M > 0.0f) {"),
 ("bf16 round ties away", "u = (u + 0x7FFFu + lsb) & 0xFFFF0000u;", "u = (u + 0x8000u) & 0xFFFF0000u;"),
 ("v transposed stride", "op->vc[vrow * Skp + j]", "op->vc[vrow * g->Sk + j]"),
 ("mx qk scale index", "return deq(fmt, codes[d], scales[d / 32]);", "return deq(fmt, codes[d], scales[d / 64]);"),
 ("emu ignores causal", "      int nk = last_visible(g, i) + 1;\n      double* o = out + n * D;\n      for (int d = 0; d < D; ++d) o[d] = 0.0;\n      int fb = 0", "      int nk = g->Sk;\n      double* o = out + n * D;\n      for (int d = 0; d < D; ++d) o[d] = 0.0;\n      int fb = 0"),
 ("emu normalise +1", "        for (int d = 0; d < D; ++d) o[d] = l > 0.0 ? o[d] / l : 0.0;\n        if (A) {", "        for (int d = 0; d < D; ++d) o[d] = l > 0.0 ? o[d] / (l + 1.0) : 0.0;\n        if (A) {"),
 ("emu tmax from M", "            float tmax = smax * c - M;", "            float tmax = 0.0f;"),
 ("emu block max wrong", "            for (int j = jb; j < je; ++j) if (s[j - j0] > smax) smax = s[j - j0];\n            float tmax", "            smax = s[jb - j0];\n            float tmax"),
 ("k scale row", "op->kc + krow * D, op->ks + krow * nb, D, d)", "op->kc + krow * D, op->ks, D, d)"),
 ("nvfp4 scale index", "orc_decode(0, scales[d / 16])", "orc_decode(0, scales[d / 32])"),
 ("nvfp4 scale from amax/4", "orc_encode(0, amax / 6.0)", "orc_encode(0, amax / 4.0)"),
 ("nvfp4 codes times scale", "orc_encode(2, xv[i] / sv)", "orc_encode(2, xv[i] * sv)"),
 ("nvfp4 nan scale byte", "scales[r * scales_stride + b] = 0x7F;", "scales[r * scales_stride + b] = 0x7E;"),
 ("nvfp4 pads with ones", "int64_t idx = b * 16 + i;\n        xv[i] = idx < len ? bf16_to_double(x[r * row_stride + idx * elem_stride]) : 0.0;",
  "int64_t idx = b * 16 + i;\n        xv[i] = idx < len ? bf16_to_double(x[r * row_stride + idx * elem_stride]) : 1.0;"),
 ("v scale index", "op->vs[vrow * (Skp / 32) + j / 32]", "op->vs[vrow * (Skp / 32)]"),
 ("mx pads with ones", "int64_t idx = b * 32 + i;\n        xv[i] = idx < len ? bf16_to_double(x[r * row_stride + idx * elem_stride]) : 0.0;",
  "int64_t idx = b * 32 + i;\n        xv[i] = idx < len ? bf16_to_double(x[r * row_stride + idx * elem_stride]) : 1.0;"),
 ("groups by batch only", "k[n].key = (int64_t)b * g->Hkv + kvh;", "k[n].key = (int64_t)b;"),
 ("exact v from k", "kv->vh[(int64_t)d * nk + j] = bf16_to_double(v[base + (int64_t)j * D + d]);",
  "kv->vh[(int64_t)d * nk + j] = bf16_to_double(k[base + (int64_t)j * D + d]);"),
 ("ambiguity too small", "#define AMB_S 4.76837158203125e-07   /* 2^-21 */", "#define AMB_S 1e-9"),
 ("tiles not counted", "          ++tv;\n", ""),
 ("fallbacks not counted", "              ++fb;\n", ""),
 ("efq beta sign", "float Bk = opt->beta - opt->efq_a * bE;", "float Bk = -opt->beta - opt->efq_a * bE;"),
 ("efq offset without E", "float Bk = opt->beta - opt->efq_a * bE;", "float Bk = opt->beta - opt->efq_a * M;"),
 ("efq phi ignored", "  const float phi = efq ? opt->phi : 0.0f;", "  const float phi = 0.0f;"),
 ("phi on the exp path", "  const float phi = efq ? opt->phi : 0.0f;", "  const float phi = opt->phi;"),
 ("efq codes not clamped below", "                if (!(kk > 0.0)) kk = 0.0;", ""),
 ("bf16 rescale keeps l", "            l *= alpha;\n            M = x;", "            M = x;"),
 ("exact no max shift", "        if (s[j] > m) m = s[j];\n      }\n      double l = 0.0;",
  "        m = 0.0;\n      }\n      double l = 0.0;"),
 ("amb ignores fallback test", "<= dx + dM + rt * fabs(thr) && rt > 0.0) undetermined = 1;", "< 0.0) undetermined = 1;"),
 ("given codes ignored", "const uint32_t used = (dump && dump->p_in) ? dump->p_in[n * Skp + j] : code;",
  "const uint32_t used = code;"),
 ("given scores ignored", "            s[j - j0] = (dump && dump->s_in) ? dump->s_in[n * Skp + j] : (float)(acc * (1.0 + opt->s_perturb));",
  "            s[j - j0] = (float)(acc * (1.0 + opt->s_perturb));"),
 ("amb alpha exact", "const double ra = 0.6931471805599453 * (dM + dx) + AMB_X;", "const double ra = 0.0;"),
 ("amb block exponent", "if (Elo != Ehi && Ehi - emax > -127 && Elo - emax < 127) blk_undet = 1;", "blk_undet = 0;"),
 ("amb block step", "dp = 0.25 * pt[j - j0] + orc_decode(efmt, 1) * sc * 2.0;", "dp = 0.0;"),
 ("e4m3 no nan", "  if (fmt == 0 && e == 15 && m == 7) return NAN;\n", ""),
 ("nan loses sign", "if (isnan(x)) return fmt == 0 ? (sbit | 0x7F) : sbit;", "if (isnan(x)) return fmt == 0 ? 0x7F : sbit;"),
 ("subnormal quantum", "int emin = 1 - f.bias;                       /* exponent of the smallest normal */",
  "int emin = -f.bias;"),
 ("nonfinite codes", "c[i] = (uint8_t)(fmt == 0 ? 0x7F : 0);", "c[i] = (uint8_t)0x7F;"),
]


def run(selected):
    src = open(os.path.join(HERE, "fsa_oracle.c")).read()
    survivors = []
    for idx, (name, old, new) in enumerate(M):
        if selected and idx not in selected:
            continue
        if src.count(old) != 1:
            print(f"{idx:2d} {name:24s} fragment occurs {src.count(old)} times")
            survivors.append(name)
            continue
        d = os.path.join(WORK, f"run{idx:02d}")
        shutil.rmtree(d, ignore_errors=True)
        os.makedirs(d)
        shutil.copytree(HERE, os.path.join(d, "oracle"),
                        ignore=shutil.ignore_patterns("_build", "_mutants", "__pycache__"))
        shutil.copytree(os.path.join(ROOT, "tests"), os.path.join(d, "tests"),
                        ignore=shutil.ignore_patterns("__pycache__"))
        shutil.copy(os.path.join(ROOT, "workloads.py"), d)
        with open(os.path.join(d, "oracle", "fsa_oracle.c"), "w") as f:
            f.write(src.replace(old, new))
        tests = sorted(os.path.join("tests", t) for t in os.listdir(os.path.join(d, "tests"))
                       if t.startswith("test_oracle_"))
        r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider", *tests], cwd=d,
                           capture_output=True, text=True, env=dict(os.environ, PYTHONPATH=d), timeout=1800)
        shutil.rmtree(d, ignore_errors=True)
        caught = r.returncode != 0
        tag = "caught" if caught else ("survived (equivalent)" if name in EQUIVALENT else "SURVIVED")
        print(f"{idx:2d} {name:24s} {tag}", flush=True)
        if not caught and name not in EQUIVALENT:
            survivors.append(name)
    shutil.rmtree(WORK, ignore_errors=True)
    return survivors


if __name__ == "__main__":
    left = run({int(a) for a in sys.argv[1:]})
    print("all non-equivalent mutants caught" if not left else f"missed: {left}")
    sys.exit(1 if left else 0)
