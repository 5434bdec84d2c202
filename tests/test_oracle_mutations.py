"""The oracle's pins catch plausible mistakes: each case plants one mistake in
a copy of oracle/oracle.c (a dropped term, a wrong sign or index, a transposed
operand, an off-by-one threshold, ...), builds it, and runs the pin suite
against it; the pins must fail. The unmodified copy must pass. CPU only."""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "oracle.c")

# (name, original text, planted mistake)
MUTATIONS = [
    ("softmax head index", "double s = scores[e * H + h];", "double s = scores[e * H];"),
    ("softmax normaliser dropped", "out[e * H + h] = exp((double)scores[e * H + h] - m) / Z;",
     "out[e * H + h] = exp((double)scores[e * H + h] - m);"),
    ("softmax without max subtraction", "Z += exp((double)scores[e * H + h] - m);",
     "Z += exp((double)scores[e * H + h]);"),
    ("spmm gathers the destination row", "int64_t src = col_idx[e];\n            for (int32_t h = 0; h < H; ++h) {\n                double we",
     "int64_t src = i;\n            for (int32_t h = 0; h < H; ++h) {\n                double we"),
    ("spmm weight of the wrong head", "double we = w[e * H + h];", "double we = w[e * H];"),
    ("sddmm scale dropped", "out[e * H + h] = scale * acc;", "out[e * H + h] = acc;"),
    ("sddmm operands swapped in the COO form", "int64_t t = row_ptr ? r : dst_idx[e];",
     "int64_t t = row_ptr ? r : src_idx[e];"),
    ("fused score sign", "s[e - e0] = scale * acc;", "s[e - e0] = -scale * acc;"),
    ("fused weights not normalised", "double w = exp(s[e - e0] - m) / Z;",
     "double w = exp(s[e - e0] - m);"),
    ("fused value of the wrong source", "double val = elem(v, dtype, src * HD + (int64_t)h * Dh + d);",
     "double val = elem(v, dtype, i * HD + (int64_t)h * Dh + d);"),
    ("LayerNorm unbiased variance", "            var /= D;", "            var /= (D - 1);"),
    ("LayerNorm without beta", "* rstd * ln_w[d] + ln_b[d];", "* rstd * ln_w[d];"),
    ("SiLU sign", "hid[p] = a / (1.0 + exp(-a));", "hid[p] = a / (1.0 + exp(a));"),
    ("relation bias of the wrong head", "a += (double)W2[h * P + p] * hid[p];",
     "a += (double)W2[p] * hid[p];"),
    ("head slice ignored", "dot += Q[i * D + h * dh + c] * K[j * D + h * dh + c];",
     "dot += Q[i * D + c] * K[j * D + c];"),
    ("attention scale dropped", "double l = dot * inv_sqrt_dh + rel", "double l = dot + rel"),
    ("residual dropped", "o[n * D + r] = (double)x[n * D + r] + a;", "o[n * D + r] = a;"),
    ("out projection transposed", "a += (double)Wout[r * D + c] * ctx[n * D + c];",
     "a += (double)Wout[c * D + r] * ctx[n * D + c];"),
    ("plan threshold off by one", "if (d <= heavy_threshold)", "if (d < heavy_threshold)"),
    ("plan chunks rounded down", "int64_t c = (d + chunk - 1) / chunk;", "int64_t c = d / chunk;"),
    ("bf16 widened with the wrong shift", "uint32_t u = (uint32_t)bits << 16;",
     "uint32_t u = (uint32_t)bits << 15;"),
    ("backward Delta dropped", "const double ds = ae * (da[e - e0] - Delta);",
     "const double ds = ae * da[e - e0];"),
    ("backward dv weighted by the wrong factor", "dv[kj + d] += ae * gv;",
     "dv[kj + d] += da[e - e0] * gv;"),
    ("backward dk from k", "dk[kj + d] += scale * ds * qv;", "dk[kj + d] += scale * ds * kv;"),
    ("backward dq scale dropped", "dq[qi + d] += scale * ds * kv;", "dq[qi + d] += ds * kv;"),
    ("transpose counts shifted", "src_ptr[col_idx[e] + 1] += 1;", "src_ptr[col_idx[e]] += 1;"),
    ("transpose records the source as the row", "dst[k] = (int32_t)i;", "dst[k] = col_idx[e];"),
    ("e4m3 exponent bias", "v = ldexp(1.0 + (double)m / 8.0, e - 7);",
     "v = ldexp(1.0 + (double)m / 8.0, e - 8);"),
    ("e4m3 subnormal scale", "v = ldexp((double)m / 8.0, -6);", "v = ldexp((double)m / 8.0, -7);"),
    ("e4m3 ties away from zero", "if (r > 0.5 || (r == 0.5 && fmod(fl, 2.0) != 0.0))",
     "if (r >= 0.5)"),
    ("fp8 quantiser range", "volatile float sc = amax > 0.0f ? amax / 448.0f : 1.0f;",
     "volatile float sc = amax > 0.0f ? amax / 240.0f : 1.0f;"),
    ("fp8 fused layer v scaled by k's scale", "(double)vs[src * H + h];", "(double)ks[src * H + h];"),
    ("backward da against k", "dd += elem(dout, dtype, qi + d) * elem(v, dtype, kj + d);",
     "dd += elem(dout, dtype, qi + d) * elem(k, dtype, kj + d);"),
]


def _build(src_text, tmp_path, tag):
    c = tmp_path / f"oracle_{tag}.c"
    so = tmp_path / f"liboracle_{tag}.so"
    c.write_text(src_text)
    subprocess.run(["gcc", "-std=c11", "-O2", "-fno-fast-math", "-ffp-contract=off", "-fPIC",
                    "-shared", "-o", str(so), str(c), "-lm"], check=True)
    return str(so)


def _run_pins(lib_path):
    env = dict(os.environ, GAT_ORACLE_LIB=lib_path)
    r = subprocess.run([sys.executable, "-m", "pytest", os.path.join(ROOT, "tests", "test_oracle_pins.py"),
                        "-x", "-q", "-p", "no:cacheprovider"], cwd=ROOT, env=env,
                       capture_output=True, text=True, timeout=600)
    return r.returncode, r.stdout[-2000:]


def test_unmodified_copy_passes(tmp_path):
    rc, out = _run_pins(_build(open(SRC).read(), tmp_path, "orig"))
    assert rc == 0, out


@pytest.mark.parametrize("name,orig,bad", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_pins_catch_planted_mistake(tmp_path, name, orig, bad):
    src = open(SRC).read()
    assert src.count(orig) >= 1, f"mutation anchor not found: {orig!r}"
    rc, out = _run_pins(_build(src.replace(orig, bad, 1), tmp_path, "mut"))
    assert rc != 0, f"no pin caught: {name}\n{out}"
