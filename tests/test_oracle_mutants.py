"""Plants plausible mistakes in a temporary copy of the oracle (CPU only) and
checks that the pins in test_oracle_pins.py catch every one of them."""
import os
import subprocess
import sys
import tempfile

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "moe_oracle.c")

# (name, exact text in moe_oracle.c, replacement)
MUTANTS = [
    ("nibble order swapped", "(c % 2 == 0) ? (byte & 15) : (byte >> 4)", "(c % 2 == 0) ? (byte >> 4) : (byte & 15)"),
    ("E2M1 exponent bias", "ldexp(1.0 + 0.5 * m, e - 1)", "ldexp(1.0 + 0.5 * m, e - 2)"),
    ("E2M1 sign dropped", "return s ? -mag : mag;", "return mag;"),
    ("E8M0 bias off by one", "ldexp(1.0, byte - 127)", "ldexp(1.0, byte - 128)"),
    ("scale block index", "sr[c / 32]", "sr[c / 16 % (K / 32)]"),
    ("router W transposed", "load_val(w, w_dtype, (size_t)e * d + i)", "load_val(w, w_dtype, (size_t)i * E + e)"),
    ("router bias dropped", "if (bias) s += (double)bias[e];", ""),
    ("tie goes to higher index", "l[e] > l[best]", "l[e] >= l[best]"),
    ("gates not renormalised", "- lmax) / den;", "- lmax);"),
    ("bucketing not stable", "for (int p = 0; p < P; ++p) pair_ids[fill[topk_idx[p]]++] = p;",
     "for (int p = P - 1; p >= 0; --p) pair_ids[fill[topk_idx[p]]++] = p;"),
    ("SwiGLU gate term dropped", "return g * sigmoid(g) * u;", "return sigmoid(g) * u;"),
    ("gate and up swapped", "h[r] = or_act(g, u, act);\n  }\n  for (int r = 0; r < d; ++r) {\n    or_mxfp4_row",
     "h[r] = or_act(u, g, act);\n  }\n  for (int r = 0; r < d; ++r) {\n    or_mxfp4_row"),
    ("down uses up matrix", "or_mxfp4_row(d_codes, d_scales, ff, r, w);", "or_mxfp4_row(u_codes, u_scales, ff, r, w);"),
    ("combine drops residual", "(x_resid ? x_resid[(size_t)t * d + i] : 0.0) + s", "s"),
    ("combine uses wrong slot", "y_pairs[((size_t)t * k + j) * d + i]", "y_pairs[((size_t)t * k + (k - 1 - j)) * d + i]"),
    ("RVQ stage dropped", "for (int s = 0; s < 3; ++s) {\n        int c", "for (int s = 0; s < 2; ++s) {\n        int c"),
    ("RVQ codebook stride", "cb[((size_t)s * 256 + c) * 8 + i]", "cb[((size_t)s * 256 + c) + i]"),
    ("RVQ codes read row-major", "codes[((size_t)s * nv + v) * rows + r]", "codes[((size_t)s * rows + r) * nv + v]"),
    ("RVQ row-major reader indexed position-major", "codes[((size_t)s * rows + r) * nv + v]",
     "codes[((size_t)s * nv + v) * rows + r]"),
    ("RVQ row-major expert reads position-major rows", "row_major ? or_rvq3_row_rowmajor : or_rvq3_row",
     "or_rvq3_row"),
    ("SiTU cap", "25.0 * tanh(u / 25.0)", "25.0 * tanh(u / 20.0)"),
    ("f16 exponent bias", "ldexp(1024.0 + m, e - 25)", "ldexp(1024.0 + m, e - 24)"),
    ("selection-only gates take the biased logits", "topk_select_gates(l, plain ? plain : l,",
     "topk_select_gates(l, l,"),
    ("shared experts dropped", "0, E + n_shared, nthreads, yp);", "0, E, nthreads, yp);"),
    ("shared expert reads a routed record", ": E + (j - k);", ": (j - k);"),
    ("shared expert weighted like a routed one", ": 1.0;", ": g[(size_t)t * k];"),
    ("projection W transposed", "load_val(w, w_dtype, (size_t)n * K + k)", "load_val(w, w_dtype, (size_t)k * N + n)"),
    ("latent residual dropped", "out[i] = load_val(x, x_dtype, i) + back[i];", "out[i] = back[i];"),
    ("latent input not rounded to bf16", "zb[i] = or_round_bf16(z[i]);", "zb[i] = or_round_bf16(z[i] * 1.001);"),
    ("bf16 ties rounded up", "fmod(m, 2.0) != 0.0", "1"),
    ("latent delta projected with the input matrix", "or_project(u, OR_F64, w_out,", "or_project(u, OR_F64, w_in,"),
    ("CRC generator not reflected", "reg ^= 0xEDB88320u;", "reg ^= 0x04C11DB7u;"),
    ("CRC register starts at zero", "uint32_t reg = 0xFFFFFFFFu;", "uint32_t reg = 0u;"),
    ("CRC result not complemented", "return reg ^ 0xFFFFFFFFu;", "return reg;"),
    ("CRC bits most significant first", "(p[i] >> b) & 1u", "(p[i] >> (7 - b)) & 1u"),
]


def _build_mutant(src_text, old, new, out_dir):
    assert src_text.count(old) >= 1, old
    mutated = src_text.replace(old, new, 1)
    c = os.path.join(out_dir, "moe_oracle.c")
    with open(c, "w") as f:
        f.write(mutated)
    hdr = os.path.join(ROOT, "oracle")
    so = os.path.join(out_dir, "libmut.so")
    subprocess.check_call(["gcc", "-O1", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared", "-I", hdr, "-o", so, c,
                           "-lm"])
    return so


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_mutant(name, old, new, tmp_path):
    with open(SRC) as f:
        src = f.read()
    so = _build_mutant(src, old, new, str(tmp_path))
    env = dict(os.environ, MOE_ORACLE_LIB=so)
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle_pins.py")], cwd=ROOT, env=env,
                       capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, f"mutant '{name}' survived the pins:\n{r.stdout[-2000:]}"
