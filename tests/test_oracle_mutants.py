"""The pins are strong enough: each plausible mistake planted in a copy of the oracle
(on the CPU) makes at least one pin test fail."""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "rkv_oracle.c")

MUTANTS = {
    "mean divides by k, not k_i": ("s / (double)ki", "s / 4.0"),
    "ties go to the higher slot": ("return (a->slot > b->slot) - (a->slot < b->slot);",
                                   "return (a->slot < b->slot) - (a->slot > b->slot);"),
    "Swish on the second projection": ("hv[f] = rkvo_swish(a1) * a2;", "hv[f] = a1 * rkvo_swish(a2);"),
    "sigmoid instead of Swish": ("return u / (1.0 + exp(-u));", "return 1.0 / (1.0 + exp(-u));"),
    "round down instead of half-up": ("floor((z[c] - lo) / dl + 0.5)", "floor((z[c] - lo) / dl)"),
    "step divides by 2^b": ("double dl = (hi - lo) / (double)qmax;", "double dl = (hi - lo) / (double)(qmax + 1);"),
    "z adds the encodings": ("zz[c] = f1[c] - f2[c];", "zz[c] = f1[c] + f2[c];"),
    "pool sees later references": ("if (ref_pos[m] < t) n_pool++;", "if (ref_pos[m] < t + 8) n_pool++;"),
    "FP8 exponent bias 8": ("v = ldexp(1.0 + m / 8.0, e - 7);", "v = ldexp(1.0 + m / 8.0, e - 8);"),
    "L1 instead of squared L2": ("d += u * u;", "d += fabs(u);"),
    "W_c3 indexed transposed": ("s += hv[f] * W3t[(size_t)j * d_ff + f];", "s += hv[f] * W3t[(size_t)f * d_c + j];"),
    "dynamic stride without floor": ("p = p + s0 + (long long)floor(alpha * (double)(p - n_sink));",
                                     "p = p + s0 + (long long)ceil(alpha * (double)(p - n_sink));"),
    "dequantise without the minimum": ("zq[c] = (double)q[c] * delta[c / group] + zmin[c / group];",
                                       "zq[c] = (double)q[c] * delta[c / group];"),
    "RoPE on the value half": ("for (int h = 0; h < N; h++) rkvo_rope(ko + (size_t)h * D, D, (double)one, rope_base);",
                               "for (int h = 0; h < N; h++) rkvo_rope(vo + (size_t)h * D, D, (double)one, rope_base);"),
    "RoPE pairs half a head apart": ("double x0 = x[2 * i], x1 = x[2 * i + 1];",
                                     "double x0 = x[i], x1 = x[i + D / 2];"),
    "RoPE frequency exponent -i/D": ("double theta = pow(base, -2.0 * (double)i / (double)D);",
                                     "double theta = pow(base, -(double)i / (double)D);"),
    "RoPE rotates the other way": ("x[2 * i] = x0 * c - x1 * s;", "x[2 * i] = x0 * c + x1 * s;"),
    "decoder weights transposed": ("s += z[j] * Wd[(size_t)c * d_c + j];", "s += z[j] * Wd[(size_t)j * W + c];"),
    "keys take the value half of the decoder": ("ko[c] = dec[c] + mean[c];", "ko[c] = dec[dk + c] + mean[c];"),
    "value without the reference mean": ("vo[c] = dec[dk + c] + mean[dk + c];", "vo[c] = dec[dk + c];"),
    "attention scaled by 1/D": ("s[t] = d / sqrt((double)D);", "s[t] = d / (double)D;"),
    "query heads mapped round-robin": ("int h = j / G;", "int h = j % N;"),
    "padding rows attended": ("if (valid[t]) den += exp(s[t] - mx);", "den += exp(s[t] - mx);"),
    "attention reads keys as values": ("acc += exp(s[t] - mx) * V[(size_t)t * N * D + (size_t)h * D + c];",
                                       "acc += exp(s[t] - mx) * K[(size_t)t * N * D + (size_t)h * D + c];"),
}


@pytest.mark.parametrize("name", list(MUTANTS))
def test_pins_catch_planted_mistake(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) >= 1, "mutation site not found: " + old
    mut = tmp_path / "mutant.c"
    mut.write_text(src.replace(old, new))
    so = tmp_path / "libmutant.so"
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-o", str(so), str(mut), "-lm"])
    env = dict(os.environ, RKV_ORACLE_LIB=str(so))
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle_pins.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, "planted mistake '%s' passed every pin" % name
