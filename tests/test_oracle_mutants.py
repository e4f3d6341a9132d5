"""The oracle's pins catch plausible mistakes (CPU).

Each case below plants one mistake in a copy of the oracle's C source -- a
dropped term, a wrong sign, offset, bit index or byte index, a different
rounding or tie rule -- builds that copy, and runs the pin tests
(tests/test_oracle_pins.py) against it: at least one pin must fail.  The
unmodified source, built the same way, must pass them all.  The mistakes are
planted in the oracle only, on the CPU; nothing here touches the GPU path.
"""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "ggq_oracle.c")

# (name, text in the source, replacement)
MUTANTS = [
    ("q4_0 offset", "return nib - 8;", "return nib - 7;"),
    ("q4_k high scale bits from the wrong byte", "*sc = (sc12[s + 4] & 15) | ((sc12[s - 4] >> 6) << 4);",
     "*sc = (sc12[s + 4] & 15) | ((sc12[s] >> 6) << 4);"),
    ("q4_k min low bits", "*m = (sc12[s + 4] >> 4) | ((sc12[s] >> 6) << 4);",
     "*m = (sc12[s + 4] & 15) | ((sc12[s] >> 6) << 4);"),
    ("q5_k high bit index", "nib += 16 * ((b[16 + l] >> s) & 1);", "nib += 16 * ((b[16 + l] >> (s + 1)) & 1);"),
    ("q6_k offset", "return (nib | (hi << 4)) - 32;", "return (nib | (hi << 4)) - 31;"),
    ("q6_k high bits", "int hi = (qh[32 * h + l] >> (2 * g)) & 3;", "int hi = (qh[32 * h + l] >> (2 * g + 1)) & 3;"),
    ("e2m1 exponent", "ldexp(1.0 + 0.5 * m, e - 1);", "ldexp(1.0 + 0.5 * m, e);"),
    ("quantizer ties to even", "float r = roundf(v);", "float r = rintf(v);"),
    ("k-quant mins sign", "- orc_half_to_double(rd16(b + 2)) * c[1]", "+ orc_half_to_double(rd16(b + 2)) * c[1]"),
    ("k-quant mins: one bsum dropped",
     "B += m * (rds16(xb + 260 + 2 * (2 * s)) + rds16(xb + 260 + 2 * (2 * s + 1)));",
     "B += m * rds16(xb + 260 + 2 * (2 * s));"),
    ("q6_k scale index", "A += (int8_t)b[192 + g] * S;", "A += (int8_t)b[192 + (g ^ 1)] * S;"),
    ("router ties to the higher index", "if (best < 0 || l[e] > l[best]) best = e;",
     "if (best < 0 || l[e] >= l[best]) best = e;"),
    ("router without renormalisation", "for (int j = 0; j < k; ++j) weights[t * k + j] /= psel;", ""),
    ("silu sign", "return z / (1.0 + exp(-z));", "return z / (1.0 + exp(z));"),
    ("combine without the routing weight", "s += weights[t * k + j] * o[(t * k + j) * H + n];",
     "s += o[(t * k + j) * H + n];"),
    ("q8_k sub-block offset", "default: return (const int8_t*)(xrow + (j / 8) * 292 + 4 + (j % 8) * 32);",
     "default: return (const int8_t*)(xrow + (j / 8) * 292 + 4 + (j % 8) * 16);"),
    ("fp16 subnormal scale", "v = ldexp((double)m, -24);", "v = ldexp((double)m, -23);"),
    ("fp16 encode truncates", "double r = rint(ldexp(a, 11 - e));", "double r = floor(ldexp(a, 11 - e));"),
    ("mxfp4 dequant scale", "out[i] = ldexp((double)q, (int)b[0] - 128);", "out[i] = ldexp((double)q, (int)b[0] - 127);"),
    ("q4_k dequant mins sign", "out[i] = orc_half_to_double(rd16(b)) * sc * q - orc_half_to_double(rd16(b + 2)) * m;",
     "out[i] = orc_half_to_double(rd16(b)) * sc * q + orc_half_to_double(rd16(b + 2)) * m;"),
    ("q6_k dequant scale group", "(int8_t)b[192 + i / 16] * q; break;", "(int8_t)b[192 + i / 32] * q; break;"),
    ("q8_1 s without d", "float s = d * (float)sum;", "float s = (float)sum;"),
    ("q8_0 activation scale from the wrong block", "case ORC_Q8_0: return orc_half_to_double(rd16(xrow + j * 34));",
     "case ORC_Q8_0: return orc_half_to_double(rd16(xrow + (j ^ 1) * 34));"),
    ("q8_0 activation quants shifted", "case ORC_Q8_0: return (const int8_t*)(xrow + j * 34 + 2);",
     "case ORC_Q8_0: return (const int8_t*)(xrow + j * 34 + 1);"),
    ("q8_k bsums over 8", "for (int i = 0; i < 16; ++i) s += q[16 * g + i];",
     "for (int i = 0; i < 8; ++i) s += q[16 * g + i];"),
    ("q2_k bit pair", "return (b[16 + 32 * n + l] >> (2 * j)) & 3;", "return (b[16 + 32 * n + l] >> (2 * j + 1)) & 3;"),
    ("q2_k half offset", "return (b[16 + 32 * n + l] >> (2 * j)) & 3;", "return (b[16 + 16 * n + l] >> (2 * j)) & 3;"),
    ("q2_k min from the scale nibble", "(b[i / 16] >> 4);\n", "(b[i / 16] & 15);\n"),
    ("q2_k integer mins dropped", "B += (b[g] >> 4) * rds16(xb + 260 + 2 * g);", ""),
    ("q3_k high bit index", "int hbit = (b[l] >> (4 * n + j)) & 1;", "int hbit = (b[l] >> (4 * j + n)) & 1;"),
    ("q3_k high bit sense", "return lo - (hbit ? 0 : 4);", "return lo - (hbit ? 4 : 0);"),
    ("q3_k scale high bits", "int hi = (sc12[8 + s % 4] >> (2 * (s / 4))) & 3;", "int hi = (sc12[8 + s / 4] >> (2 * (s % 4))) & 3;"),
    ("q3_k scale offset", "(orc_q3k_scale(b + 96, i / 16) - 32) * q;", "(orc_q3k_scale(b + 96, i / 16) - 31) * q;"),
    ("q3_k integer scale group", "A += (orc_q3k_scale(b + 96, g) - 32) * S;", "A += (orc_q3k_scale(b + 96, g ^ 1) - 32) * S;"),
]


def _build(text, path):
    src = path + ".c"
    with open(src, "w") as f:
        f.write(text)
    r = subprocess.run(["gcc", "-O1", "-std=gnu99", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math",
                        "-fno-strict-aliasing", "-I", os.path.join(ROOT, "oracle"), src, "-o", path, "-lm"],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr[-2000:]
    return path


def _pins_pass(lib_path):
    env = dict(os.environ, GGQ_ORACLE_LIB=lib_path)
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle_pins.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    return r.returncode == 0, r.stdout[-1500:]


@pytest.fixture(scope="module")
def source():
    with open(SRC) as f:
        return f.read()


def test_unmodified_oracle_passes_the_pins(source, tmp_path):
    ok, out = _pins_pass(_build(source, str(tmp_path / "liborc_ref.so")))
    assert ok, out


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_a_planted_mistake_fails_a_pin(source, tmp_path, name, old, new):
    assert source.count(old) == 1, f"mutation site of '{name}' not found once in the oracle source"
    ok, out = _pins_pass(_build(source.replace(old, new), str(tmp_path / "liborc_mut.so")))
    assert not ok, f"no pin caught the planted mistake '{name}'"
