"""Mutation check of the oracle's pins.  Each case plants one plausible
mistake in a copy of oracle/oracle.cpp -- a dropped term, a wrong sign, a
transposed operand, a wrong index, order or constant -- builds the copy
and runs the pins (tests/test_oracle_pins.py, test_oracle_mixed.py)
against it: at least one pin must fail.  CPU only; the planted mistakes live in temporary copies and
never touch the oracle itself or the product."""
import os
import shutil
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "oracle.cpp")

# (what the mistake is, text in oracle.cpp, what it becomes); the first
# occurrence of the text is changed -- the 1-bit functions come first in
# the file, the mixed-width codecs later
MUTATIONS = [
    ("momentum betas swapped",
     "float mw = (b1 * m[k]) + (ob1 * g[k]);", "float mw = (ob1 * m[k]) + (b1 * g[k]);"),
    ("worker error not added",
     "float xv = (s * mw) + (r * e[k]);", "float xv = (s * mw);"),
    ("sigma not applied",
     "float xv = (s * mw) + (r * e[k]);", "float xv = mw + (r * e[k]);"),
    ("rho not applied to the worker error",
     "float xv = (s * mw) + (r * e[k]);", "float xv = (s * mw) + e[k];"),
    ("sign of zero negative",
     "bool b = (xv >= 0.0f);", "bool b = (xv > 0.0f);"),
    ("bits MSB first",
     "if (b) bits[k >> 5] |= (1u << (k & 31));", "if (b) bits[k >> 5] |= (1u << (31 - (k & 31)));"),
    ("worker error sign flipped",
     "e[k] = xv - (scale * sg);", "e[k] = xv + (scale * sg);"),
    ("scale over the padded chunk length",
     "float scale = real ? sum / (float)real : 0.0f;", "float scale = real ? sum / (float)len : 0.0f;"),
    ("server sum not divided by W",
     "      z = z / fW;\n", "      (void)fW;\n"),
    ("server error not added",
     "ys[q] = (r * e_s[k]) + z;", "ys[q] = z;"),
    ("server error sign flipped",
     "e_s[k] = ys[q] - (sscale * (b ? 1.0f : -1.0f));",
     "e_s[k] = ys[q] + (sscale * (b ? 1.0f : -1.0f));"),
    ("Adam step direction flipped",
     "p[k] = p[k] - t;", "p[k] = p[k] + t;"),
    ("eps inside the square root",
     "float d = std::sqrt(v[k]);\n      d = d + eps;", "float d = std::sqrt(v[k] + eps);"),
    ("LAMB gradient not divided by (1 - b1)",
     "float gt = (mt - (b1 * m[k])) / ob1;", "float gt = (mt - (b1 * m[k]));"),
    ("LAMB ratio inverted",
     "float ratio = v_frozen[k] / vt;", "float ratio = vt / v_frozen[k];"),
    ("LAMB ratio clip band too wide",
     "float lo = (1.0f - r_thr) * r_prev[l];", "float lo = (1.0f - 2.0f * r_thr) * r_prev[l];"),
    ("LAMB coefficient history not shifted",
     "c_prev2[l] = c_prev[l];", "c_prev2[l] = c_prev2[l];"),
    ("rho inverted",
     "rho[l] = c_prev2[l] / c_prev[l];", "rho[l] = c_prev[l] / c_prev2[l];"),
    ("pass B without the coefficient",
     "float t1 = lr * c[l];", "float t1 = lr;"),
    ("warmup gradients not averaged",
     "    gb = gb / fW;\n", "    (void)fW;\n"),
    ("canonical sum in lane-contiguous order",
     "uint64_t idx = (uint64_t)(1024 * i + 4 * p + c);",
     "uint64_t idx = (uint64_t)(16 * p + 4 * i + c);"),
    ("INT8 scale over 128",
     "float scale = mx / 127.0f;", "float scale = mx / 128.0f;"),
    ("INT8 rounding comparison not strict",
     "float qf = f + ((u < frac) ? 1.0f : 0.0f);", "float qf = f + ((u <= frac) ? 1.0f : 0.0f);"),
    ("Philox key schedule constant",
     "k1 += 0xBB67AE85u;", "k1 += 0xBB67AE86u;"),
    ("uniform from the low bits",
     "return (float)(wd >> 8) * (1.0f / 16777216.0f);",
     "return (float)(wd & 0xFFFFFFu) * (1.0f / 16777216.0f);"),
    ("Philox multiplier constant",
     "uint64_t p0 = (uint64_t)0xD2511F53u * (uint64_t)c0;",
     "uint64_t p0 = (uint64_t)0xD2511F55u * (uint64_t)c0;"),
    ("LAMB fresh variance with b2 and 1 - b2 swapped",
     "float vt = (b2 * v_fresh[k]) + (ob2 * (gt * gt));",
     "float vt = (ob2 * v_fresh[k]) + (b2 * (gt * gt));"),
    ("LAMB momentum not divided by sigma",
     "float mt = M / sigma[l];", "float mt = M;"),
    ("clip of the compensated value with the wrong sign",
     "if (xv < -clip) xv = -clip;", "if (xv < -clip) xv = clip;"),
    ("canonical sum pairs warps 0+2, 1+3",
     "float s01 = warp[0] + warp[1], s23 = warp[2] + warp[3];",
     "float s01 = warp[0] + warp[2], s23 = warp[1] + warp[3];"),
    ("LAMB ratio clipped to r_min from above",
     "r = fmin_plain(fmax_plain(r, r_min), r_max);", "r = fmin_plain(fmax_plain(r, r_min), r_min);"),
    ("LAMB coefficient not clipped above",
     "c = fmin_plain(fmax_plain(c, c_min), c_max);", "c = fmax_plain(c, c_min);"),
    ("sigma inverted at the end of warmup",
     "s[l] = (rms[l] == 0.0f) ? 1.0f : mean / rms[l];",
     "s[l] = (rms[l] == 0.0f) ? 1.0f : rms[l] / mean;"),
    ("c_avg not divided by the warmup steps",
     "float ca = c_sum[l] / (float)warmup_steps;", "float ca = c_sum[l];"),
    ("INT8 code clamped at 128",
     "if (qf > 127.0f) qf = 127.0f;", "if (qf > 128.0f) qf = 127.0f;"),
    ("error monitor sums |e| instead of e^2",
     "for (uint64_t q = 0; q < real; ++q) sq[q] = e[start + q] * e[start + q];",
     "for (uint64_t q = 0; q < real; ++q) sq[q] = std::fabs(e[start + q]);"),
    ("error monitor takes the mean instead of the sum",
     "out[g_id] = orc_cr_sum(sq.data(), real);",
     "out[g_id] = real ? orc_cr_sum(sq.data(), real) / (float)real : 0.0f;"),
    # mixed widths: the b-bit block codec and the FP16 codec
    ("b-bit code range one too wide",
     "const float qmax = (float)((1 << (bits - 1)) - 1);",
     "const float qmax = (float)(1 << (bits - 1));"),
    ("b-bit codes not sign-extended",
     "return field >= (1 << (bits - 1)) ? field - (1 << bits) : field;", "return field;"),
    ("b-bit fields MSB first",
     "words[bit / 32] |= field << (bit % 32);", "words[bit / 32] |= field << (32 - bits - bit % 32);"),
    ("b-bit workers share their uniforms",
     "x.data(), seed, step, w * L->n_pad,", "x.data(), seed, step, 0,"),
    ("b-bit server uses worker 0's uniforms",
     "y.data(), seed, step, L->W * L->n_pad,", "y.data(), seed, step, 0,"),
    ("b-bit server sum not divided by W",
     "      z = z / fW;\n      y[i] = e_s[b0 + i] + z;", "      (void)fW;\n      y[i] = e_s[b0 + i] + z;"),
    ("b-bit error sign flipped",
     "e[i] = x[i] - (qf * scale);", "e[i] = x[i] + (qf * scale);"),
    ("binary16 ties rounded away from zero",
     "const double r = std::nearbyint(a / step);", "const double r = std::round(a / step);"),
    ("binary16 overflow threshold at the largest half",
     "if (a >= 65520.0) return", "if (a >= 65504.0) return"),
    ("binary16 subnormal step halved",
     "const double step = sub ? std::ldexp(1.0, -24) : std::ldexp(1.0, e - 10);",
     "const double step = sub ? std::ldexp(1.0, -25) : std::ldexp(1.0, e - 10);"),
    ("FP16 group drops the error on a step without exchange",
     "      e[k] = x;\n", "      e[k] = 0.0f;\n"),
]


@pytest.mark.parametrize("name,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_a_planted_mistake_fails_a_pin(tmp_path, name, old, new):
    src = open(SRC).read()
    assert old in src, f"{name}: the text to mutate is missing"
    cxx = os.environ.get("CXX", "g++")
    if shutil.which(cxx) is None:
        pytest.skip("no C++ compiler")
    (tmp_path / "oracle.cpp").write_text(src.replace(old, new, 1))
    lib = str(tmp_path / "liboracle.so")
    subprocess.run([cxx, "-std=c++17", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
                    "-shared", "-o", lib, str(tmp_path / "oracle.cpp")], check=True)
    env = dict(os.environ, ORACLE_LIB=lib)
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle_pins.py"),
                        os.path.join(ROOT, "tests", "test_oracle_mixed.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode != 0 and "failed" in r.stdout, f"{name}: every pin passed"
