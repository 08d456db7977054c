"""Planted mistakes in the oracle must fail its pins.

The oracle is trusted because its pins (tests/test_oracle.py and
tests/test_golden.py) tie it to what the pages and the mathematics fix.
This test checks that the pins are sharp enough.  Each case copies
oracle/muon_oracle.c and changes one expression the way a plausible slip
would -- a dropped term, a wrong sign, a factor in the wrong place, a
wrong operand, a wrong rounding or ordering rule -- builds the copy with
the oracle's own compiler flags, and runs the pins against it in a child
pytest (MUON_ORACLE_LIB points the oracle at the copy).  Every such run
must fail.  The unchanged copy, built the same way, must pass, so a failing
run is the planted mistake being caught and not the harness.  Nothing here
touches the GPU library.
"""
import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "muon_oracle.c")
PINS = ["tests/test_oracle.py", "tests/test_golden.py"]

# (what the slip is, the exact text it replaces, the slipped text)
MUTANTS = [
    ("bf16 rounds toward zero",
     "if (dropped > 0x8000u || (dropped == 0x8000u && (kept & 1u)))", "if (0)"),
    ("bf16 ties round away from zero",
     "(dropped == 0x8000u && (kept & 1u))", "(dropped == 0x8000u)"),
    ("momentum without the (1 - mu) factor",
     "float gterm = one_minus_mu * g;", "float gterm = g;"),
    ("Nesterov look-ahead without mu",
     "u[i] = nesterov ? gterm + mu * mnew : mnew;", "u[i] = nesterov ? gterm + mnew : mnew;"),
    ("Nesterov flag read the other way round",
     "u[i] = nesterov ? gterm + mu * mnew : mnew;", "u[i] = nesterov ? mnew : gterm + mu * mnew;"),
    ("norm's eps under the square root",
     "const float s = (float)(1.0 / (sqrt(ss) + (double)eps));",
     "const float s = (float)(1.0 / sqrt(ss + (double)eps));"),
    ("NS polynomial takes A where A A belongs (bf16 path)",
     "float t2 = c * (float)AA[i];", "float t2 = c * (float)A[i];"),
    ("NS polynomial with the wrong sign on c (fp64 path)",
     "Bm[i] = (double)b * A[i] + (double)c * AA[i];", "Bm[i] = (double)b * A[i] - (double)c * AA[i];"),
    ("NS update drops the a X term (bf16 path)",
     "float t1 = axs * (float)X[i];", "float t1 = 0.0f * (float)X[i];"),
    ("NS input scale applied on every step",
     "const float xs = s == 0 ? x_scale : 1.0f;", "const float xs = x_scale;"),
    ("NS Gram matrix from the wrong product order",
     "matmul(X, XT, A, rows, cols, rows, acc);", "matmul(X, XT, A, rows, cols, rows, acc);\n"
     "        for (int64_t i = 0; i < rows; ++i) for (int64_t j = 0; j < i; ++j) A[i * rows + j] = A[j * rows + i] * 1.0009765625;"),
    ("update scale from min(rows, cols)",
     "const int64_t np = rows > cols ? rows : cols;\n    return", "const int64_t np = rows > cols ? cols : rows;\n    return"),
    ("Muon decay not multiplied by lr",
     "float delta = lr * (decay + step);", "float delta = decay + lr * step;"),
    ("Muon update added instead of subtracted",
     "W[r * cols + c] = w - delta;", "W[r * cols + c] = w + delta;"),
    ("AdamW first moment without bias correction",
     "float m_hat = mi / bc1;", "float m_hat = mi;"),
    ("AdamW eps under the square root",
     "float den = sqrtf(v_hat) + hp->eps;", "float den = sqrtf(v_hat + hp->eps);"),
    ("AdamW decay not multiplied by lr",
     "p[i] = p[i] - hp->lr * (upd + decay);", "p[i] = p[i] - hp->lr * upd - decay;"),
    ("AdamW second moment of g instead of g squared",
     "float g2 = gi * gi;", "float g2 = fabsf(gi);"),
    ("plan sort not stable on equal shapes",
     "if (om > cm || (om == cm && on > cn)) {", "if (om > cm || (om == cm && on >= cn)) {"),
    ("fp32 accumulation in descending k",
     "for (int64_t k = 0; k < K; ++k) {\n            const float a = (float)A[i * K + k];",
     "for (int64_t k = K - 1; k >= 0; --k) {\n            const float a = (float)A[i * K + k];"),
    ("block accumulation rounded to nearest instead of toward zero",
     "c[j] = f32_toward_zero((double)c[j] + run[j]);", "c[j] = (float)((double)c[j] + run[j]);"),
    ("first step's Gram matrix scaled by s instead of s^2",
     "const float xs2 = xs * xs;", "const float xs2 = xs;"),
    ("first step's update without s on B X",
     "float t2 = xs * (float)BX[i];", "float t2 = (float)BX[i];"),
    ("AdamW second moment corrected by the first moment's factor",
     "float v_hat = vi / bc2;", "float v_hat = vi / bc1;"),
    ("AdamW first moment decaying with beta2",
     "float mi = hp->beta1 * m[i] + one_minus_b1 * gi;", "float mi = hp->beta2 * m[i] + one_minus_b1 * gi;"),
    ("clip factor not capped at 1",
     "return (float)(c < 1.0 ? c : 1.0);", "return (float)c;"),
    ("guard counting NaN but not inf",
     "if (!isfinite(G[k][i]))", "if (isnan(G[k][i]))"),
    ("muP scale with the ratio inverted",
     "double r = sqrt((double)rows / (double)cols);", "double r = sqrt((double)cols / (double)rows);"),
    ("cast-after-scale reading rounding twice",
     "const float scaled = u[r * cols + c] * s;", "const float scaled = bf16_round(u[r * cols + c]) * s;"),
    ("update RMS averaged over one element too few",
     "*update_rms = sqrt(so / (double)n);", "*update_rms = sqrt(so / (double)(n - 1));"),
]


def _build(tmp, name, text):
    src = os.path.join(tmp, name + ".c")
    lib = os.path.join(tmp, name + ".so")
    with open(src, "w") as f:
        f.write(text)
    subprocess.run(["gcc", *oracle.CFLAGS, "-o", lib, src, "-lm"], check=True)
    return lib


def _pins(lib):
    env = dict(os.environ, MUON_ORACLE_LIB=lib, OMP_NUM_THREADS="2")
    r = subprocess.run([sys.executable, "-m", "pytest", *PINS, "-x", "-q", "-m", "not gpu", "-p", "no:cacheprovider"],
                       cwd=ROOT, env=env, capture_output=True, text=True)
    return r.returncode, r.stdout[-600:]


@pytest.fixture(scope="module")
def source():
    with open(SRC) as f:
        return f.read()


def test_every_planted_mistake_fails_a_pin(source, tmp_path):
    if shutil.which("gcc") is None:
        pytest.skip("gcc is needed to build the planted copies")
    for what, old, new in MUTANTS:
        assert source.count(old) == 1, f"{what}: the text to replace must occur once"
    libs = [_build(str(tmp_path), "unchanged", source)]
    for k, (what, old, new) in enumerate(MUTANTS):
        libs.append(_build(str(tmp_path), f"mutant{k}", source.replace(old, new)))
    with ThreadPoolExecutor(max_workers=4) as ex:
        results = list(ex.map(_pins, libs))
    rc, out = results[0]
    assert rc == 0, "the unchanged copy must pass the pins:\n" + out
    survivors = [(what, rc, out) for (what, _, _), (rc, out) in zip(MUTANTS, results[1:]) if rc != 1]
    assert not survivors, "planted mistakes no pin caught:\n" + "\n".join(
        f"- {what} (pytest exit {rc})\n{out}" for what, rc, out in survivors)
