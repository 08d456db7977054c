"""Pins against numbers the pages print (tests/golden/pages_printed_values.json).

Each fixture names its page and section.  The oracle and the library's
state layout are checked against them; no expected value here comes from
the GPU path.

  [OPT] "LLM training series, part 2: optimizers" (mhpq.cn article)
  [K2]  "Kimi K2 ... what is worth noting" (Zhihu answer by toothacher17)
"""
import json
import math
import os
import re

import numpy as np
import pytest

import oracle

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)

with open(os.path.join(HERE, "golden", "pages_printed_values.json")) as f:
    GOLDEN = {v["id"]: v for v in json.load(f)["values"]}


def gold(key):
    return GOLDEN[key]["value"]


def test_every_fixture_cites_a_page_section():
    for v in GOLDEN.values():
        assert re.match(r"(OPT|K2) section \d", v["source"]), v


def header_pointer_types(func):
    """Parameter types of `func` as declared in include/muon_step.h."""
    with open(os.path.join(ROOT, "include", "muon_step.h")) as f:
        text = f.read()
    m = re.search(r"\b%s\s*\(([^)]*)\)" % func, text)
    assert m, func
    return [p.strip() for p in m.group(1).split(",")]


def test_state_layout_reproduces_the_7b_memory_table():
    """[OPT] section 2.4: AdamW keeps FP32 m and v (56 GB for 7B) and an FP32
    master copy (28 GB), 84 GB in all; a single FP32 momentum is 28 GB.
    The library keeps exactly that state: adamw_step takes float p, m, v,
    and the Muon step one float momentum M beside the float master W."""
    params = 7e9
    adamw = header_pointer_types("adamw_step")
    assert adamw[0].startswith("float*") and adamw[2].startswith("float*") and adamw[3].startswith("float*")
    with open(os.path.join(ROOT, "include", "muon_step.h")) as f:
        text = f.read()
    mt = re.search(r"typedef struct\s*\{(.*?)\}\s*muon_matrix_t;", text, re.S).group(1)
    assert re.search(r"float\s*\*\s*W;", mt) and re.search(r"float\s*\*\s*M;", mt)
    f32 = np.dtype(np.float32).itemsize
    # the oracle's state buffers are fp32 too
    p, m, v = oracle.adamw_step(np.zeros(4, np.float32), np.ones(4, np.float32),
                                np.zeros(4, np.float32), np.zeros(4, np.float32))
    assert p.dtype == m.dtype == v.dtype == np.float32
    assert 2 * f32 * params / 1e9 == gold("adam_states_7b_gb")
    assert f32 * params / 1e9 == gold("fp32_master_7b_gb")
    assert gold("adam_states_7b_gb") + gold("fp32_master_7b_gb") == gold("adamw_optimizer_total_7b_gb")
    assert f32 * params / 1e9 == gold("momentum_state_7b_gb")   # Muon's one momentum buffer
    assert 2 * 1 * params / 1e9 == gold("adamw_8bit_states_7b_gb")


def test_beta1_keeps_the_printed_fresh_fraction():
    """[OPT] section 3.2: with beta1 = 0.9 the new first moment is 10% the
    current gradient and 90% its history."""
    b1 = gold("beta1_default")
    g = np.array([1.0, -2.0, 0.5, 8.0], np.float32)
    m0 = np.array([4.0, 4.0, -4.0, 0.0], np.float32)
    hp = oracle.AdamwConfig(beta1=b1, beta2=0.999, weight_decay=0.0)
    _, m1, _ = oracle.adamw_step(np.zeros(4, np.float32), g, m0, np.zeros(4, np.float32), hp, t=1)
    fresh = gold("beta1_fresh_fraction")
    np.testing.assert_allclose(m1, fresh * g + (1 - fresh) * m0, rtol=2e-7, atol=1e-7)


def test_beta2_window_is_about_a_thousand_steps():
    """[OPT] section 3.2: beta2 = 0.999 averages about the past 1000 steps.
    The EMA's weights sum to 1 - beta2^t; half of the total weight sits in
    the last ~693 steps and 1 - 1/e of it in the last 1000 (the window
    1/(1-beta2))."""
    b2 = gold("beta2_default")
    assert round(1.0 / (1.0 - b2)) == gold("beta2_window_steps")
    # the oracle's second moment after 1000 steps of g = 1 from v = 0 is the
    # weight of those 1000 steps, 1 - beta2^1000 = 1 - 1/e (to 0.05%)
    hp = oracle.AdamwConfig(beta1=0.9, beta2=b2, weight_decay=0.0, lr=0.0)
    p = np.zeros(1, np.float32)
    m = np.zeros(1, np.float32)
    v = np.zeros(1, np.float32)
    g = np.ones(1, np.float32)
    for t in range(1, gold("beta2_window_steps") + 1):
        p, m, v = oracle.adamw_step(p, g, m, v, hp, t=t)
    assert abs(float(v[0]) - (1 - math.exp(-1))) < 5e-4


@pytest.mark.parametrize("eps", [1e-8, 1e-6])
def test_printed_eps_values_on_the_first_step(eps):
    """[OPT] sections 2.3/3.2: the first bias-corrected step is
    lr * g / (|g| + eps), with eps one of the printed 1e-8 / 1e-6."""
    assert eps in gold("eps_examples")
    g = np.array([1e-3, -1e-5, 1e-7, 3.0], np.float32)
    lr = 1e-2
    hp = oracle.AdamwConfig(lr=lr, beta1=0.9, beta2=0.999, eps=eps, weight_decay=0.0)
    p, _, _ = oracle.adamw_step(np.zeros(4, np.float32), g, np.zeros(4, np.float32), np.zeros(4, np.float32), hp, t=1)
    expected = -lr * g.astype(np.float64) / (np.abs(g.astype(np.float64)) + eps)
    np.testing.assert_allclose(p, expected, rtol=1e-5)


def test_page_cubic_pulls_singular_values_to_one():
    """[OPT] section 4.2: X <- (3X - X X^T X)/2, typically 5 times, moves the
    singular values towards 1: small ones grow, large ones shrink, 1 stays.
    On a diagonal input the singular values are the diagonal, and the
    iteration acts on each one as s <- (3 s - s^3) / 2."""
    a, b = gold("ns_cubic_coefficients")
    assert (a, b, 0.0) == oracle.CUBIC
    steps = gold("ns_typical_iterations")
    sig = np.array([0.05, 0.3, 1.0, 1.4, 1.6])
    X = np.zeros((5, 8))
    X[np.arange(5), np.arange(5)] = sig
    out = oracle.newton_schulz(X, steps=steps, coeffs=oracle.CUBIC, emulate_bf16=False)
    got = np.sort(np.linalg.svd(out, compute_uv=False))
    s = sig.copy()
    for _ in range(steps):
        s = (3 * s - s ** 3) / 2
    np.testing.assert_allclose(got, np.sort(s), rtol=1e-12, atol=1e-14)
    # small values grow, values above 1 (below sqrt 3) shrink, 1 is fixed
    assert s[0] > sig[0] and s[1] > sig[1] and abs(s[2] - 1) < 1e-15 and s[3] < sig[3]
    assert abs(s[1] - 1) < abs(sig[1] - 1) and abs(s[3] - 1) < abs(sig[3] - 1)


def test_library_default_runs_the_typical_iteration_count():
    """[OPT] section 4.2: 5 iterations is the common choice; it is the
    library's and the oracle's default."""
    import optimizer_muon_step_gb300 as m
    assert m.MuonHparams().ns_steps == gold("ns_typical_iterations")
    assert oracle.MuonConfig().ns_steps == gold("ns_typical_iterations")


def test_muon_update_rms_sits_at_the_adamw_band():
    """[K2] section 3.1: AdamW's update RMS is empirically 0.2-0.4, and the
    Muon update is scaled to match it.  With lr = 1 and no decay, the
    update of an orthogonalised gradient has RMS 0.2 * rms(sigma(O)), and
    sigma(O) lies in the quintic's band, so the update RMS lands at the
    lower edge of the printed band (0.2 * [0.68, 1.2])."""
    lo, hi = gold("adamw_update_rms_band")
    rng = np.random.default_rng(3)
    for rows, cols in ((96, 256), (256, 96)):
        W = np.zeros((rows, cols), np.float32)
        G = (rng.standard_normal((rows, cols)) * 1e-2).astype(np.float32)
        M = np.zeros((rows, cols), np.float32)
        hp = oracle.MuonConfig(lr=1.0, weight_decay=0.0, rms_scale=lo)
        W1, _, _, _ = oracle.muon_step_matrix(W, G, M, hp)
        rms = float(np.sqrt(np.mean(W1.astype(np.float64) ** 2)))
        assert 0.68 * lo < rms < min(1.21 * lo, hi), (rows, cols, rms)


@pytest.mark.parametrize("max_norm", [1.0, 2.0, 5.0])
def test_printed_clip_thresholds_bound_the_global_norm(max_norm):
    """[OPT] section 5.4: gradient clipping stays on as a safety net with
    max_grad_norm 1.0, or 2.0 / 5.0 on large models.  After the oracle's
    clip the global norm of all gradients of the call is at most the
    threshold, and gradients already below it are left alone."""
    assert max_norm in gold("max_grad_norm_examples")
    rng = np.random.default_rng(int(max_norm))
    Gs = [rng.standard_normal((16, 24)).astype(np.float32) * 3, rng.standard_normal((24, 8)).astype(np.float32)]
    sumsq, bad = oracle.grad_stats(Gs)
    assert bad == 0
    clip = oracle.clip_factor(sumsq, max_norm)
    clipped = math.sqrt(sum(float(np.sum((clip * g.astype(np.float64)) ** 2)) for g in Gs))
    assert clipped <= max_norm * (1 + 1e-6)
    small = [g * (0.5 * max_norm / math.sqrt(sumsq)) for g in Gs]
    s2, _ = oracle.grad_stats(small)
    assert oracle.clip_factor(s2, max_norm) == 1.0
