"""Pins for the oracle: checks against facts fixed by the pages or by
mathematics, never against the oracle's own formula retyped.

Sources:
  [OPT] "LLM training series, part 2: optimizers" (mhpq.cn article)
  [K2]  "Kimi K2 ... what is worth noting" (Zhihu answer by toothacher17)
"""
import math

import numpy as np
import pytest
import torch

import oracle

QUINTIC = tuple(float(np.float32(c)) for c in oracle.QUINTIC)


def scalar_poly_iterate(sigma, coeffs, steps):
    """The NS map restricted to one singular value: s <- a s + b s^3 + c s^5."""
    a, b, c = coeffs
    s = np.asarray(sigma, dtype=np.float64)
    for _ in range(steps):
        s = a * s + b * s ** 3 + c * s ** 5
    return s


def rand_wide(rows, cols, seed, scale=None):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((rows, cols))
    return x / np.linalg.norm(x) if scale is None else x * scale


# --------------------------------------------------------------------------
# bf16 rounding
# --------------------------------------------------------------------------

def test_bf16_hand_cases():
    # 1 + 2^-8 is exactly half-way between 1 and 1 + 2^-7: ties go to the
    # even mantissa (1.0); 1 + 3*2^-8 lies half-way between 1 + 2^-7 (odd)
    # and 1 + 2^-6 (even) and must round up.
    x = np.float32([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, 1.0 + 2 ** -8 + 2 ** -20,
                    -2.0, 0.0, -0.0])
    bits = oracle.bf16_bits(x)
    assert list(bits) == [0x3F80, 0x3F80, 0x3F82, 0x3F81, 0xC000, 0x0000, 0x8000]


def test_bf16_special_values():
    x = np.float32([np.inf, -np.inf, np.nan, np.finfo(np.float32).max, 1e-40, -1e-45])
    v = oracle.bf16_values(oracle.bf16_bits(x))
    assert v[0] == np.inf and v[1] == -np.inf and np.isnan(v[2])
    assert v[3] == np.inf  # rounds past the largest finite bf16
    assert v[4] > 0 and v[5] <= 0  # subnormals keep their sign


def test_bf16_matches_library_cast_on_random_bits():
    # torch's float32 -> bfloat16 cast is round-to-nearest-even; compare on
    # finite values spanning the whole exponent range.
    rng = np.random.default_rng(1)
    bits = rng.integers(0, 2 ** 32, size=200_000, dtype=np.uint64).astype(np.uint32)
    x = bits.view(np.float32)
    x = x[np.isfinite(x)]
    ours = oracle.bf16_bits(x)
    ref = torch.from_numpy(x.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)


# --------------------------------------------------------------------------
# Newton-Schulz ([OPT] section 4.2)
# --------------------------------------------------------------------------

@pytest.mark.parametrize("shape", [(1, 1), (2, 3), (7, 13), (16, 16), (32, 64), (5, 40)])
@pytest.mark.parametrize("coeffs", [QUINTIC, (1.5, -0.5, 0.0)])
def test_ns_equals_singular_value_polynomial(shape, coeffs):
    """NS acts on each singular value independently: for X = U S V^T the
    iteration returns U p^k(S) V^T (exact algebra; fp64, no bf16)."""
    X = rand_wide(*shape, seed=sum(shape))
    U, S, Vt = np.linalg.svd(X, full_matrices=False)
    expected = (U * scalar_poly_iterate(S, coeffs, 5)) @ Vt
    got = oracle.newton_schulz(X, steps=5, coeffs=coeffs, emulate_bf16=False)
    err = np.linalg.norm(got - expected) / np.linalg.norm(expected)
    assert err < 1e-10


def test_ns_zero_steps_is_identity():
    X = oracle.bf16_round(rand_wide(8, 24, 3))
    assert np.array_equal(oracle.newton_schulz(X, steps=0), X)


def test_input_scale_enters_the_first_step_only():
    """newton_schulz(X, x_scale=s) iterates on s * X: in fp64 it equals the
    iteration on the pre-scaled input; emulating bf16 with a power-of-two s
    (every fp32 product then scales exactly) it equals it bit for bit; with
    no steps it is bf16(s * X)."""
    X = oracle.bf16_round(rand_wide(16, 40, 11))
    s = float(np.float32(0.37))  # the scale is an fp32 argument
    a = oracle.newton_schulz(X, emulate_bf16=False, x_scale=s)
    b = oracle.newton_schulz(s * X.astype(np.float64), emulate_bf16=False)
    assert np.linalg.norm(a - b) / np.linalg.norm(b) < 1e-12
    R = rand_wide(16, 40, 11)
    for p2 in (2.0 ** -3, 2.0 ** 5):
        Xp = oracle.bf16_round((R / (np.linalg.norm(R) * p2)).astype(np.float32))  # p2 * Xp has norm ~1
        c = oracle.newton_schulz(Xp, x_scale=p2)
        d = oracle.newton_schulz(oracle.bf16_round((p2 * Xp).astype(np.float32)))
        assert np.all(np.isfinite(d)) and np.array_equal(c, d)
    e = oracle.newton_schulz(X, steps=0, x_scale=s)
    assert np.array_equal(e, oracle.bf16_round((np.float32(s) * X).astype(np.float32)))


def test_quintic_band_on_random_input():
    """For singular values of the normalised input in [1.5e-3, 1] the
    5-fold quintic lands in the scalar map's image of that interval."""
    grid = np.linspace(1.5e-3, 1.0, 200_001)
    image = scalar_poly_iterate(grid, QUINTIC, 5)
    lo, hi = image.min(), image.max()
    assert 0.67 < lo < 0.69 and 1.19 < hi < 1.21
    X = rand_wide(128, 320, seed=7)
    s_in = np.linalg.svd(X, compute_uv=False)
    assert s_in.min() > 1.5e-3 and s_in.max() <= 1.0
    s_out = np.linalg.svd(oracle.newton_schulz(X, emulate_bf16=False), compute_uv=False)
    assert s_out.min() >= lo - 1e-9 and s_out.max() <= hi + 1e-9
    # with bf16 storage the band holds up to bf16 rounding noise
    Xb = oracle.bf16_round(X)
    s_b = np.linalg.svd(oracle.newton_schulz(Xb, emulate_bf16=True), compute_uv=False)
    assert s_b.min() > lo - 0.02 and s_b.max() < hi + 0.02


def test_cubic_converges_to_polar_factor():
    """[OPT] section 4.2: the cubic X <- (3X - X X^T X)/2 pushes every
    singular value to 1, i.e. towards the polar factor U V^T, with no SVD."""
    rng = np.random.default_rng(11)
    U, _ = np.linalg.qr(rng.standard_normal((12, 12)))
    V, _ = np.linalg.qr(rng.standard_normal((30, 12)))
    S = np.linspace(0.3, 1.0, 12)
    X = (U * S) @ V.T
    got = oracle.newton_schulz(X, steps=40, coeffs=(1.5, -0.5, 0.0), emulate_bf16=False)
    assert np.linalg.norm(got - U @ V.T) < 1e-10
    assert np.linalg.norm(got @ got.T - np.eye(12)) < 1e-10


@pytest.mark.parametrize("mp,np_", [(16, 16), (64, 128), (256, 512)])
def test_orthogonal_input_scales_by_scalar_gain(mp, np_):
    """An input with orthonormal rows, normalised to unit Frobenius norm,
    has every singular value 1/sqrt(m'); NS returns p^5(1/sqrt(m')) times
    the orthonormal matrix."""
    rng = np.random.default_rng(mp)
    Q, _ = np.linalg.qr(rng.standard_normal((np_, mp)))
    Q = Q.T  # mp x np_ with orthonormal rows
    gain = float(scalar_poly_iterate(1.0 / math.sqrt(mp), QUINTIC, 5))
    got = oracle.newton_schulz(Q / math.sqrt(mp), emulate_bf16=False)
    assert np.linalg.norm(got - gain * Q) / np.linalg.norm(gain * Q) < 1e-12


def test_orthogonal_gains_known_values():
    # p^5(1/sqrt(m')) for the shapes the workloads use (fp64 scalar map)
    want = {256: 1.07052, 1408: 1.02553, 2048: 0.74461, 7168: 0.83242}
    for mp, g in want.items():
        assert abs(float(scalar_poly_iterate(1 / math.sqrt(mp), QUINTIC, 5)) - g) < 5e-5


def test_ns_rejects_tall_input():
    with pytest.raises(ValueError):
        oracle.newton_schulz(np.zeros((5, 3)))


# --------------------------------------------------------------------------
# Muon step
# --------------------------------------------------------------------------

def _inputs(rows, cols, seed, g_std=1e-2, m_std=1e-2):
    rng = np.random.default_rng(seed)
    W = (rng.standard_normal((rows, cols)) * 0.02).astype(np.float32)
    G = (rng.standard_normal((rows, cols)) * g_std).astype(np.float32)
    M = (rng.standard_normal((rows, cols)) * m_std).astype(np.float32)
    return W, G, M


def test_zero_gradient_and_momentum_gives_pure_decay():
    """u = 0 -> X0 = 0/(0+eps) = 0 -> NS(0) = 0 -> W' = W (1 - lr wd)."""
    W, _, _ = _inputs(24, 40, 0)
    Z = np.zeros_like(W)
    hp = oracle.MuonConfig()
    W1, M1, X0, O = oracle.muon_step_matrix(W, Z, Z, hp)
    assert not np.any(M1) and not np.any(X0) and not np.any(O)
    expect = W.astype(np.float64) * (1 - float(np.float32(hp.lr)) * float(np.float32(hp.weight_decay)))
    assert np.allclose(W1, expect, rtol=4e-7, atol=0)


def test_momentum_is_an_exponential_average():
    """[OPT] section 2.1: with g equal to the running average the average
    does not move (a fixed point); with mu = 0 the average is g itself."""
    W, G, _ = _inputs(8, 16, 1)
    hp = oracle.MuonConfig(momentum=0.5)  # 0.5 keeps every product exact
    _, M1, _, _ = oracle.muon_step_matrix(W, G, G, hp)
    assert np.array_equal(M1, G)
    hp0 = oracle.MuonConfig(momentum=0.0)
    _, M2, X0, _ = oracle.muon_step_matrix(W, G, np.ones_like(G), hp0)
    assert np.array_equal(M2, G)
    # mu = 0: the look-ahead is G itself, so X0 = bf16(G) (the NS input is
    # X0 / ||G|| up to eps): within half a bf16 ulp of G
    ref = G.astype(np.float64)
    assert np.all(np.abs(X0 - ref) <= np.abs(ref) * 2.0 ** -8 + 1e-30)


def test_nesterov_uses_updated_momentum():
    """With g = 0 the updated average is mu*M; the Nesterov look-ahead takes
    one more step of the same average: u = mu*(mu*M), so X0 ~ M.  Without
    Nesterov u = mu*M.  Both normalise to the direction of M; what differs
    is the momentum written back, and for g != 0 the direction."""
    W, G, M = _inputs(16, 24, 2)
    Z = np.zeros_like(G)
    hp = oracle.MuonConfig(momentum=0.5)
    _, M1, X0, _ = oracle.muon_step_matrix(W, Z, M, hp)
    assert np.array_equal(M1, 0.5 * M)
    ref = 0.25 * M.astype(np.float64)  # u = mu * (mu * M), exact for mu = 0.5
    assert np.all(np.abs(X0 - ref) <= np.abs(ref) * 2.0 ** -8 + 1e-30)
    # g != 0: Nesterov direction is (1-mu) g + mu M_new, plain is M_new
    hpn = oracle.MuonConfig(momentum=0.5, nesterov=True)
    hpp = oracle.MuonConfig(momentum=0.5, nesterov=False)
    _, _, Xn, _ = oracle.muon_step_matrix(W, G, M, hpn)
    _, _, Xp, _ = oracle.muon_step_matrix(W, G, M, hpp)
    Mnew = 0.5 * M.astype(np.float64) + 0.5 * G
    un = 0.5 * G + 0.5 * Mnew
    for X, u in ((Xn, un), (Xp, Mnew)):
        # the normalised input X0 / ||u|| is the direction of u
        r = u / np.linalg.norm(u)
        assert np.all(np.abs(X / np.linalg.norm(u) - r) <= np.abs(r) * 2.0 ** -8 + 1e-12)


def test_normalised_input_has_unit_norm():
    """The NS input s * X0, with X0 = bf16(u) and s = 1 / (||u|| + eps), has
    unit Frobenius norm to bf16 rounding; the step's X0 is that bf16(u)."""
    W, G, M = _inputs(48, 80, 3)
    _, _, X0, _ = oracle.muon_step_matrix(W, G, M)
    _, u = oracle.momentum(G, M, 0.95, True)
    X0b, s = oracle.normalize(u)
    assert np.array_equal(X0, X0b)
    assert np.array_equal(X0b, oracle.bf16_round(u))
    assert abs(np.linalg.norm(s * X0b.astype(np.float64)) - 1.0) < 2.0 ** -8


def test_norm_eps_is_added_to_the_norm():
    """The guard term sits outside the root, s = 1 / (||u|| + eps), as Adam
    adds eps to sqrt(v) ([OPT] sections 2.2-2.3; the reading the step
    takes).  With eps and the entries powers of two the normalised entries
    are exact: a single entry eps gives eps / (eps + eps) = 1/2, a single
    entry 3 eps gives 3/4, and the zero matrix gets s = 1/eps (its input stays
    zero).  eps under the root would give about 2^-10 and 3 * 2^-10 here."""
    eps = 2.0 ** -20
    for entry, expect in ((eps, 0.5), (3 * eps, 0.75)):
        u = np.zeros((4, 6), np.float32)
        u[1, 2] = entry
        X0, s = oracle.normalize(u, eps)
        assert s * float(X0[1, 2]) == expect
        assert np.count_nonzero(X0) == 1
    X0, s = oracle.normalize(np.zeros((4, 6), np.float32), eps)
    assert s == 2.0 ** 20 and not X0.any()


def test_update_rms_matches_adamw_band():
    """[K2] section 3.1: the update is scaled to match AdamW's update RMS
    (0.2-0.4).  With wd = 0, dW = -lr * 0.2 sqrt(max(m,n)) O, and since
    ||O||_F^2 = sum sigma_i^2 the update RMS is lr * 0.2 * rms(sigma(O))
    (in the wide orientation O has min(m,n) singular values over m*n
    entries)."""
    for rows, cols in ((64, 160), (160, 64)):
        W, G, M = _inputs(rows, cols, 4)
        hp = oracle.MuonConfig(weight_decay=0.0)
        W1, _, _, O = oracle.muon_step_matrix(W, G, M, hp)
        dW = W1.astype(np.float64) - W
        sig = np.linalg.svd(O.astype(np.float64), compute_uv=False)
        rms_expected = float(np.float32(hp.lr)) * 0.2 * math.sqrt(np.mean(sig ** 2))
        rms = math.sqrt(np.mean(dW ** 2))
        assert abs(rms / rms_expected - 1) < 1e-3
        # the update points against O (a descent step)
        Ow = O.T if rows > cols else O
        cos = np.sum(dW * Ow) / (np.linalg.norm(dW) * np.linalg.norm(Ow))
        assert cos < -0.999999
        # and NS has brought sigma into the quintic band -> RMS in [0.14, 0.24]*lr
        assert 0.6 < np.min(sig) and np.max(sig) < 1.25


def test_tall_matrix_equals_transposed_wide():
    """A tall matrix is orthogonalised in its transposed orientation, so the
    step on W^T gives the transpose of the step on W."""
    W, G, M = _inputs(96, 40, 5)
    W1, M1, X0a, Oa = oracle.muon_step_matrix(W, G, M)
    W2, M2, X0b, Ob = oracle.muon_step_matrix(W.T, G.T, M.T)
    assert np.array_equal(M1, M2.T)
    assert np.array_equal(X0a, X0b)
    assert np.linalg.norm(Oa - Ob) / np.linalg.norm(Ob) < 1e-2
    assert np.allclose(W1, W2.T, rtol=1e-5, atol=1e-7)


def test_decay_uses_old_weight():
    """[OPT] section 3.1: decoupled decay subtracts lr*wd*theta_t, the
    weight before this step's update.  With O = 0 (zero grad and momentum)
    the result is the same for wd applied once to the old W."""
    W, _, _ = _inputs(4, 4, 6)
    Z = np.zeros_like(W)
    hp = oracle.MuonConfig(lr=0.5, weight_decay=0.5)
    W1, *_ = oracle.muon_step_matrix(W, Z, Z, hp)
    assert np.array_equal(W1, W * np.float32(0.75))


# --------------------------------------------------------------------------
# AdamW ([OPT] sections 2.3, 3.1)
# --------------------------------------------------------------------------

def _adam_inputs(n, seed):
    rng = np.random.default_rng(seed)
    p = (rng.standard_normal(n) * 0.02).astype(np.float32)
    g = (rng.standard_normal(n) * 1e-3).astype(np.float32)
    m = (rng.standard_normal(n) * 1e-3).astype(np.float32)
    v = np.abs(rng.standard_normal(n) * 1e-6).astype(np.float32)
    return p, g, m, v


def test_adam_first_step_is_sign_like():
    """At t = 1 from m = v = 0 the bias corrections undo the averaging:
    m_hat = g, v_hat = g^2, so the step is lr * g / (|g| + eps)."""
    p, g, _, _ = _adam_inputs(4096, 0)
    z = np.zeros_like(p)
    hp = oracle.AdamwConfig(weight_decay=0.0)
    p1, m1, v1 = oracle.adamw_step(p, g, z, z, hp, t=1)
    lr, eps = float(np.float32(hp.lr)), float(np.float32(hp.eps))
    g64 = g.astype(np.float64)
    expect = p - lr * g64 / (np.abs(g64) + eps)
    assert np.allclose(p1, expect, rtol=0, atol=2e-6 * lr + 4e-8)
    assert np.all(np.sign(p - p1) == np.sign(g))


def test_adamw_decay_only():
    """g = 0, m = v = 0 -> m_hat = 0 -> 0/(0+eps) = 0: p' = p (1 - lr wd)."""
    p, _, _, _ = _adam_inputs(1000, 1)
    z = np.zeros_like(p)
    hp = oracle.AdamwConfig(lr=1e-2, weight_decay=0.1)
    p1, m1, v1 = oracle.adamw_step(p, z, z, z, hp, t=7)
    assert not np.any(m1) and not np.any(v1)
    expect = p.astype(np.float64) * (1 - float(np.float32(1e-2)) * float(np.float32(0.1)))
    assert np.allclose(p1, expect, rtol=3e-7, atol=0)


def test_adam_scale_invariance_is_exact():
    """With eps = 0 and wd = 0 Adam's step is invariant to scaling the
    gradient history by k (m by k, v by k^2).  k = 4 keeps every product
    exact, so the results must be bit-identical."""
    p, g, m, v = _adam_inputs(2048, 2)
    hp = oracle.AdamwConfig(eps=0.0, weight_decay=0.0)
    p1, m1, v1 = oracle.adamw_step(p, g, m, v, hp, t=3)
    p2, m2, v2 = oracle.adamw_step(p, 4 * g, 4 * m, 16 * v, hp, t=3)
    assert np.array_equal(p1, p2)
    assert np.array_equal(m2, 4 * m1) and np.array_equal(v2, 16 * v1)


def test_adam_bias_correction_vanishes_late():
    """For large t, 1 - beta^t -> 1 and the step is lr * m / (sqrt(v)+eps)."""
    p, g, m, v = _adam_inputs(1024, 3)
    hp = oracle.AdamwConfig(weight_decay=0.0)
    p1, m1, v1 = oracle.adamw_step(p, g, m, v, hp, t=100000)
    lr, eps = float(np.float32(hp.lr)), float(np.float32(hp.eps))
    step = lr * m1.astype(np.float64) / (np.sqrt(v1.astype(np.float64)) + eps)
    err = np.abs(p1 - (p - step))
    assert np.all(err <= 1e-6 * np.abs(step) + 2 * np.spacing(np.abs(p)))


def test_adam_moments_are_exponential_averages():
    """beta = 0.5 halves exactly, so m is the correctly rounded (m + g)/2."""
    p, g, m, v = _adam_inputs(512, 4)
    g = np.float32(2.0) ** np.round(np.log2(np.abs(g))).astype(np.float32) * np.sign(g)
    hp = oracle.AdamwConfig(beta1=0.5, beta2=0.5)
    _, m1, v1 = oracle.adamw_step(p, g, m, v, hp, t=2)
    assert np.array_equal(m1, ((m.astype(np.float64) + g) / 2).astype(np.float32))
    assert np.allclose(v1, (v.astype(np.float64) + g.astype(np.float64) ** 2) / 2, rtol=2 ** -23)


# --------------------------------------------------------------------------
# Plan
# --------------------------------------------------------------------------

def _check_plan(shapes, ws, plan):
    n = len(shapes)
    assert sorted(plan["mat_idx"].tolist()) == list(range(n))
    keys = [(min(shapes[i]), max(shapes[i]), i) for i in plan["mat_idx"]]
    assert keys == sorted(keys)  # (m', n') ascending, ties by caller index
    distinct = sorted({(min(s), max(s)) for s in shapes})
    for e in plan:
        r, c = shapes[e["mat_idx"]]
        assert e["transposed"] == int(r > c)
        assert (e["mp"], e["np"]) == (min(r, c), max(r, c))
        assert distinct[e["group_id"]] == (e["mp"], e["np"])
    # chunks: contiguous, within budget, and greedy (next one would not fit)
    per = [oracle.ws_bytes_per_matrix(e["mp"], e["np"]) for e in plan]
    chunks = plan["chunk_id"].tolist()
    assert chunks == sorted(chunks) and (not chunks or chunks[0] == 0)
    for cid in set(chunks):
        idx = [k for k, c in enumerate(chunks) if c == cid]
        assert idx == list(range(idx[0], idx[-1] + 1))
        assert sum(per[k] for k in idx) <= ws
        if idx[-1] + 1 < n:
            assert sum(per[k] for k in idx) + per[idx[-1] + 1] > ws
        # slots count within (chunk, group)
        seen = {}
        for k in idx:
            gid = plan["group_id"][k]
            assert plan["slot"][k] == seen.get(gid, 0)
            seen[gid] = seen.get(gid, 0) + 1


def test_plan_brute_force_random_lists():
    rng = np.random.default_rng(0)
    dims = [8, 16, 24, 128, 1408, 2048]
    for trial in range(60):
        n = int(rng.integers(0, 40))
        shapes = [(int(rng.choice(dims)), int(rng.choice(dims))) for _ in range(n)]
        need = max([oracle.ws_bytes_per_matrix(min(s), max(s)) for s in shapes] or [1])
        ws = int(need * rng.uniform(1.0, 6.0))
        _check_plan(shapes, ws, oracle.plan(shapes, ws))


def test_plan_rejects_matrix_larger_than_workspace():
    with pytest.raises(ValueError):
        oracle.plan([(2048, 2048)], 1024)


def test_workspace_bytes_formula():
    # two bf16 X buffers (m' x ld(n')), two bf16 Gram buffers (m' x ld(m')),
    # 256-byte padding, plus an 8 KiB record
    assert oracle.ws_bytes_per_matrix(2048, 2048) == 4 * 2048 * 2048 * 2 + 8192
    assert oracle.ws_bytes_per_matrix(7, 13) == 2 * 256 + 2 * 256 + 8192


@pytest.mark.parametrize("kind", ["gaussian"])
def test_bf16_emulated_ns_tracks_exact_iteration(kind):
    """The bf16-storage path differs from the fp64 iteration only by bf16
    rounding noise (each stored value has relative error <= 2^-9), so a
    dropped term or flipped sign in its epilogues shows up as an O(1) gap.
    The input has no tiny singular values: NS multiplies a singular value
    near 0 by up to a^5 ~ 480, so directions with sigma near the bf16
    noise floor are dominated by rounding noise in any bf16 evaluation."""
    from workloads import ns_input
    X = ns_input(64, 192, seed=3, kind=kind).float().numpy()
    exact = oracle.newton_schulz(X, emulate_bf16=False)
    emul = oracle.newton_schulz(X, emulate_bf16=True)
    assert np.linalg.norm(emul - exact) / np.linalg.norm(exact) < 2e-2
    # and every stored value is a bf16 value
    assert np.array_equal(oracle.bf16_round(emul.astype(np.float32)), emul.astype(np.float32))


def test_stage_functions_compose_to_the_step():
    """The step is momentum -> normalise -> NS -> final update; the staged
    entry points reproduce it exactly (tall input, so the transpose path
    is exercised too)."""
    W, G, M = _inputs(40, 24, 8)
    hp = oracle.MuonConfig()
    W1, M1, X0, O = oracle.muon_step_matrix(W, G, M, hp)
    M2, u = oracle.momentum(G, M, hp.momentum, hp.nesterov)
    X0b, s = oracle.normalize(u, hp.norm_eps)
    Ob = oracle.newton_schulz(X0b, hp.ns_steps, x_scale=s).astype(np.float32)
    W2 = oracle.final_update(W, Ob, hp.lr, hp.weight_decay, hp.rms_scale)
    assert np.array_equal(M1, M2) and np.array_equal(X0, X0b)
    assert np.array_equal(O, Ob) and np.array_equal(W1, W2)
    assert s > 0 and abs(np.linalg.norm(u.astype(np.float64)) * s - 1) < 1e-6


# --------------------------------------------------------------------------
# Spread variants: the same step evaluated with fp32-accumulated products,
# or with the cast to bf16 after the normalisation.  They measure how far
# two faithful bf16 evaluations lie apart; each is pinned on its own.
# --------------------------------------------------------------------------

def test_fp32_accumulation_is_ascending_and_rounds_every_sum():
    """1 + 2^-24 + 2^-24: summed in fp32 in ascending k, each addition ties
    back to 1 (round half to even), so the result is exactly 1; in fp64 it is
    1 + 2^-23.  Summed in the other order fp32 gives 1 + 2^-23 as well, so
    the pair pins both the precision and the order."""
    x = np.array([[1.0, 2.0 ** -12, 2.0 ** -12]])
    assert oracle.matmul(x, x.T)[0, 0] == 1.0 + 2.0 ** -23
    assert oracle.matmul(x, x.T, accum=oracle.ACC_FP32)[0, 0] == 1.0
    r = x[:, ::-1].copy()
    assert oracle.matmul(r, r.T, accum=oracle.ACC_FP32)[0, 0] == 1.0 + 2.0 ** -23


def test_blockwise_round_toward_zero_accumulation():
    """ACC_FP32_RZ16: each run of 16 products is summed exactly and added
    to the fp32 sum with one rounding toward zero.  Hand cases (all factors
    bf16 values, so every product is exact):
      * 1 in the first run and 3 * 2^-24 in the second: 1 + 1.5 ulp
        truncates to 1 + 2^-23, where round-to-nearest (fp64 then fp32, or
        fp32 throughout) ties to even at 1 + 2^-22;
      * 1 and eight products of -2^-26 in one run: the run sums exactly to
        1 - 2^-23, while one rounded-to-nearest fp32 addition per product
        loses each -2^-26 (below half an ulp) and stays at 1."""
    a = np.zeros((1, 32))
    b = np.zeros((32, 1))
    a[0, 0], b[0, 0] = 1.0, 1.0
    a[0, 16], b[16, 0] = 3.0 * 2.0 ** -12, 2.0 ** -12
    assert oracle.matmul(a, b, accum=oracle.ACC_FP32_RZ16)[0, 0] == 1.0 + 2.0 ** -23
    assert oracle.matmul(a, b, accum=oracle.ACC_FP32)[0, 0] == 1.0 + 2.0 ** -22
    assert np.float32(oracle.matmul(a, b)[0, 0]) == np.float32(1.0 + 2.0 ** -22)
    a = np.array([[1.0] + [-2.0 ** -13] * 8])
    b = np.array([[1.0] + [2.0 ** -13] * 8]).T
    assert oracle.matmul(a, b, accum=oracle.ACC_FP32_RZ16)[0, 0] == 1.0 - 2.0 ** -23
    assert oracle.matmul(a, b, accum=oracle.ACC_FP32)[0, 0] == 1.0
    assert oracle.matmul(a, b)[0, 0] == 1.0 - 2.0 ** -23
    # a negative sum truncates toward zero too: -(1 + 1.5 ulp) -> -(1 + 2^-23)
    a = np.zeros((1, 17))
    a[0, 0], a[0, 16] = -1.0, -3.0 * 2.0 ** -12
    b = np.zeros((17, 1))
    b[0, 0], b[16, 0] = 1.0, 2.0 ** -12
    assert oracle.matmul(a, b, accum=oracle.ACC_FP32_RZ16)[0, 0] == -(1.0 + 2.0 ** -23)


def test_fp32_accumulation_exact_on_small_integers():
    """Products and sums of small integers are exact in fp32: both
    accumulations give numpy's integer product (a transposed or misindexed
    operand would not)."""
    rng = np.random.default_rng(21)
    A = rng.integers(-8, 9, size=(7, 33))
    B = rng.integers(-8, 9, size=(33, 5))
    ref = (A @ B).astype(np.float64)
    assert np.array_equal(oracle.matmul(A, B), ref)
    assert np.array_equal(oracle.matmul(A, B, accum=oracle.ACC_FP32), ref)
    assert np.array_equal(oracle.matmul(A, B, accum=oracle.ACC_FP32_RZ16), ref)


def test_ns_fp32_accumulation_exact_on_integer_input():
    """One NS step with (a, b, c) = (1, 1, 1) on a small {-1, 0, 1} matrix
    stays within the integers bf16 holds exactly (|values| < 256), so both
    accumulations must return X + (A + A A) X with A = X X^T, computed here in
    integer arithmetic."""
    rng = np.random.default_rng(22)
    X = rng.integers(-1, 2, size=(3, 5))
    A = X @ X.T
    ref = (X + (A + A @ A) @ X).astype(np.float64)
    assert np.abs(ref).max() < 256
    for accum in (oracle.ACC_FP64, oracle.ACC_FP32, oracle.ACC_FP32_RZ16):
        got = oracle.newton_schulz(X.astype(np.float64), steps=1, coeffs=(1.0, 1.0, 1.0), accum=accum)
        assert np.array_equal(got, ref), accum


def test_ns_fp32_accumulation_stays_within_bf16_noise():
    """The fp32-accumulating iteration differs from the fp64 one only where a
    sum lands near a bf16 rounding boundary: on a well-conditioned input the
    two outputs are close but not identical."""
    from workloads import ns_input
    X = ns_input(96, 256, seed=4).float().numpy()
    a = oracle.newton_schulz(X)
    for accum in (oracle.ACC_FP32, oracle.ACC_FP32_RZ16):
        b = oracle.newton_schulz(X, accum=accum)
        rel = np.linalg.norm(a - b) / np.linalg.norm(a)
        assert 0 < rel < 1e-2, accum


@pytest.mark.parametrize("shape", [(16, 64), (64, 16)])
def test_cast_after_scale_equals_cast_before_for_power_of_two_norms(shape):
    """When s = 1/||u|| is a power of two (eps = 0, every |u| = 2^-6 over
    1024 elements: ||u|| = 2^-1), scaling commutes with every rounding, so
    the two readings of where the cast falls give bit-identical steps, in
    both orientations.  The other reading applying s twice, or not at all,
    would break this."""
    rng = np.random.default_rng(23)
    G = (rng.choice([-1.0, 1.0], size=shape) * 2.0 ** -6).astype(np.float32)
    W = (rng.standard_normal(shape) * 0.02).astype(np.float32)
    M = np.zeros(shape, np.float32)
    hp = oracle.MuonConfig(momentum=0.0, norm_eps=0.0)    # u = G exactly
    ref = oracle.muon_step_matrix(W, G, M, hp)
    var = oracle.muon_step_matrix(W, G, M, hp, cast_after_scale=True)
    assert np.array_equal(ref[0], var[0]) and np.array_equal(ref[3], var[3])
    assert np.array_equal(var[2], ref[2] * np.float32(2.0))  # X0 = bf16(u s), s = 2


def test_cast_after_scale_input_has_unit_norm():
    """X0 = bf16(u s) is the normalised look-ahead itself: unit Frobenius
    norm up to bf16 rounding (relative 2^-8 per element)."""
    W, G, M = _inputs(48, 80, 9)
    _, u = oracle.momentum(G, M)
    X0, s = oracle.normalize(u, cast_after_scale=True)
    assert abs(np.linalg.norm(X0.astype(np.float64)) - 1.0) < 2 ** -8
    X0b, sb = oracle.normalize(u)
    assert s == sb
    # one rounding of u s, not the double rounding bf16(bf16(u) s)
    assert np.array_equal(oracle.bf16_round(u * np.float32(s)), X0)
    assert not np.array_equal(oracle.bf16_round(X0b * np.float32(s)), X0)


def test_step_variants_route_through_the_staged_functions():
    """Each variant of the step is the staged functions with that choice:
    fp32 products in every NS stage, or the NS run unscaled on bf16(u s)."""
    W, G, M = _inputs(40, 24, 10)
    hp = oracle.MuonConfig()
    _, u = oracle.momentum(G, M, hp.momentum, hp.nesterov)
    X0, s = oracle.normalize(u)
    for accum in (oracle.ACC_FP32, oracle.ACC_FP32_RZ16):
        O32 = oracle.newton_schulz(X0, hp.ns_steps, x_scale=s, accum=accum).astype(np.float32)
        assert np.array_equal(oracle.muon_step_matrix(W, G, M, hp, accum=accum)[3], O32)
    X0c, _ = oracle.normalize(u, cast_after_scale=True)
    Oc = oracle.newton_schulz(X0c, hp.ns_steps).astype(np.float32)
    assert np.array_equal(oracle.muon_step_matrix(W, G, M, hp, cast_after_scale=True)[3], Oc)



# --------------------------------------------------------------------------
# Next rows: per-step NS coefficients, the muP update scale, the gradient
# guard
# --------------------------------------------------------------------------

def test_ns_per_step_coefficients_compose_scalar_maps():
    """With a different (a, b, c) at each step NS still acts on each
    singular value independently: the result is U (p_k o ... o p_1)(S) V^T."""
    table = [(1.5, -0.5, 0.0), QUINTIC, (1.5, -0.5, 0.0), (2.0, -1.5, 0.5)]
    X = rand_wide(12, 30, seed=4)
    U, S, Vt = np.linalg.svd(X, full_matrices=False)
    s = S.copy()
    for a, b, c in (tuple(float(np.float32(v)) for v in t) for t in table):
        s = a * s + b * s ** 3 + c * s ** 5
    got = oracle.newton_schulz(X, steps=len(table), coeffs=table, emulate_bf16=False)
    assert np.linalg.norm(got - (U * s) @ Vt) / np.linalg.norm(got) < 1e-10
    # a table repeating one triple equals that triple
    Xb = oracle.bf16_round(rand_wide(16, 48, seed=5))
    assert np.array_equal(oracle.newton_schulz(Xb, 3, [QUINTIC] * 3), oracle.newton_schulz(Xb, 3, QUINTIC))


def test_mup_scale_mode():
    """[K2] section 3.2: the per-matrix adjustment max(1, sqrt(d_out/d_in)):
    1 for wide or square (out <= in) weights, sqrt(out/in) for tall ones;
    and mode 0 is 0.2 * sqrt(max(m, n))."""
    assert oracle.update_scale(2048, 2048, 0.2, 1) == 1.0
    assert oracle.update_scale(1024, 4096, 0.2, 1) == 1.0
    assert oracle.update_scale(4096, 1024, 0.2, 1) == 2.0
    assert oracle.update_scale(256, 512, 0.2, 0) == np.float32(0.2 * math.sqrt(512))
    # the step's update uses it: with wd = 0, dW = -lr * 2 * O for a 4:1 tall matrix
    W, G, M = _inputs(64, 16, 9)
    hp = oracle.MuonConfig(weight_decay=0.0, scale_mode=1)
    W1, _, _, O = oracle.muon_step_matrix(W, G, M, hp)
    dW = W1.astype(np.float64) - W
    assert np.allclose(dW, -float(np.float32(hp.lr)) * 2.0 * O.T.astype(np.float64), rtol=1e-5, atol=1e-9)


def test_grad_guard_skips_on_nonfinite():
    """[OPT] section 5.4: an anomaly anywhere skips the whole step."""
    mats = [_inputs(8, 12, 20 + i) for i in range(3)]
    Ws, Gs, Ms = [m[0] for m in mats], [m[1].copy() for m in mats], [m[2] for m in mats]
    Gs[1][2, 3] = np.inf
    out, skipped = oracle.muon_step_list(Ws, Gs, Ms, oracle.MuonConfig(skip_nonfinite=True))
    assert skipped
    for (W1, M1), W, M in zip(out, Ws, Ms):
        assert np.array_equal(W1, W) and np.array_equal(M1, M)
    s, bad = oracle.grad_stats(Gs)
    assert bad == 1 and s == np.inf


def test_grad_clip_bounds_the_global_norm():
    """Clipping scales every gradient by one factor so the global norm is
    max_grad_norm: from M = 0 the new momentum is (1-mu) clip G, whose global
    norm is (1-mu) * max_grad_norm."""
    mats = [_inputs(16, 24, 30 + i, g_std=1.0) for i in range(3)]
    Ws, Gs = [m[0] for m in mats], [m[1] for m in mats]
    Ms = [np.zeros_like(m[2]) for m in mats]
    norm = math.sqrt(sum(float((g.astype(np.float64) ** 2).sum()) for g in Gs))
    hp = oracle.MuonConfig(max_grad_norm=norm / 3, momentum=0.5)
    out, skipped = oracle.muon_step_list(Ws, Gs, Ms, hp)
    assert not skipped
    got = math.sqrt(sum(float((M1.astype(np.float64) ** 2).sum()) for _, M1 in out))
    assert abs(got - 0.5 * norm / 3) / (0.5 * norm / 3) < 1e-6


def test_grad_clip_inactive_below_threshold_and_direction_only_above():
    """Below the threshold the clip factor is exactly 1 (results identical
    to no clipping); above it the clipped gradient depends only on the
    gradient's direction, so doubling every gradient changes nothing."""
    mats = [_inputs(16, 24, 40 + i) for i in range(2)]
    Ws, Gs, Ms = [m[0] for m in mats], [m[1] for m in mats], [m[2] for m in mats]
    plain, _ = oracle.muon_step_list(Ws, Gs, Ms, oracle.MuonConfig())
    loose, _ = oracle.muon_step_list(Ws, Gs, Ms, oracle.MuonConfig(max_grad_norm=1e9))
    for (a, b), (c, d) in zip(plain, loose):
        assert np.array_equal(a, c) and np.array_equal(b, d)
    hp = oracle.MuonConfig(max_grad_norm=1e-3)
    one, _ = oracle.muon_step_list(Ws, Gs, Ms, hp)
    two, _ = oracle.muon_step_list(Ws, [2 * g for g in Gs], Ms, hp)
    for (W1, M1), (W2, M2) in zip(one, two):
        assert np.allclose(M1, M2, rtol=1e-6, atol=0)
        assert np.allclose(W1, W2, rtol=1e-6, atol=1e-9)


# ---- per-matrix step statistics (monitoring output) -------------------------

def test_step_stats_u_norm_is_the_frobenius_norm():
    """u_norm is ||u||_F: numpy's norm of the fp64 widening, a separate route."""
    rng = np.random.default_rng(11)
    for rows, cols in ((37, 53), (90, 20)):
        u = (rng.standard_normal((rows, cols)) * 1e-2).astype(np.float32)
        O = np.zeros((min(rows, cols), max(rows, cols)), np.float32)
        un, _ = oracle.step_stats(u, O)
        assert abs(un / np.linalg.norm(u.astype(np.float64)) - 1) < 1e-12


@pytest.mark.parametrize("rows,cols", [(48, 112), (112, 48)])
def test_step_stats_update_rms_of_orthonormal_rows(rows, cols):
    """An O with orthonormal rows ([I 0], every singular value 1) has
    ||O||_F^2 = m', so the RMS of scale * O over the m*n entries is
    scale * sqrt(m' / (m n)) = 0.2 sqrt(n') / sqrt(n') = 0.2: the update RMS
    the RMS matching of [K2] section 3.1 targets."""
    mp, np_ = min(rows, cols), max(rows, cols)
    O = np.zeros((mp, np_), np.float32)
    O[:, :mp] = np.eye(mp, dtype=np.float32)
    u = np.ones((rows, cols), np.float32)
    _, rms = oracle.step_stats(u, O)
    # each scaled square is rounded to fp32: within one fp32 rounding (2^-24)
    scale = float(np.float32(0.2 * math.sqrt(np_)))
    assert abs(rms / (scale * math.sqrt(mp / (rows * cols))) - 1) < 2.0 ** -24
    assert abs(rms - 0.2) < 1e-7
    # muP-style scale: max(1, sqrt(rows / cols)) * sqrt(m' / (m n))
    _, rms1 = oracle.step_stats(u, O, scale_mode=1)
    s1 = float(np.float32(max(1.0, math.sqrt(rows / cols))))
    assert abs(rms1 / (s1 * math.sqrt(mp / (rows * cols))) - 1) < 2.0 ** -24


def test_step_stats_update_rms_from_singular_values():
    """For a real NS output, ||O||_F^2 = sum sigma_i^2 (from an SVD, not the
    element sum), so update_rms = scale * sqrt(sum sigma^2 / (m n)) up to the
    fp32 rounding of each scaled element; and it lies in the 0.2-0.4 band of
    [K2] section 3.1 (low end: the quintic leaves sigma in about [0.7, 1.2])."""
    for rows, cols in ((64, 160), (160, 64)):
        W, G, M = _inputs(rows, cols, 7)
        hp = oracle.MuonConfig()
        _, u = oracle.momentum(G, M, hp.momentum, hp.nesterov)
        _, _, _, O = oracle.muon_step_matrix(W, G, M, hp)
        _, rms = oracle.step_stats(u, O)
        sig = np.linalg.svd(O.astype(np.float64), compute_uv=False)
        scale = float(np.float32(0.2 * math.sqrt(max(rows, cols))))
        expected = scale * math.sqrt(np.sum(sig ** 2) / (rows * cols))
        assert abs(rms / expected - 1) < 1e-6
        assert 0.14 < rms < 0.4
