"""Low-rank, ill-conditioned inputs on the GPU: the input class real
gradients resemble, and the one where a bf16 Newton-Schulz result is least
unique.

The iteration ("LLM training series, part 2: optimizers", section 4.2)
pushes every singular value of the normalised input towards 1.  A singular
value sigma near 0 is multiplied by about a^5 ~ 480 over five quintic
steps, so on a rank-8-plus-noise input the many noise-floor directions of
the output carry amplified bf16 rounding noise: two equally faithful bf16
evaluations (fp32 vs fp64 accumulation, or the cast to bf16 before vs after
the normalisation) disagree there by 1e-2 to 0.45 of the whole output.
The checks therefore compare what is unique and check that the rest is
valid:
  * the dominant part -- the output projected on the top-8 left singular
    vectors of the input -- against the oracle within 1e-2 (the oracle's
    own variants agree there to about 1e-3);
  * those 8 singular values of the output against the scalar map p^5 of
    the input's (NS acts on each singular value independently);
  * every singular value of the output inside the quintic's band, below
    1.21 (its image of (0, 1] tops out at 1.2024, plus bf16 noise);
  * the whole output's distance from the oracle within SPREAD_FACTOR of the
    oracle's own variant that accumulates the products in fp32 with one
    round-toward-zero per 16-product block (rz16).  Tensor-core fp32
    accumulation behaves that way in measurement: on these inputs the GPU
    lies 0.96-1.02 times as far from the fp64 evaluation as rz16 does, and
    2-5 times as far as round-to-nearest fp32 accumulation, whose errors
    cancel where truncation's do not;
  * the energy of the noise-floor part of the output within 1% of the
    oracle's: it is the input's own noise, amplified the same way (measured
    within 2e-4).
"""
import json
import os

import numpy as np
import pytest
import torch

import oracle
import optimizer_muon_step_gb300 as m
import workloads

pytestmark = pytest.mark.gpu

DEV = "cuda"
TOL = 1e-2
RANK = 8
SPREAD_FACTOR = 1.5
SIGMA_MAX = 1.21


def rel_fro(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    return np.linalg.norm(a - b) / np.linalg.norm(b)


def scalar_map(sigma, steps=5):
    a, b, c = (float(np.float32(x)) for x in oracle.QUINTIC)
    s = np.asarray(sigma, dtype=np.float64)
    for _ in range(steps):
        s = a * s + b * s ** 3 + c * s ** 5
    return s


def check_output(O_gpu, O_ref, O_rz16, X, what, normalise):
    """The checks of the module docstring, for wide or tall O (same
    orientation as X, whose left singular vectors define the dominant part).
    normalise: the NS input was X / ||X||_F (the step), else X itself."""
    O_gpu, O_ref, O_rz16 = (np.asarray(o, dtype=np.float64) for o in (O_gpu, O_ref, O_rz16))
    U, S, _ = np.linalg.svd(np.asarray(X, dtype=np.float64), full_matrices=False)
    P = U[:, :RANK]
    top = rel_fro(P.T @ O_gpu, P.T @ O_ref)
    whole = rel_fro(O_gpu, O_ref)
    spread = rel_fro(O_rz16, O_ref)
    sv = np.linalg.svd(O_gpu, compute_uv=False)
    sv_top = np.linalg.svd(P.T @ O_gpu, compute_uv=False)
    want_top = scalar_map(S[:RANK] / (np.linalg.norm(S) if normalise else 1.0))
    floor_gpu = np.linalg.norm(O_gpu - P @ (P.T @ O_gpu))
    floor_ref = np.linalg.norm(O_ref - P @ (P.T @ O_ref))
    info = dict(what=what, top=top, whole=whole, spread_rz16=spread, sigma_max=float(sv.max()),
                top_sv_err=float(np.abs(np.sort(sv_top) - np.sort(want_top)).max()),
                floor_ratio=float(floor_gpu / floor_ref))
    path = os.environ.get("MUON_PARITY_REPORT")
    if path:
        with open(path, "a") as f:
            f.write(json.dumps({k: (float(v) if not isinstance(v, str) else v) for k, v in info.items()}) + "\n")
    assert top < TOL, info
    assert sv.max() < SIGMA_MAX, info
    assert info["top_sv_err"] < 2e-2, info
    assert whole <= SPREAD_FACTOR * spread, info
    assert 0.99 < info["floor_ratio"] < 1.01, info


@pytest.mark.parametrize("shape", [(200, 328), (1408, 2048), (2048, 5632)])
def test_ns_on_lowrank_input(lib, shape):
    """Newton-Schulz alone (single-CTA tiles at 200 rows, CTA pairs at 1408
    and 2048) on a bf16 rank-8 input with 1e-3 noise."""
    mp, np_ = shape
    X = workloads.ns_input(mp, np_, seed=31, kind="lowrank")
    got = m.muon_newton_schulz(X.to(DEV)).float().cpu().numpy()
    Xf = X.float().numpy()
    ref = oracle.newton_schulz(Xf)
    rz16 = oracle.newton_schulz(Xf, accum=oracle.ACC_FP32_RZ16)
    check_output(got, ref, rz16, Xf, f"ns {shape}", normalise=False)


@pytest.mark.parametrize("shape", [(200, 328), (1408, 2048), (2048, 1408), (2048, 5632)])
def test_step_on_lowrank_gradient(lib, shape):
    """The whole Muon step on a rank-8-plus-noise gradient whose momentum
    shares its dominant column space (as consecutive gradients do).  The
    momentum is bit-exact; the update's NS part O = -(dW / lr + wd W) / scale
    is checked as above, in W's own orientation."""
    rows, cols = shape
    gen = torch.Generator().manual_seed(rows + cols)
    W = torch.randn(rows, cols, generator=gen) * 0.02
    G = workloads.lowrank(rows, cols, seed=41, std=1e-2)
    M = workloads.lowrank(rows, cols, seed=42, std=1e-2, basis_seed=41) * 0.05
    W0, G0, M0 = W.numpy().copy(), G.numpy().copy(), M.numpy().copy()
    Wd, Gd, Md = W.to(DEV), G.to(DEV), M.to(DEV)
    hp = m.MuonHparams(**workloads.MUON_HPARAMS)
    ws = m.muon_step_batched([Wd], [Gd], [Md], hp)
    assert m.muon_query_status(ws) == 0
    cfg = oracle.MuonConfig(**workloads.MUON_HPARAMS)
    oW, oM, _, _ = oracle.muon_step_matrix(W0, G0, M0, cfg)
    zW = oracle.muon_step_matrix(W0, G0, M0, cfg, accum=oracle.ACC_FP32_RZ16)[0]
    assert np.array_equal(Md.cpu().numpy(), oM)
    _, u = oracle.momentum(G0, M0, hp.momentum, hp.nesterov)
    lr, wd = float(np.float32(hp.lr)), float(np.float32(hp.weight_decay))
    scale = oracle.update_scale(rows, cols)

    def o_part(W1):
        return -((W1.astype(np.float64) - W0) / lr + wd * W0.astype(np.float64)) / scale

    check_output(o_part(Wd.cpu().numpy()), o_part(oW), o_part(zW), u, f"step {shape}", normalise=True)
