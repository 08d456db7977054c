"""GPU parity of the step's optional behaviours against the oracle:

  * per-step Newton-Schulz coefficients ("LLM training series, part 2:
    optimizers", section 4.2: the cubic X <- (3X - X X^T X)/2 or any
    schedule of odd polynomials);
  * the muP-style update scale max(1, sqrt(d_out/d_in)) ("Kimi K2 ... what
    is worth noting", section 3.2);
  * the call-wide gradient guard of section 5.4 of the optimizer article:
    skip the step when any gradient is non-finite, clip all gradients by
    their global norm.

Tolerances as in test_gpu_kernels.py; with clipping on, the clip factor is
computed from fp32 tile sums on the GPU and an fp64 running sum in the
oracle, so the momentum matches to a relative 1e-6 instead of bit for bit.
"""
import numpy as np
import pytest
import torch

import oracle
import optimizer_muon_step_gb300 as m
import workloads

pytestmark = pytest.mark.gpu

DEV = "cuda"
TOL = 1e-2
SCHEDULE = [(1.5, -0.5, 0.0), oracle.QUINTIC, oracle.QUINTIC, (2.0, -1.5, 0.5), (1.5, -0.5, 0.0)]


def rel_fro(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    return np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30)


def make_mats(shapes, seed, g_std=1e-2):
    gen = torch.Generator(device=DEV).manual_seed(seed)
    W = [torch.randn(r, c, device=DEV, generator=gen) * 0.02 for r, c in shapes]
    G = [torch.randn(r, c, device=DEV, generator=gen) * g_std for r, c in shapes]
    M = [torch.randn(r, c, device=DEV, generator=gen) * 1e-2 for r, c in shapes]
    return W, G, M


def host(ts):
    return [t.float().cpu().numpy() for t in ts]


def cfg_of(hp: m.MuonHparams) -> oracle.MuonConfig:
    return oracle.MuonConfig(lr=hp.lr, weight_decay=hp.weight_decay, momentum=hp.momentum,
                             nesterov=hp.nesterov, ns_steps=hp.ns_steps, ns_a=hp.ns_a, ns_b=hp.ns_b,
                             ns_c=hp.ns_c, norm_eps=hp.norm_eps, rms_scale=hp.rms_scale,
                             scale_mode=hp.scale_mode, skip_nonfinite=hp.skip_nonfinite,
                             max_grad_norm=hp.max_grad_norm, ns_coeffs=hp.ns_coeffs)


@pytest.mark.parametrize("shape", [(200, 328), (768, 900)])  # single-CTA and CTA-pair kernels
def test_ns_per_step_coefficients(lib, shape):
    X = torch.stack([workloads.ns_input(*shape, seed=21 + i) for i in range(2)]).to(DEV)
    got = m.muon_newton_schulz(X, steps=len(SCHEDULE), coeffs=SCHEDULE).float().cpu().numpy()
    for i in range(2):
        ref = oracle.newton_schulz(X[i].float().cpu().numpy(), steps=len(SCHEDULE), coeffs=SCHEDULE)
        assert rel_fro(got[i], ref) < TOL


def test_step_with_coefficient_table_and_mup_scale(lib):
    shapes = [(256, 512), (640, 160), (130, 70)]
    W, G, M = make_mats(shapes, seed=5)
    W0, G0, M0 = host(W), host(G), host(M)
    hp = m.MuonHparams(ns_steps=len(SCHEDULE), ns_coeffs=SCHEDULE, scale_mode=1)
    m.muon_step_batched(W, G, M, hp)
    cfg = cfg_of(hp)
    for i in range(len(shapes)):
        oW, oM, _, _ = oracle.muon_step_matrix(W0[i], G0[i], M0[i], cfg)
        assert np.array_equal(M[i].cpu().numpy(), oM)
        assert rel_fro(W[i].cpu().numpy().astype(np.float64) - W0[i], oW.astype(np.float64) - W0[i]) < TOL


def test_guard_skips_the_whole_step_on_nonfinite(lib):
    shapes = [(256, 512), (512, 256), (64, 64)]
    W, G, M = make_mats(shapes, seed=6)
    G[1][7, 9] = float("nan")
    W0, M0 = [w.clone() for w in W], [x.clone() for x in M]
    ws = m.muon_step_batched(W, G, M, m.MuonHparams(skip_nonfinite=True))
    assert m.muon_query_status(ws) == m.MUON_STEP_SKIPPED
    for a, b in zip(W + M, W0 + M0):
        assert torch.equal(a, b)
    # the next call with clean gradients runs normally and reports nothing
    G[1][7, 9] = 0.0
    m.muon_step_batched(W, G, M, m.MuonHparams(skip_nonfinite=True), workspace=ws)
    assert m.muon_query_status(ws) == 0
    assert not torch.equal(W[0], W0[0])


@pytest.mark.parametrize("chunked", [False, True])
def test_guard_clips_by_global_norm(lib, chunked):
    shapes = [(256, 512), (640, 160), (512, 900), (33, 65)]
    W, G, M = make_mats(shapes, seed=7, g_std=0.05)
    W0, G0, M0 = host(W), host(G), host(M)
    norm = float(np.sqrt(sum((g.astype(np.float64) ** 2).sum() for g in G0)))
    hp = m.MuonHparams(max_grad_norm=0.3 * norm)
    ws = None
    if chunked:
        ws = m.allocate_workspace(max(m.muon_workspace_bytes_per_matrix(*s) for s in shapes))
        assert m.muon_plan(shapes, ws.numel())["chunk_id"].max() >= 1  # at least two chunks
    ws = m.muon_step_batched(W, G, M, hp, workspace=ws)
    assert m.muon_query_status(ws) == 0
    ref, skipped = oracle.muon_step_list(W0, G0, M0, cfg_of(hp))
    assert not skipped
    for i, (oW, oM) in enumerate(ref):
        assert np.allclose(M[i].cpu().numpy(), oM, rtol=1e-6, atol=1e-12)
        assert rel_fro(W[i].cpu().numpy().astype(np.float64) - W0[i], oW.astype(np.float64) - W0[i]) < TOL


def test_guard_loose_clip_changes_nothing(lib):
    shapes = [(256, 512), (512, 256)]
    W, G, M = make_mats(shapes, seed=8)
    W2, M2 = [w.clone() for w in W], [x.clone() for x in M]
    m.muon_step_batched(W, G, M, m.MuonHparams())
    m.muon_step_batched(W2, G, M2, m.MuonHparams(max_grad_norm=1e9, skip_nonfinite=True))
    for a, b in zip(W + M, W2 + M2):
        assert torch.equal(a, b)
