"""Per-matrix step statistics (muon_step_batched_stats) against the oracle.

For every matrix the step reports ||u||_F, the norm of the look-ahead it
normalised, and the RMS of the RMS-matched update scale * O ("Kimi K2 ...
what is worth noting", section 3.1: matched to AdamW's 0.2-0.4).  The
oracle computes both in fp64 from its own u and O (oracle.step_stats).

Tolerances: u_norm 1e-5 relative (the GPU adds fp32 tile sums of u^2 in
fp64); update_rms 2e-3 relative (the GPU's O and the oracle's agree to
bf16 rounding per element, and the RMS averages over the matrix).
Requesting statistics must not change W or M by a single bit, and a step
the non-finite guard skips reports NaN.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import optimizer_muon_step_gb300 as m

pytestmark = pytest.mark.gpu

DEV = "cuda"


def make_mats(shapes, seed):
    gen = torch.Generator(device=DEV).manual_seed(seed)
    W = [torch.randn(r, c, device=DEV, generator=gen) * 0.02 for r, c in shapes]
    G = [(torch.randn(r, c, device=DEV, generator=gen) * 1e-2).to(
        torch.bfloat16 if i % 2 else torch.float32) for i, (r, c) in enumerate(shapes)]
    M = [torch.randn(r, c, device=DEV, generator=gen) * 1e-2 for r, c in shapes]
    return W, G, M


def cfg_of(hp):
    return oracle.MuonConfig(lr=hp.lr, weight_decay=hp.weight_decay, momentum=hp.momentum,
                             nesterov=hp.nesterov, ns_steps=hp.ns_steps, ns_a=hp.ns_a, ns_b=hp.ns_b,
                             ns_c=hp.ns_c, norm_eps=hp.norm_eps, rms_scale=hp.rms_scale,
                             scale_mode=hp.scale_mode, skip_nonfinite=hp.skip_nonfinite,
                             max_grad_norm=hp.max_grad_norm, ns_coeffs=hp.ns_coeffs)


def oracle_stats(W0, G0, M0, hp):
    cfg = cfg_of(hp)
    out = []
    for w, g, mm in zip(W0, G0, M0):
        _, u = oracle.momentum(g, mm, cfg.momentum, cfg.nesterov)
        _, _, _, O = oracle.muon_step_matrix(w, g, mm, cfg)
        out.append(oracle.step_stats(u, O, cfg.rms_scale, cfg.scale_mode))
    return out


SHAPES = [(256, 512), (512, 256), (130, 70), (70, 130), (1024, 1100), (7, 13), (333, 300)]


@pytest.mark.parametrize("ns_steps,scale_mode", [(5, 0), (5, 1), (0, 0)])
def test_stats_match_the_oracle(lib, ns_steps, scale_mode):
    W, G, M = make_mats(SHAPES, seed=51)
    W0 = [w.cpu().numpy() for w in W]
    G0 = [g.float().cpu().numpy() for g in G]
    M0 = [x.cpu().numpy() for x in M]
    hp = m.MuonHparams(ns_steps=ns_steps, scale_mode=scale_mode)
    stats = torch.full((len(SHAPES), 2), -1.0, dtype=torch.float64, device=DEV)
    m.muon_step_batched(W, G, M, hp, stats=stats)
    got = stats.cpu().numpy()
    for i, (un, rms) in enumerate(oracle_stats(W0, G0, M0, hp)):
        assert abs(got[i, 0] / un - 1) < 1e-5, (i, got[i, 0], un)
        assert abs(got[i, 1] / rms - 1) < 2e-3, (i, got[i, 1], rms)
        if ns_steps == 5 and scale_mode == 0 and min(SHAPES[i]) >= 64:
            assert 0.14 < got[i, 1] < 0.4   # the band RMS matching aims at


def test_stats_leave_the_step_unchanged_and_cover_every_chunk(lib):
    W, G, M = make_mats(SHAPES, seed=52)
    Wb, Mb = [w.clone() for w in W], [x.clone() for x in M]
    W0 = [w.cpu().numpy() for w in W]
    G0 = [g.float().cpu().numpy() for g in G]
    M0 = [x.cpu().numpy() for x in M]
    hp = m.MuonHparams()
    ws_bytes = max(m.muon_workspace_bytes_per_matrix(*s) for s in SHAPES)
    assert m.muon_plan(SHAPES, ws_bytes)["chunk_id"].max() >= 1   # at least two chunks
    ws = m.allocate_workspace(ws_bytes)
    stats = torch.zeros((len(SHAPES), 2), dtype=torch.float64, device=DEV)
    m.muon_step_batched(W, G, M, hp, workspace=ws, stats=stats)
    m.muon_step_batched(Wb, G, Mb, hp, workspace=ws)
    for a, b in zip(W + M, Wb + Mb):
        assert torch.equal(a, b)
    got = stats.cpu().numpy()
    for i, (un, rms) in enumerate(oracle_stats(W0, G0, M0, hp)):
        assert abs(got[i, 0] / un - 1) < 1e-5
        assert abs(got[i, 1] / rms - 1) < 2e-3


def test_stats_of_a_skipped_step_are_nan(lib):
    W, G, M = make_mats(SHAPES[:3], seed=53)
    G[1][3, 4] = float("nan")
    batch = m.MuonBatch(W, G, M)
    stats = batch.step_with_stats(m.MuonHparams(skip_nonfinite=True))
    assert m.muon_query_status(batch.workspace) == m.MUON_STEP_SKIPPED
    assert bool(torch.isnan(stats).all())
    G[1][3, 4] = 0.0
    stats = batch.step_with_stats(m.MuonHparams(skip_nonfinite=True), out=stats)
    assert m.muon_query_status(batch.workspace) == 0
    assert bool(torch.isfinite(stats).all())
    assert math.isfinite(float(stats[0, 1])) and float(stats[0, 1]) > 0
