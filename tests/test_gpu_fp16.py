"""fp16 gradients (MUON_F16) against the oracle.

FP16 mixed-precision training hands the optimizer fp16 gradients, and "LLM
training series, part 2: optimizers" (section 5.4) describes what goes
wrong there: a gradient that overflows fp16 becomes inf, and the guard
should skip the step rather than let it into the state.  fp16 widens to
fp32 exactly, so the oracle takes the widened values: the momentum buffer
must match bit for bit, W within the usual 1e-2 relative Frobenius error.
"""
import numpy as np
import pytest
import torch

import oracle
import optimizer_muon_step_gb300 as m

pytestmark = pytest.mark.gpu

DEV = "cuda"
TOL = 1e-2


def rel_fro(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    return np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30)


def cfg_of(hp):
    return oracle.MuonConfig(lr=hp.lr, weight_decay=hp.weight_decay, momentum=hp.momentum,
                             nesterov=hp.nesterov, ns_steps=hp.ns_steps, ns_a=hp.ns_a, ns_b=hp.ns_b,
                             ns_c=hp.ns_c, norm_eps=hp.norm_eps, rms_scale=hp.rms_scale,
                             scale_mode=hp.scale_mode, skip_nonfinite=hp.skip_nonfinite,
                             max_grad_norm=hp.max_grad_norm, ns_coeffs=hp.ns_coeffs)


def make_fp16(shapes, seed, g_std=1e-2, offset=0):
    """fp32 W, M and fp16 G; with offset > 0 each G starts `offset` elements
    into a larger buffer (2-byte aligned only: the scalar paths)."""
    gen = torch.Generator(device=DEV).manual_seed(seed)
    W = [torch.randn(r, c, device=DEV, generator=gen) * 0.02 for r, c in shapes]
    G = []
    for r, c in shapes:
        buf = (torch.randn(r * c + offset, device=DEV, generator=gen) * g_std).half()
        G.append(buf[offset:].view(r, c))
    M = [torch.randn(r, c, device=DEV, generator=gen) * 1e-2 for r, c in shapes]
    return W, G, M


def host(ts):
    return [t.float().cpu().numpy() for t in ts]


# wide and tall (the tall pass's prefetching 2-byte kernel), pairs and single
# CTAs, a tall matrix with several 64x256-row units per column tile
SHAPES = [(256, 512), (512, 256), (130, 70), (70, 130), (1100, 1024), (2100, 130)]


@pytest.mark.parametrize("offset", [0, 1])
def test_fp16_gradients_match_the_oracle(lib, offset):
    W, G, M = make_fp16(SHAPES, seed=71, offset=offset)
    W0, G0, M0 = host(W), host(G), host(M)
    hp = m.MuonHparams()
    m.muon_step_batched(W, G, M, hp)
    cfg = cfg_of(hp)
    for i in range(len(SHAPES)):
        oW, oM, _, _ = oracle.muon_step_matrix(W0[i], G0[i], M0[i], cfg)
        assert np.array_equal(M[i].cpu().numpy(), oM), i
        dW = W[i].cpu().numpy().astype(np.float64) - W0[i]
        assert rel_fro(dW, oW.astype(np.float64) - W0[i]) < TOL, i


def test_fp16_overflow_skips_the_step(lib):
    """A gradient past fp16's range (65504) is inf after the cast; with the
    guard on, nothing changes and the skip is reported; without it the inf
    stays in its own matrix."""
    W, G, M = make_fp16(SHAPES[:3], seed=72)
    G[2][5, 7] = torch.tensor(1e5).half()   # overflows to +inf
    assert torch.isinf(G[2][5, 7])
    W0, M0 = [w.clone() for w in W], [x.clone() for x in M]
    ws = m.muon_step_batched(W, G, M, m.MuonHparams(skip_nonfinite=True))
    assert m.muon_query_status(ws) == m.MUON_STEP_SKIPPED
    for a, b in zip(W + M, W0 + M0):
        assert torch.equal(a, b)
    m.muon_step_batched(W, G, M, m.MuonHparams(), workspace=ws)
    assert m.muon_query_status(ws) == 0
    assert not bool(torch.isfinite(M[2]).all())
    for i in (0, 1):
        assert bool(torch.isfinite(W[i]).all()) and bool(torch.isfinite(M[i]).all())


def test_fp16_large_gradients_clip_by_global_norm(lib):
    """Large but finite fp16 gradients (near the top of the range): clipping
    by the global norm, as the oracle computes it."""
    W, G, M = make_fp16(SHAPES[:4], seed=73, g_std=3e3)
    W0, G0, M0 = host(W), host(G), host(M)
    assert all(np.isfinite(g).all() for g in G0)
    norm = float(np.sqrt(sum((g.astype(np.float64) ** 2).sum() for g in G0)))
    hp = m.MuonHparams(max_grad_norm=1e-3 * norm, skip_nonfinite=True)
    ws = m.muon_step_batched(W, G, M, hp)
    assert m.muon_query_status(ws) == 0
    ref, skipped = oracle.muon_step_list(W0, G0, M0, cfg_of(hp))
    assert not skipped
    for i, (oW, oM) in enumerate(ref):
        assert np.allclose(M[i].cpu().numpy(), oM, rtol=1e-6, atol=1e-9)
        dW = W[i].cpu().numpy().astype(np.float64) - W0[i]
        assert rel_fro(dW, oW.astype(np.float64) - W0[i]) < TOL
