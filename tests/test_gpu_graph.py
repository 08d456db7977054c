"""The Muon step captured as a CUDA graph.

muon_step_batched enqueues kernels and one memset only (the per-matrix
records travel as kernel parameters), so the whole launch sequence can be
captured once and replayed.  A replay must do exactly what the eager call
does: the same kernels on the same parameters, so W and M agree bit for bit
with eager steps on the same inputs, and the eager path itself agrees with
the oracle.  Covered here:

  * muon_step_graph_create / _launch through MuonBatch.capture, two replays
    with new gradient values written in place between them (a replay reads
    the current G);
  * several workspace chunks, the gradient guard (a replay over a NaN
    gradient skips the step and reports MUON_STEP_SKIPPED);
  * more matrices than one record upload carries (several upload launches);
  * a capture made by the caller (torch.cuda.graph) around MuonBatch.step,
    and around adamw_step_batched;
  * the launch count and timing rules of captured launches.
"""
import numpy as np
import pytest
import torch

import oracle
import optimizer_muon_step_gb300 as m

pytestmark = pytest.mark.gpu

DEV = "cuda"
TOL = 1e-2  # relative Frobenius error of the update, as in the other Muon tests


def rel_fro(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    return np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30)


def make_mats(shapes, dtypes, seed):
    gen = torch.Generator(device=DEV).manual_seed(seed)
    W, G, M = [], [], []
    for (r, c), dt in zip(shapes, dtypes):
        W.append(torch.randn(r, c, device=DEV, generator=gen) * 0.02)
        G.append((torch.randn(r, c, device=DEV, generator=gen) * 1e-2).to(dt))
        M.append(torch.randn(r, c, device=DEV, generator=gen) * 1e-2)
    return W, G, M


def clones(ts):
    return [t.clone() for t in ts]


def new_gradients(G, seed):
    gen = torch.Generator(device=DEV).manual_seed(seed)
    return [(torch.randn(g.shape, device=DEV, generator=gen) * 1e-2).to(g.dtype) for g in G]


def cfg_of(hp: m.MuonHparams) -> oracle.MuonConfig:
    return oracle.MuonConfig(lr=hp.lr, weight_decay=hp.weight_decay, momentum=hp.momentum,
                             nesterov=hp.nesterov, ns_steps=hp.ns_steps, ns_a=hp.ns_a, ns_b=hp.ns_b,
                             ns_c=hp.ns_c, norm_eps=hp.norm_eps, rms_scale=hp.rms_scale,
                             scale_mode=hp.scale_mode, skip_nonfinite=hp.skip_nonfinite,
                             max_grad_norm=hp.max_grad_norm, ns_coeffs=hp.ns_coeffs)


SHAPES = [(256, 512), (640, 160), (130, 70), (1024, 1024), (1100, 700)]  # single CTAs and CTA pairs
DTYPES = [torch.float32, torch.bfloat16, torch.float32, torch.bfloat16, torch.float32]


def test_graph_replays_equal_eager_steps_and_the_oracle(lib):
    W, G, M = make_mats(SHAPES, DTYPES, seed=31)
    We, Ge, Me = clones(W), clones(G), clones(M)      # eager
    Wg, Gg, Mg = clones(W), clones(G), clones(M)      # graph
    W0, G0, M0 = [t.float().cpu().numpy() for t in W], [t.float().cpu().numpy() for t in G], \
        [t.float().cpu().numpy() for t in M]
    hp = m.MuonHparams(lr=0.03, weight_decay=0.05)
    eager = m.MuonBatch(We, Ge, Me)
    graph = m.MuonBatch(Wg, Gg, Mg).capture(hp)
    try:
        eager.step(hp)
        graph.launch()
        torch.cuda.synchronize()
        for a, b in zip(We + Me, Wg + Mg):
            assert torch.equal(a, b)
        # the first replay against the oracle
        cfg = cfg_of(hp)
        for i in range(len(SHAPES)):
            oW, oM, _, _ = oracle.muon_step_matrix(W0[i], G0[i], M0[i], cfg)
            assert np.array_equal(Mg[i].cpu().numpy(), oM)
            dW = Wg[i].cpu().numpy().astype(np.float64) - W0[i]
            assert rel_fro(dW, oW.astype(np.float64) - W0[i]) < TOL
        # new gradient values, written in place, are what the next replay reads
        for ge, gg, new in zip(Ge, Gg, new_gradients(G, seed=32)):
            ge.copy_(new)
            gg.copy_(new)
        eager.step(hp)
        graph.launch()
        torch.cuda.synchronize()
        for a, b in zip(We + Me, Wg + Mg):
            assert torch.equal(a, b)
    finally:
        graph.destroy()


def test_graph_over_chunks_with_the_gradient_guard(lib):
    shapes = [(256, 512), (512, 256), (640, 160), (64, 64)]
    dtypes = [torch.float32, torch.bfloat16, torch.float32, torch.float32]
    W, G, M = make_mats(shapes, dtypes, seed=33)
    ws_bytes = max(m.muon_workspace_bytes_per_matrix(*s) for s in shapes)
    assert m.muon_plan(shapes, ws_bytes)["chunk_id"].max() >= 1  # several chunks
    We, Me, Wg, Mg = clones(W), clones(M), clones(W), clones(M)
    hp = m.MuonHparams(skip_nonfinite=True, max_grad_norm=0.5)
    eager = m.MuonBatch(We, G, Me, workspace=m.allocate_workspace(ws_bytes))
    gbatch = m.MuonBatch(Wg, G, Mg, workspace=m.allocate_workspace(ws_bytes))
    graph = gbatch.capture(hp)
    try:
        eager.step(hp)
        graph.launch()
        assert m.muon_query_status(gbatch.workspace) == 0
        for a, b in zip(We + Me, Wg + Mg):
            assert torch.equal(a, b)
        # a non-finite gradient: the replay changes nothing and reports the skip
        G[2][5, 3] = float("inf")
        Wk, Mk = clones(Wg), clones(Mg)
        graph.launch()
        assert m.muon_query_status(gbatch.workspace) == m.MUON_STEP_SKIPPED
        for a, b in zip(Wg + Mg, Wk + Mk):
            assert torch.equal(a, b)
        # clean again: the replay steps as the eager call does
        G[2][5, 3] = 0.0
        eager.step(hp)
        graph.launch()
        assert m.muon_query_status(gbatch.workspace) == 0
        for a, b in zip(We + Me, Wg + Mg):
            assert torch.equal(a, b)
    finally:
        graph.destroy()


def test_graph_with_several_record_uploads(lib):
    # 500 matrices: more records than one upload launch carries (224)
    shapes = [(24, 40)] * 250 + [(40, 24)] * 150 + [(64, 96)] * 100
    dtypes = [torch.bfloat16 if i % 3 == 0 else torch.float32 for i in range(len(shapes))]
    W, G, M = make_mats(shapes, dtypes, seed=34)
    W0 = [t.float().cpu().numpy() for t in W]
    G0 = [t.float().cpu().numpy() for t in G]
    M0 = [t.float().cpu().numpy() for t in M]
    We, Me, Wg, Mg = clones(W), clones(M), clones(W), clones(M)
    hp = m.MuonHparams()
    eager = m.MuonBatch(We, G, Me)
    graph = m.MuonBatch(Wg, G, Mg).capture(hp)
    try:
        timing_before = m.muon_launch_count()
        eager.step(hp)
        per_step = m.muon_launch_count() - timing_before
        graph.launch()
        torch.cuda.synchronize()
        for a, b in zip(We + Me, Wg + Mg):
            assert torch.equal(a, b)
        cfg = cfg_of(hp)
        for i in (0, 223, 224, 249, 250, 399, 400, 499):   # both sides of each upload boundary
            oW, oM, _, _ = oracle.muon_step_matrix(W0[i], G0[i], M0[i], cfg)
            assert np.array_equal(Mg[i].cpu().numpy(), oM)
            dW = Wg[i].cpu().numpy().astype(np.float64) - W0[i]
            assert rel_fro(dW, oW.astype(np.float64) - W0[i]) < TOL
        assert per_step >= 3 + 3 * hp.ns_steps   # three record uploads among them
    finally:
        graph.destroy()


def test_caller_capture_of_the_eager_step(lib):
    W, G, M = make_mats(SHAPES[:3], DTYPES[:3], seed=35)
    We, Me, Wg, Mg = clones(W), clones(M), clones(W), clones(M)
    hp = m.MuonHparams()
    eager = m.MuonBatch(We, G, Me)
    gbatch = m.MuonBatch(Wg, G, Mg)
    gbatch.step(hp)   # warm-up outside the capture (kernel attributes)
    eager.step(hp)
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    cg = torch.cuda.CUDAGraph()
    with torch.cuda.graph(cg, stream=side):
        gbatch.step(hp, stream=side)
    for _ in range(2):
        eager.step(hp)
        cg.replay()
    torch.cuda.synchronize()
    for a, b in zip(We + Me, Wg + Mg):
        assert torch.equal(a, b)


def test_captured_launches_are_counted_per_replay_and_never_timed(lib):
    W, G, M = make_mats(SHAPES[:2], DTYPES[:2], seed=36)
    batch = m.MuonBatch(W, G, M)
    hp = m.MuonHparams()
    n0 = m.muon_launch_count()
    batch.step(hp)
    per_step = m.muon_launch_count() - n0
    m.muon_set_timing(1)
    try:
        n1 = m.muon_launch_count()
        graph = batch.capture(hp)
        assert m.muon_launch_count() == n1          # capturing launches nothing
        graph.launch()
        graph.launch()
        assert m.muon_launch_count() == n1 + 2 * per_step
        torch.cuda.synchronize()
        assert all(cnt == 0 for _, cnt in m.muon_timing_read().values())
        graph.destroy()
    finally:
        m.muon_set_timing(0)


def test_caller_capture_of_batched_adamw(lib):
    """adamw_step_batched enqueues kernels only (its tensor table is a kernel
    parameter), so a graph captured by the caller replays the same update."""
    gen = torch.Generator(device=DEV).manual_seed(37)
    sizes = [5000, 1, 333, 1 << 16]
    quads = [tuple(torch.randn(n, device=DEV, generator=gen).abs() * 1e-3 for _ in range(4)) for n in sizes]
    twins = [tuple(x.clone() for x in q) for q in quads]
    hp = m.AdamwHparams()
    m.adamw_step_batched(quads, hp, step=7)   # warm-up outside the capture
    m.adamw_step_batched(twins, hp, step=7)
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    cg = torch.cuda.CUDAGraph()
    with torch.cuda.graph(cg, stream=side):
        m.adamw_step_batched(quads, hp, step=7, stream=side)
    for _ in range(2):
        cg.replay()
        m.adamw_step_batched(twins, hp, step=7)
    torch.cuda.synchronize()
    for a, b in zip(quads, twins):
        for x, y in zip(a, b):
            assert torch.equal(x, y)
