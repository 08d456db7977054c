"""Full-size workloads on the GPU, in the launch configuration bench.py uses
(one MuonBatch over every matrix, 16 GiB workspace budget), checked against
the oracle.

Per workload:
  * sampled matrices (seeded choice) run through the full oracle step:
    momentum M bit-exact, Muon update dW within rel. Frobenius 1e-2;
  * the oracle's own spread beside the GPU's error: for one sampled matrix
    of each distinct (m', n') the oracle also runs its variants, each as
    faithful to the method as the reference evaluation -- the NS products
    accumulated in fp32 with one rounding per addition (acc32) or with one
    round-toward-zero per 16-product block (rz16, how tensor-core fp32
    accumulation behaves in measurement), and the cast to bf16 after the
    normalisation instead of before it (cast).  The GPU (fp32 accumulation
    in the tensor cores, the reference's rounding points) must sit within
    SPREAD_FACTOR of the larger fp32 spread, not merely under 1e-2.  With
    MUON_PARITY_REPORT=<path> every comparison is appended there as one
    JSON line;
  * every matrix (c2, c4): momentum M bit-exact against the oracle's
    element-wise momentum; every matrix (c1-c4): the update's
    singular-value content checked through the
    identity rms(dW_update) = lr * 0.2 * rms(sigma(O)) with sigma(O) in the
    quintic's band (a property that holds at any size);
  * the 7168x18432 / 7168x7168 layer is beyond the oracle's reach (about
    10 TFLOP per matrix on the CPU), so only the properties apply there,
    plus the band of the orthogonalised output's singular values.
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
BUDGET = 16 << 30
# The GPU's error against the fp64-accumulating oracle may be at most this
# multiple of the larger of the acc32 and rz16 variants' errors: all three
# accumulate in fp32, so they sit a similar distance from the fp64
# evaluation (measured: the GPU at 0.96-1.10 times).
SPREAD_FACTOR = 1.5


def rel_fro(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    return np.linalg.norm(a - b) / np.linalg.norm(b)


def oracle_cfg():
    return oracle.MuonConfig(**workloads.MUON_HPARAMS)


def run_workload(name, sample):
    w = workloads.get(name)
    t = workloads.make_muon(w, device=DEV)
    host = {i: (t.W[i].cpu().numpy(), t.G[i].float().cpu().numpy(), t.M[i].cpu().numpy())
            for i in sample}
    W_before = [x.clone() for x in t.W] if w.muon_params < 1e10 else None
    batch = m.MuonBatch(t.W, t.G, t.M, budget_bytes=BUDGET)
    hp = m.MuonHparams(**workloads.MUON_HPARAMS)
    batch.step(hp)
    assert m.muon_query_status(batch.workspace) == 0
    return w, t, host, W_before, hp


def report(rec):
    path = os.environ.get("MUON_PARITY_REPORT")
    if path:
        with open(path, "a") as f:
            f.write(json.dumps(rec) + "\n")


def check_sampled(t, host, w=None):
    """Sampled matrices against the oracle; for the first sampled matrix of
    each distinct (m', n') also the oracle's spread (acc32, rz16 and cast
    variants)."""
    cfg = oracle_cfg()
    seen = set()
    for i, (W0, G0, M0) in host.items():
        oW, oM, _, _ = oracle.muon_step_matrix(W0, G0, M0, cfg)
        assert np.array_equal(t.M[i].cpu().numpy(), oM), i
        W1 = t.W[i].cpu().numpy()
        W0d = W0.astype(np.float64)
        d_ref = oW.astype(np.float64) - W0d
        err = rel_fro(W1.astype(np.float64) - W0d, d_ref)
        rec = {"workload": w.name if w else None, "matrix": i, "shape": list(W0.shape), "gpu_err": err}
        key = (min(W0.shape), max(W0.shape))
        if key not in seen:
            seen.add(key)
            for name, kw in (("acc32", dict(accum=oracle.ACC_FP32)), ("rz16", dict(accum=oracle.ACC_FP32_RZ16)),
                             ("cast", dict(cast_after_scale=True))):
                var = oracle.muon_step_matrix(W0, G0, M0, cfg, **kw)[0]
                rec["spread_" + name] = rel_fro(var.astype(np.float64) - W0d, d_ref)
        report(rec)
        assert err < TOL, (i, err)
        if "spread_acc32" in rec:
            assert err <= SPREAD_FACTOR * max(rec["spread_acc32"], rec["spread_rz16"]), rec


def update_sigma_rms(W0, W1, hp, rows, cols):
    """rms(sigma(O)) recovered from dW = -lr (wd W0 + 0.2 sqrt(n') O)."""
    lr, wd = np.float32(hp.lr), np.float32(hp.weight_decay)
    d = (W1.double() - W0.double()) / float(lr) + float(wd) * W0.double()
    scale = hp.rms_scale * max(rows, cols) ** 0.5
    O = -d / scale
    return float(torch.sqrt((O * O).sum() / min(rows, cols)))


def check_update_rms(w, t, W_before, hp):
    for i, s in enumerate(w.matrices):
        if W_before is not None:
            r = update_sigma_rms(W_before[i], t.W[i], hp, s.rows, s.cols)
            assert 0.45 < r < 1.25, (i, r)


@pytest.mark.parametrize("name", ["c1", "c3"])
def test_workload_fp32_grads(lib, name):
    w = workloads.get(name)
    sample = workloads.parity_sample(w)
    if name == "c3":
        # one matrix of each distinct shape keeps the oracle's share short
        seen, pick = set(), []
        for i in sample:
            key = (w.matrices[i].rows, w.matrices[i].cols)
            if key not in seen:
                seen.add(key)
                pick.append(i)
        sample = pick
    w, t, host, W_before, hp = run_workload(name, sample)
    check_sampled(t, host, w)
    check_update_rms(w, t, W_before, hp)


def test_workload_c2_dense_decoder(lib):
    w = workloads.get("c2")
    # the first and the last layer's q (2048x2048), gate (5632x2048, tall) and
    # down (2048x5632); seven matrices per layer
    last = 7 * (len(w.matrices) // 7 - 1)
    sample = [0, 4, 6, last, last + 4, last + 6]
    # momentum of every matrix is checked element-wise against the oracle
    t0 = workloads.make_muon(w, device=DEV)
    G_all = [g.float().cpu().numpy() for g in t0.G]
    M_all = [x.cpu().numpy() for x in t0.M]
    del t0
    w, t, host, W_before, hp = run_workload("c2", sample)
    check_sampled(t, host, w)
    for i in range(len(w.matrices)):
        oM, _ = oracle.momentum(G_all[i], M_all[i], hp.momentum, hp.nesterov)
        assert np.array_equal(t.M[i].cpu().numpy(), oM), i
    check_update_rms(w, t, W_before, hp)


def scalar_map(sigma, steps=5):
    """The NS iteration restricted to one singular value (fp32 coefficients)."""
    a, b, c = (float(np.float32(x)) for x in oracle.QUINTIC)
    s = sigma.clone()
    for _ in range(steps):
        s = a * s + b * s ** 3 + c * s ** 5
    return s


def spectrum(X):
    """Singular values of a wide fp64 CUDA matrix via eigvalsh of X X^T."""
    return torch.linalg.eigvalsh(X @ X.t()).clamp_min(0).sqrt()


def test_workload_c4_large_layer_properties(lib):
    """7168 x 18432 layer, beyond the oracle's reach: momentum is bit-exact
    for every matrix, and the orthogonalised update has exactly the
    spectrum NS must produce: NS maps each singular value sigma of the
    normalised input to p^5(sigma) independently, so the sorted output
    spectrum (recovered from dW) equals the sorted p^5 of the input
    spectrum (from the oracle's look-ahead u), up to bf16 noise."""
    w = workloads.get("c4")
    t = workloads.make_muon(w, device=DEV)
    G_host = [g.float().cpu().numpy() for g in t.G]
    M_host = [x.cpu().numpy() for x in t.M]
    W0 = [x.clone() for x in t.W]
    batch = m.MuonBatch(t.W, t.G, t.M, budget_bytes=BUDGET)
    hp = m.MuonHparams(**workloads.MUON_HPARAMS)
    batch.step(hp)
    assert m.muon_query_status(batch.workspace) == 0
    for i, s in enumerate(w.matrices):
        oM, u = oracle.momentum(G_host[i], M_host[i], hp.momentum, hp.nesterov)
        assert np.array_equal(t.M[i].cpu().numpy(), oM), i
        U = torch.from_numpy(u).to(DEV).double()
        X0 = U / torch.linalg.norm(U)
        lr, wd = float(np.float32(hp.lr)), float(np.float32(hp.weight_decay))
        d = (t.W[i].double() - W0[i].double()) / lr + wd * W0[i].double()
        O = -d / (hp.rms_scale * max(s.rows, s.cols) ** 0.5)
        if s.rows > s.cols:
            O, X0 = O.t(), X0.t()
        expect = torch.sort(scalar_map(spectrum(X0))).values
        got = torch.sort(spectrum(O)).values
        diff = (got - expect).abs()
        assert diff.max().item() < 0.03 and diff.mean().item() < 0.005, (i, diff.max().item(), diff.mean().item())
        assert got.max().item() < 1.21
        del U, X0, d, O


def test_workload_c5_full_mixed_step(lib):
    """6144 expert matrices under Muon plus AdamW on the 163840x7168
    embedding and LM head, the largest workload."""
    w = workloads.get("c5")
    sample = workloads.parity_sample(w)
    sample = [sample[0], sample[-1]]   # a wide gate or up, and a tall down
    w, t, host, _, hp = run_workload("c5", sample)
    check_sampled(t, host, w)
    del t
    torch.cuda.empty_cache()
    ahp = m.AdamwHparams(**workloads.ADAMW_HPARAMS)
    rng = np.random.default_rng(w.seed + 100)
    win = 1 << 20
    for i, (r, c) in enumerate(w.adamw_shapes):
        n = r * c
        b = workloads.make_adamw(n, seed=w.seed + i, device=DEV)
        starts = [0, n - 16 * win] + sorted(int(x) for x in rng.integers(0, n - win, 8))
        lens = [16 * win, 16 * win] + [win] * 8
        before = [[x[s:s + L].cpu().numpy() for x in (b.p, b.g, b.m, b.v)] for s, L in zip(starts, lens)]
        m.adamw_step(b.p, b.g, b.m, b.v, ahp, workloads.ADAMW_STEP)
        for (s, L), (p0, g0, m0, v0) in zip(zip(starts, lens), before):
            rp, rm, rv = oracle.adamw_step(p0, g0, m0, v0, oracle.AdamwConfig(**workloads.ADAMW_HPARAMS),
                                           t=workloads.ADAMW_STEP)
            assert np.array_equal(b.p[s:s + L].cpu().numpy(), rp)
            assert np.array_equal(b.m[s:s + L].cpu().numpy(), rm)
            assert np.array_equal(b.v[s:s + L].cpu().numpy(), rv)
        del b
        torch.cuda.empty_cache()


def test_nonfinite_gradient_propagates_without_trap(lib):
    """A NaN in one matrix's gradient makes that matrix's update NaN (the
    step does not guard against non-finite values) and leaves the others
    untouched; the device status stays clean."""
    gen = torch.Generator(device=DEV).manual_seed(0)
    W = [torch.randn(128, 256, device=DEV, generator=gen) * 0.02 for _ in range(2)]
    G = [torch.randn(128, 256, device=DEV, generator=gen) * 1e-2 for _ in range(2)]
    M = [torch.zeros(128, 256, device=DEV) for _ in range(2)]
    G[0][3, 5] = float("nan")
    W1 = W[1].cpu().numpy()
    G1, M1 = G[1].cpu().numpy(), M[1].cpu().numpy()
    ws = m.muon_step_batched(W, G, M, m.MuonHparams())
    assert m.muon_query_status(ws) == 0
    assert torch.isnan(W[0]).all()
    oW, _, _, _ = oracle.muon_step_matrix(W1, G1, M1, oracle.MuonConfig())
    assert rel_fro(W[1].cpu().numpy().astype(np.float64) - W1, oW.astype(np.float64) - W1) < TOL


def test_empty_batch_is_noop(lib):
    ws = m.allocate_workspace(4096)
    m.muon_step_batched([], [], [], m.MuonHparams(), workspace=ws)
    x = torch.zeros(0, device=DEV)
    m.adamw_step(x, x.clone(), x.clone(), x.clone(), m.AdamwHparams(), 1)


@pytest.mark.skipif(not os.environ.get("MUON_SLOW"), reason="about 4 minutes of oracle time; set MUON_SLOW=1")
def test_workload_c4_attention_matrix_against_the_oracle(lib):
    """One 7168 x 7168 matrix of the large layer (its q projection, bf16
    gradient) through the whole step against the oracle: momentum bit-exact,
    the update within 1e-2 and within SPREAD_FACTOR of the oracle's rz16
    variant (fp32 accumulation rounding toward zero per 16-product block).
    The 7168 x 18432 matrices, about 23 TFLOP each for the oracle, stay with
    the singular-value check above."""
    w = workloads.get("c4")
    i = 3
    assert w.matrices[i].name == "q" and (w.matrices[i].rows, w.matrices[i].cols) == (7168, 7168)
    w, t, host, _, hp = run_workload("c4", [i])
    W0, G0, M0 = host[i]
    cfg = oracle_cfg()
    oW, oM, _, _ = oracle.muon_step_matrix(W0, G0, M0, cfg)
    assert np.array_equal(t.M[i].cpu().numpy(), oM)
    W0d = W0.astype(np.float64)
    d_ref = oW.astype(np.float64) - W0d
    err = rel_fro(t.W[i].cpu().numpy().astype(np.float64) - W0d, d_ref)
    zW = oracle.muon_step_matrix(W0, G0, M0, cfg, accum=oracle.ACC_FP32_RZ16)[0]
    spread = rel_fro(zW.astype(np.float64) - W0d, d_ref)
    report({"workload": "c4", "matrix": i, "shape": [7168, 7168], "gpu_err": err, "spread_rz16": spread})
    assert err < TOL
    assert err <= SPREAD_FACTOR * spread, (err, spread)
