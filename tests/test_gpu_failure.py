"""Failure detection on the GPU without a fault: every wait in the kernels
is bounded, and a wait that runs out leaves a status the host reads while
the context stays usable.  The self-check entry point makes one such wait
run out (an mbarrier nothing arrives on) with a short limit."""
import time

import numpy as np
import pytest
import torch

import oracle
import optimizer_muon_step_gb300 as m

pytestmark = pytest.mark.gpu

DEV = "cuda"


def test_bounded_wait_reports_timeout_and_context_survives(lib):
    ws = m.allocate_workspace(1 << 22)
    t0 = time.perf_counter()
    m.muon_check_bounded_wait(ws, limit_us=20000)
    assert m.muon_query_status(ws) == 6  # MUON_ERR_TIMEOUT
    elapsed = time.perf_counter() - t0
    assert 0.015 < elapsed < 5.0  # the wait ran its limit, then returned
    # the status word was cleared by the query, and the context still runs a step
    assert m.muon_query_status(ws) == 0
    gen = torch.Generator(device=DEV).manual_seed(3)
    W = [torch.randn(96, 160, device=DEV, generator=gen) * 0.02]
    G = [torch.randn(96, 160, device=DEV, generator=gen) * 1e-2]
    M = [torch.randn(96, 160, device=DEV, generator=gen) * 1e-2]
    W0, G0, M0 = (x[0].cpu().numpy() for x in (W, G, M))
    m.muon_step_batched(W, G, M, m.MuonHparams(), workspace=ws)
    assert m.muon_query_status(ws) == 0
    oW, oM, _, _ = oracle.muon_step_matrix(W0, G0, M0)
    assert np.array_equal(M[0].cpu().numpy(), oM)
    d = W[0].cpu().numpy().astype(np.float64) - W0
    assert np.linalg.norm(d - (oW - W0)) / np.linalg.norm(oW - W0) < 1e-2


def test_bounded_wait_argument_checks(lib):
    ws = m.allocate_workspace(4096)
    for bad in (0, -5, 10 ** 8):
        with pytest.raises(m.MuonError):
            m.muon_check_bounded_wait(ws, limit_us=bad)


_DEBUG_SCRIPT = """
import sys
import torch
sys.path.insert(0, sys.argv[2])
import optimizer_muon_step_gb300 as m
gen = torch.Generator(device="cuda").manual_seed(61)
shapes = [(256, 512), (130, 70), (520, 256)]
W = [torch.randn(r, c, device="cuda", generator=gen) * 0.02 for r, c in shapes]
G = [torch.randn(r, c, device="cuda", generator=gen) * 1e-2 for r, c in shapes]
M = [torch.randn(r, c, device="cuda", generator=gen) * 1e-2 for r, c in shapes]
ws = m.muon_step_batched(W, G, M, m.MuonHparams(skip_nonfinite=True))
m.adamw_step(W[0].view(-1), G[0].view(-1), M[0].view(-1), W[1].new_zeros(W[0].numel()), m.AdamwHparams(), 1)
torch.cuda.synchronize()
assert m.muon_query_status(ws) == 0
torch.save([w.cpu() for w in W] + [x.cpu() for x in M], sys.argv[1])
"""


def test_debug_mode_synchronises_and_changes_nothing(lib, tmp_path):
    """MUON_DEBUG=1 waits for every launch and names a failed one on stderr;
    a clean run prints nothing and computes the same bits as a normal run
    (each run in its own process: the variable is read once per process)."""
    import os
    import subprocess
    import sys
    from conftest import ROOT
    script = tmp_path / "debug_step.py"
    script.write_text(_DEBUG_SCRIPT)
    out = {}
    for flag in ("1", "0"):
        path = tmp_path / f"out_{flag}.pt"
        r = subprocess.run([sys.executable, str(script), str(path), ROOT], capture_output=True, text=True,
                           env=dict(os.environ, MUON_DEBUG=flag), timeout=600)
        assert r.returncode == 0, r.stderr[-2000:]
        assert "muon: kernel" not in r.stderr
        out[flag] = torch.load(path)
    for a, b in zip(out["1"], out["0"]):
        assert torch.equal(a, b)
