"""The benchmark's end-to-end path on the GPU: the step fed from pinned host
buffers through bench.py's staging ring, pipelined over three streams.

Twelve experts of the mixed step (gate, up, down, four times) and two small
AdamW buffers run with a staging slot of three experts' W, G and M, so the
step is cut into four Muon pieces of the same shapes and several AdamW
chunks.  Every input slot holds the first piece's data and is re-sent for
every piece, so after the run every Muon piece must hold exactly one step
applied to the first piece's inputs, and every AdamW chunk one AdamW step
applied to a prefix of the first chunk's inputs: the copies in landed where
the step reads, and the step ran on them.  Bit-exact against the library's
own direct calls; the byte counts are those of every input and result.
"""
import pytest
import torch

import bench
import optimizer_muon_step_gb300 as m
import workloads

pytestmark = pytest.mark.gpu


def test_e2e_pipeline_feeds_every_piece(lib):
    dev = torch.device("cuda")
    w = workloads.get("c5")
    w.matrices = w.matrices[:12]
    ws = bench.WorkloadStep(m, w, dev, 16 << 30, with_adamw=True, adamw_params=(13 << 20) + 7)
    nel = w.matrices[0].rows * w.matrices[0].cols
    slot = 3 * nel * 12                                      # W, G, M of three experts, fp32
    W0 = [x.clone() for x in ws.tens.W[:3]]
    G0 = [x.clone() for x in ws.tens.G[:3]]
    M0 = [x.clone() for x in ws.tens.M[:3]]
    chunk = (slot // 16) // 4 * 4
    first = [x[:chunk].clone() for x in (ws.adamw[0].p, ws.adamw[0].g, ws.adamw[0].m, ws.adamw[0].v)]

    pieces = bench.e2e_pieces(ws, slot)
    assert [p[3] for p in pieces if p[0] == "muon"] == [(0, 3), (3, 6), (6, 9), (9, 12)]
    res = bench.run_e2e(m, ws, 1, 1, lambda: None, lambda x: x, n_steps=2, slot_bytes=slot)
    torch.cuda.synchronize()

    m.muon_step_batched(W0, G0, M0, ws.hp)                   # the expected Muon piece
    for k in range(4):
        for i in range(3):
            assert torch.equal(ws.tens.W[3 * k + i], W0[i]), (k, i)
            assert torch.equal(ws.tens.M[3 * k + i], M0[i]), (k, i)
    n_chunks = 0
    for buf in ws.adamw:
        n = buf.p.numel()
        for lo in range(0, n, chunk):
            hi = min(n, lo + chunk)
            p, g, mm, v = (x[:hi - lo].clone() for x in first)
            m.adamw_step(p, g, mm, v, ws.ahp, workloads.ADAMW_STEP)
            assert torch.equal(buf.p[lo:hi], p) and torch.equal(buf.m[lo:hi], mm) and torch.equal(buf.v[lo:hi], v)
            n_chunks += 1
    assert n_chunks >= 4
    assert res["h2d_bytes_per_step"] == 12 * nel * 12 + ws.adamw_params * 16
    assert res["d2h_bytes_per_step"] == 12 * nel * 8 + ws.adamw_params * 12
    assert res["ms_per_step"] > 0
