"""The allocation-free Muon step (muon_step_batched_noalloc).

Some callers cannot allocate device memory -- an optimizer plug-in inside a
framework that owns all device memory through its own pool, or a C caller
with no device allocator -- so they cannot provide the workspace that
muon_step_batched needs.  The allocation-free entry point uses a static
device array inside the library instead.  This test calls it through the C
ABI and checks it against muon_step_batched with a caller workspace, on two
calls in a row (the second call finds the previous call's data still in the
shared scratch).  Both run the same kernels on the same inputs -- only the
workspace and its cut into chunks differ, which changes no bit -- so W and M
must be bit-identical; a stale record or buffer left in the scratch by the
previous call would show up as a difference.  One matrix is also checked
against the oracle.  This file sorts last so that a stop-at-first-failure
run has already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import optimizer_muon_step_gb300 as m

pytestmark = pytest.mark.gpu

DEV = "cuda"
TOL = 1e-2  # relative Frobenius error of the update against the oracle, as in the other Muon tests


def _batch(W, G, M):
    arr = (m.MuonMatrix * len(W))()
    for i, (w, g, x) in enumerate(zip(W, G, M)):
        arr[i].W, arr[i].G, arr[i].M = w.data_ptr(), g.data_ptr(), x.data_ptr()
        arr[i].rows, arr[i].cols = w.shape
        arr[i].g_dtype = m.MUON_BF16 if g.dtype == torch.bfloat16 else m.MUON_F32
    return arr


def rel_fro(a, b):
    a, b = a.double(), b.double()
    return float(torch.linalg.norm(a - b) / torch.linalg.norm(b))


def test_noalloc_matches_workspace_entry_point(lib):
    shapes = [(256, 512), (512, 256), (7, 13), (130, 70), (2048, 2048), (2048, 5632)]
    dtypes = [torch.float32, torch.bfloat16, torch.float32, torch.bfloat16, torch.float32, torch.bfloat16]
    gen = torch.Generator(device=DEV).manual_seed(7)
    W, G, M = [], [], []
    for (r, c), dt in zip(shapes, dtypes):
        W.append(torch.randn(r, c, device=DEV, generator=gen) * 0.02)
        G.append((torch.randn(r, c, device=DEV, generator=gen) * 1e-2).to(dt))
        M.append(torch.randn(r, c, device=DEV, generator=gen) * 1e-2)
    Wa, Ma = [w.clone() for w in W], [x.clone() for x in M]   # caller-workspace path
    Wb, Mb = [w.clone() for w in W], [x.clone() for x in M]   # allocation-free path
    hp = m.MuonHparams()
    ws = m.allocate_workspace(m.muon_workspace_size(shapes, 1 << 34))
    arr_b = _batch(Wb, G, Mb)
    h = hp._c()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    big = shapes.index((2048, 5632))
    for call in range(2):
        host = (Wb[big].cpu().numpy(), G[big].float().cpu().numpy(), Mb[big].cpu().numpy())
        m.muon_step_batched(Wa, G, Ma, hp, workspace=ws)
        st = lib.muon_step_batched_noalloc(ctypes.cast(arr_b, ctypes.c_void_p), len(shapes),
                                           ctypes.byref(h), stream)
        assert st == 0, st
        torch.cuda.synchronize()
        for i in range(len(shapes)):
            assert torch.equal(Ma[i], Mb[i]), (call, i)
            assert torch.equal(Wa[i], Wb[i]), (call, i)
        oW, oM, _, _ = oracle.muon_step_matrix(*host, oracle.MuonConfig())
        assert np.array_equal(Mb[big].cpu().numpy(), oM), call
        W0 = host[0].astype(np.float64)
        err = rel_fro(torch.from_numpy(Wb[big].cpu().numpy() - W0), torch.from_numpy(oW - W0))
        assert err <= TOL, (call, err)


def test_noalloc_rejects_matrices_beyond_the_scratch(lib):
    arr = (m.MuonMatrix * 2)()
    for i in range(2):
        arr[i].W = arr[i].G = arr[i].M = 1 << 20  # never dereferenced: rejected first
    arr[0].rows, arr[0].cols = 64, 64
    arr[1].rows, arr[1].cols = 4096, 8192  # needs > 64 MiB of scratch
    assert m.muon_workspace_bytes_per_matrix(4096, 8192) > (64 << 20)
    h = m.MuonHparams()._c()
    st = lib.muon_step_batched_noalloc(ctypes.cast(arr, ctypes.c_void_p), 2, ctypes.byref(h), None)
    assert st == 4  # MUON_ERR_WORKSPACE_TOO_SMALL, nothing enqueued
