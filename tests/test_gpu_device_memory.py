"""The C ABI refuses buffers that are not the current device's.

Every call that launches kernels asks the driver who owns each buffer it is
given and returns MUON_ERR_INVALID_ARG (1), with nothing enqueued, when a
buffer is host memory, another device's memory or an unknown address.
Checked here through ctypes with pinned host buffers (the one kind of
foreign memory a single-GPU machine can hand over without risk: a kernel that
did reach it would find it mapped, not fault), each in one position of an
otherwise valid call: the refused call changes nothing, and the same call
with device buffers then runs and matches the oracle.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import optimizer_muon_step_gb300 as m

pytestmark = pytest.mark.gpu

DEV = "cuda"
INVALID_ARG = 1


def _muon_batch(W, G, M):
    arr = (m.MuonMatrix * len(W))()
    for i, (w, g, x) in enumerate(zip(W, G, M)):
        arr[i].W, arr[i].G, arr[i].M = w.data_ptr(), g.data_ptr(), x.data_ptr()
        arr[i].rows, arr[i].cols = w.shape
        arr[i].g_dtype = m.MUON_F32
    return arr


def _pinned_like(t):
    return torch.empty(t.shape, dtype=t.dtype, pin_memory=True).copy_(t)


def test_muon_step_refuses_host_buffers(lib):
    gen = torch.Generator(device=DEV).manual_seed(61)
    shapes = [(256, 512), (130, 70)]
    W = [torch.randn(*s, device=DEV, generator=gen) * 0.02 for s in shapes]
    G = [torch.randn(*s, device=DEV, generator=gen) * 1e-2 for s in shapes]
    M = [torch.randn(*s, device=DEV, generator=gen) * 1e-2 for s in shapes]
    W0, G0, M0 = ([x.cpu().numpy() for x in xs] for xs in (W, G, M))
    ws = m.allocate_workspace(m.muon_workspace_size(shapes, 1 << 30))
    h = m.MuonHparams()._c()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)

    def call(Ws, Gs, Ms, workspace=ws):
        return lib.muon_step_batched(_muon_batch(Ws, Gs, Ms), len(Ws), ctypes.byref(h),
                                     ctypes.c_void_p(workspace.data_ptr()), workspace.numel(), stream)

    assert call([W[0], _pinned_like(W[1])], G, M) == INVALID_ARG
    assert call(W, [_pinned_like(G[0]), G[1]], M) == INVALID_ARG
    assert call(W, G, [M[0], _pinned_like(M[1])]) == INVALID_ARG
    assert call(W, G, M, workspace=_pinned_like(ws[:ws.numel()])) == INVALID_ARG
    assert lib.muon_step_batched_noalloc(_muon_batch([W[0], _pinned_like(W[1])], G, M), 2, ctypes.byref(h),
                                         stream) == INVALID_ARG
    stats = torch.empty(2 * 16, dtype=torch.uint8, pin_memory=True)
    assert lib.muon_step_batched_stats(_muon_batch(W, G, M), 2, ctypes.byref(h), ctypes.c_void_p(ws.data_ptr()),
                                       ws.numel(), ctypes.c_void_p(stats.data_ptr()), stream) == INVALID_ARG
    graph = ctypes.c_void_p(123)
    W_host = [W[0], _pinned_like(W[1])]
    assert lib.muon_step_graph_create(_muon_batch(W_host, G, M), 2, ctypes.byref(h),
                                      ctypes.c_void_p(ws.data_ptr()), ws.numel(), ctypes.byref(graph)) == INVALID_ARG
    assert graph.value is None
    torch.cuda.synchronize()
    for i in range(2):    # nothing was enqueued
        assert np.array_equal(W[i].cpu().numpy(), W0[i]) and np.array_equal(M[i].cpu().numpy(), M0[i])

    assert call(W, G, M) == 0
    torch.cuda.synchronize()
    for i in range(2):
        oW, oM, _, _ = oracle.muon_step_matrix(W0[i], G0[i], M0[i], oracle.MuonConfig())
        assert np.array_equal(M[i].cpu().numpy(), oM)
        dW = W[i].cpu().numpy().astype(np.float64) - W0[i]
        ref = oW.astype(np.float64) - W0[i]
        assert np.linalg.norm(dW - ref) / np.linalg.norm(ref) < 1e-2


def test_adamw_and_newton_schulz_refuse_host_buffers(lib):
    gen = torch.Generator(device=DEV).manual_seed(62)
    n = 4099
    p, g, mm, v = (torch.randn(n, device=DEV, generator=gen) * 1e-2 for _ in range(4))
    v.abs_()
    host = [x.cpu().numpy() for x in (p, g, mm, v)]
    h = m.AdamwHparams(lr=1e-3)._c()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    ptr = lambda t: ctypes.c_void_p(t.data_ptr())
    assert lib.adamw_step(ptr(_pinned_like(p)), ptr(g), ptr(mm), ptr(v), n, ctypes.byref(h), 1, stream) == INVALID_ARG
    batch = (m.AdamwTensor * 2)()
    q = torch.randn(64, device=DEV, generator=gen)
    qs = [q.clone() for _ in range(3)] + [q.abs()]
    for k, (t, pinned) in enumerate([((p, g, mm, v), False), (tuple(qs), True)]):
        tt = list(t)
        if pinned:
            tt[3] = _pinned_like(tt[3])
        batch[k].p, batch[k].g, batch[k].m, batch[k].v = (x.data_ptr() for x in tt)
        batch[k].n = tt[0].numel()
    assert lib.adamw_step_batched(batch, 2, ctypes.byref(h), 1, stream) == INVALID_ARG
    torch.cuda.synchronize()
    assert np.array_equal(p.cpu().numpy(), host[0]) and np.array_equal(v.cpu().numpy(), host[3])
    assert lib.adamw_step(ptr(p), ptr(g), ptr(mm), ptr(v), n, ctypes.byref(h), 1, stream) == 0
    torch.cuda.synchronize()
    rp, _, _ = oracle.adamw_step(*host, oracle.AdamwConfig(lr=1e-3), t=1)
    assert np.array_equal(p.cpu().numpy(), rp)

    X = torch.randn(2, 128, 256, device=DEV, generator=gen).to(torch.bfloat16)
    out_host = torch.empty(2, 128, 256, dtype=torch.bfloat16, pin_memory=True)
    ws = m.allocate_workspace(2 * m.muon_workspace_bytes_per_matrix(128, 256))
    coeffs = (ctypes.c_float * 3)(*oracle.QUINTIC)
    assert lib.muon_newton_schulz(ptr(X), ptr(out_host), 2, 128, 256, 5, coeffs, 1, ptr(ws), ws.numel(),
                                  stream) == INVALID_ARG
    assert lib.muon_check_bounded_wait(ptr(_pinned_like(ws[:256])), 1000, stream) == INVALID_ARG
