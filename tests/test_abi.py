"""Host-side checks of the C ABI: the library loads, exports what the header
declares, validates its arguments, and its plan equals the oracle's bit for
bit.  No GPU needed."""
import ctypes
import os
import re

import numpy as np
import torch
import pytest

import oracle
import optimizer_muon_step_gb300 as m
import workloads
from conftest import ROOT, cuda_available


@pytest.fixture(scope="module")
def built():
    from optimizer_muon_step_gb300 import build
    build.build()
    return m.load_library()


def header_functions():
    text = open(os.path.join(ROOT, "include", "muon_step.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*[A-Za-z_][\w\s\*]*?\b(\w+)\s*\(", text, flags=re.M)))


def test_header_symbols_exported(built):
    names = header_functions()
    assert set(names) == set(m.EXPORTS)
    for name in names:
        assert hasattr(built, name), name


def test_version_and_status_strings(built):
    assert m.version() >= 100
    assert built.muon_status_string(0) == b"ok"
    assert b"workspace" in built.muon_status_string(4)


@pytest.mark.parametrize("shape", [(1, 1), (7, 13), (13, 7), (2048, 2048), (5632, 2048), (1408, 2048),
                                   (18432, 7168)])
def test_workspace_bytes_match_oracle(built, shape):
    r, c = shape
    assert m.muon_workspace_bytes_per_matrix(r, c) == oracle.ws_bytes_per_matrix(min(r, c), max(r, c))


def _plan_equal(shapes, ws):
    got = m.muon_plan(shapes, ws)
    ref = oracle.plan(shapes, ws)
    for f in ("mat_idx", "transposed", "group_id", "slot", "chunk_id", "mp", "np"):
        assert np.array_equal(got[f], ref[f]), f


def test_plan_bit_exact_random(built):
    rng = np.random.default_rng(5)
    dims = [1, 7, 8, 64, 1408, 2048, 5632]
    for _ in range(100):
        n = int(rng.integers(0, 50))
        shapes = [(int(rng.choice(dims)), int(rng.choice(dims))) for _ in range(n)]
        need = max([oracle.ws_bytes_per_matrix(min(s), max(s)) for s in shapes] or [1])
        _plan_equal(shapes, int(need * rng.uniform(1, 8)))


@pytest.mark.parametrize("name", ["c1", "c2", "c3", "c4", "c5"])
@pytest.mark.parametrize("budget_gb", [0.25, 4, 16, 1000])
def test_plan_bit_exact_workloads(built, name, budget_gb):
    shapes = [(s.rows, s.cols) for s in workloads.get(name).matrices]
    largest = max(oracle.ws_bytes_per_matrix(min(s), max(s)) for s in shapes)
    ws = max(int(budget_gb * 2 ** 30), largest)
    _plan_equal(shapes, ws)


def test_workspace_size_rule(built):
    shapes = [(2048, 2048)] * 3 + [(7, 13)]
    per = [oracle.ws_bytes_per_matrix(min(s), max(s)) for s in shapes]
    assert m.muon_workspace_size(shapes, 1 << 40) == sum(per)
    assert m.muon_workspace_size(shapes, 1) == max(per)
    assert m.muon_workspace_size(shapes, max(per) + 10) == max(per) + 10


def test_plan_rejects_small_workspace(built):
    with pytest.raises(m.MuonError) as e:
        m.muon_plan([(2048, 2048)], 4096)
    assert e.value.status == 4


def _hp():
    return m.MuonHparams()._c()


def test_step_argument_validation(built):
    lib = built
    arr = (m.MuonMatrix * 1)()
    arr[0].W = arr[0].G = arr[0].M = 1024
    arr[0].rows, arr[0].cols = 4, 4
    ws = ctypes.c_void_p(4096)
    # count 0 is a no-op, even without a device
    assert lib.muon_step_batched(None, 0, ctypes.byref(_hp()), None, 0, None) == 0
    # null hparams
    assert lib.muon_step_batched(arr, 1, None, ws, 1 << 20, None) == 1
    bad = _hp()
    bad.momentum = 1.5
    assert lib.muon_step_batched(arr, 1, ctypes.byref(bad), ws, 1 << 20, None) == 1
    bad = _hp()
    bad.lr = float("nan")
    assert lib.muon_step_batched(arr, 1, ctypes.byref(bad), ws, 1 << 20, None) == 1
    bad = _hp()
    bad.ns_steps = -1
    assert lib.muon_step_batched(arr, 1, ctypes.byref(bad), ws, 1 << 20, None) == 1
    # bad dims, dtype, alignment, workspace
    arr[0].rows = 0
    assert lib.muon_step_batched(arr, 1, ctypes.byref(_hp()), ws, 1 << 20, None) == 1
    arr[0].rows = 4
    arr[0].g_dtype = 7
    assert lib.muon_step_batched(arr, 1, ctypes.byref(_hp()), ws, 1 << 20, None) == 2
    arr[0].g_dtype = 0
    arr[0].W = 1026
    assert lib.muon_step_batched(arr, 1, ctypes.byref(_hp()), ws, 1 << 20, None) == 3
    arr[0].W = 1024
    arr[0].reserved = 1
    assert lib.muon_step_batched(arr, 1, ctypes.byref(_hp()), ws, 1 << 20, None) == 1
    arr[0].reserved = 0
    assert lib.muon_step_batched(arr, 1, ctypes.byref(_hp()), None, 1 << 20, None) == 1
    assert lib.muon_step_batched(arr, 1, ctypes.byref(_hp()), ctypes.c_void_p(4100), 1 << 20, None) == 3


@pytest.mark.skipif(cuda_available(), reason="checks the no-device path")
def test_step_without_device_reports_no_device(built):
    arr = (m.MuonMatrix * 1)()
    arr[0].W = arr[0].G = arr[0].M = 1024
    arr[0].rows, arr[0].cols = 4, 4
    st = built.muon_step_batched(arr, 1, ctypes.byref(_hp()), ctypes.c_void_p(4096), 1 << 20, None)
    assert st == 7
    h = m.AdamwHparams()._c()
    assert built.adamw_step(ctypes.c_void_p(1024), ctypes.c_void_p(2048), ctypes.c_void_p(4096),
                            ctypes.c_void_p(8192), 4, ctypes.byref(h), 1, None) == 7


def test_adamw_argument_validation(built):
    lib = built
    h = m.AdamwHparams()._c()
    P = ctypes.c_void_p
    assert lib.adamw_step(None, None, None, None, 0, ctypes.byref(h), 1, None) == 0
    assert lib.adamw_step(P(1024), P(2048), P(4096), P(8192), 4, ctypes.byref(h), 0, None) == 1
    assert lib.adamw_step(None, P(2048), P(4096), P(8192), 4, ctypes.byref(h), 1, None) == 1
    assert lib.adamw_step(P(1026), P(2048), P(4096), P(8192), 4, ctypes.byref(h), 1, None) == 3
    # overlapping buffers
    assert lib.adamw_step(P(1024), P(1028), P(4096), P(8192), 4, ctypes.byref(h), 1, None) == 1
    bad = m.AdamwHparams(beta1=1.0)._c()
    assert lib.adamw_step(P(1024), P(2048), P(4096), P(8192), 4, ctypes.byref(bad), 1, None) == 1


def test_newton_schulz_argument_validation(built):
    lib = built
    P = ctypes.c_void_p
    one = (ctypes.c_float * 3)(1.0, 1.0, 1.0)
    c = ctypes.cast(one, P)
    # tall input is rejected, count 0 is a no-op, a small workspace is rejected
    assert lib.muon_newton_schulz(P(1024), P(2048), 1, 8, 4, 5, c, 1, P(4096), 1 << 20, None) == 1
    assert lib.muon_newton_schulz(None, None, 0, 4, 8, 5, c, 1, None, 0, None) == 0
    assert lib.muon_newton_schulz(P(1024), P(2048), 1, 4, 8, 5, c, 1, P(4096), 16, None) == 4
    # the coefficient table has one triple or one per step
    assert lib.muon_newton_schulz(P(1024), P(2048), 1, 4, 8, 5, c, 2, P(4096), 1 << 20, None) == 1
    assert lib.muon_newton_schulz(P(1024), P(2048), 1, 4, 8, 5, None, 1, P(4096), 1 << 20, None) == 1
    bad = (ctypes.c_float * 3)(1.0, float("inf"), 1.0)
    assert lib.muon_newton_schulz(P(1024), P(2048), 1, 4, 8, 1, ctypes.cast(bad, P), 1, P(4096), 1 << 20,
                                  None) == 1


def test_step_new_hparam_validation(built):
    lib = built
    arr = (m.MuonMatrix * 1)()
    arr[0].W = arr[0].G = arr[0].M = 1024
    arr[0].rows, arr[0].cols = 4, 4
    ws = ctypes.c_void_p(4096)
    for field, value in (("scale_mode", 2), ("skip_nonfinite", 3), ("reserved0", 1),
                         ("max_grad_norm", float("nan"))):
        h = _hp()
        setattr(h, field, value)
        assert lib.muon_step_batched(arr, 1, ctypes.byref(h), ws, 1 << 20, None) == 1, field
    bad = m.MuonHparams(ns_steps=2, ns_coeffs=[(1.5, -0.5, 0.0), (1.5, float("nan"), 0.0)])._c()
    assert lib.muon_step_batched(arr, 1, ctypes.byref(bad), ws, 1 << 20, None) == 1
    assert built.muon_status_string(8) == b"step skipped by the non-finite gradient guard"


def test_bounded_wait_check_validation(built):
    P = ctypes.c_void_p
    assert built.muon_check_bounded_wait(None, 1000, None) == 1
    assert built.muon_check_bounded_wait(P(4096), 0, None) == 1
    assert built.muon_check_bounded_wait(P(4096), 10 ** 8, None) == 1
    assert built.muon_check_bounded_wait(P(4100), 1000, None) == 3


def test_stats_argument_validation(built):
    lib = built
    P = ctypes.c_void_p
    arr = (m.MuonMatrix * 1)()
    arr[0].W = arr[0].G = arr[0].M = 1024
    arr[0].rows, arr[0].cols = 4, 4
    # no statistics buffer, a misaligned one; then the step's own checks
    assert lib.muon_step_batched_stats(arr, 1, ctypes.byref(_hp()), P(4096), 1 << 20, None, None) == 1
    assert lib.muon_step_batched_stats(arr, 1, ctypes.byref(_hp()), P(4096), 1 << 20, P(8196), None) == 3
    bad = _hp()
    bad.ns_steps = 101
    assert lib.muon_step_batched_stats(arr, 1, ctypes.byref(bad), P(4096), 1 << 20, P(8192), None) == 1
    arr[0].W = 1026
    assert lib.muon_step_batched_stats(arr, 1, ctypes.byref(_hp()), P(4096), 1 << 20, P(8192), None) == 3
    # no matrices: a no-op
    assert lib.muon_step_batched_stats(None, 0, ctypes.byref(_hp()), None, 0, P(8192), None) == 0


def test_adamw_batched_argument_validation(built):
    lib = built
    P = ctypes.c_void_p
    h = m.AdamwHparams()._c()
    arr = (m.AdamwTensor * 2)()
    for i, base in enumerate((1 << 20, 1 << 24)):
        arr[i].p, arr[i].g, arr[i].m, arr[i].v = base, base + 4096, base + 8192, base + 12288
        arr[i].n = 256
    assert lib.adamw_step_batched(None, 2, ctypes.byref(h), 1, None) == 1        # no table
    assert lib.adamw_step_batched(arr, 2, None, 1, None) == 1                     # no hparams
    assert lib.adamw_step_batched(arr, 2, ctypes.byref(h), 0, None) == 1          # step < 1
    assert lib.adamw_step_batched(arr, -1, ctypes.byref(h), 1, None) == 1
    assert lib.adamw_step_batched(None, 0, ctypes.byref(h), 1, None) == 0         # nothing to do
    arr[1].n = -1
    assert lib.adamw_step_batched(arr, 2, ctypes.byref(h), 1, None) == 1
    arr[1].n = 0                                                                   # empty: skipped
    arr[0].n = 0
    assert lib.adamw_step_batched(arr, 2, ctypes.byref(h), 1, None) == 0
    arr[0].n = arr[1].n = 256
    arr[1].v = (1 << 24) + 12290
    assert lib.adamw_step_batched(arr, 2, ctypes.byref(h), 1, None) == 3          # misaligned
    arr[1].v = (1 << 20) + 8192 + 512                                             # inside tensor 0's m
    assert lib.adamw_step_batched(arr, 2, ctypes.byref(h), 1, None) == 1


def test_graph_argument_validation(built):
    lib = built
    P = ctypes.c_void_p
    arr = (m.MuonMatrix * 1)()
    arr[0].W = arr[0].G = arr[0].M = 1024
    arr[0].rows, arr[0].cols = 4, 4
    out = P(12345)
    # no output handle
    assert lib.muon_step_graph_create(arr, 1, ctypes.byref(_hp()), P(4096), 1 << 20, None) == 1
    # the step's own checks, before anything is captured; the handle is cleared
    bad = _hp()
    bad.momentum = -0.5
    assert lib.muon_step_graph_create(arr, 1, ctypes.byref(bad), P(4096), 1 << 20, ctypes.byref(out)) == 1
    assert out.value is None
    arr[0].g_dtype = 7
    assert lib.muon_step_graph_create(arr, 1, ctypes.byref(_hp()), P(4096), 1 << 20, ctypes.byref(out)) == 2
    arr[0].g_dtype = 0
    assert lib.muon_step_graph_create(arr, 1, ctypes.byref(_hp()), P(4100), 1 << 20, ctypes.byref(out)) == 3
    assert lib.muon_step_graph_create(arr, 1, ctypes.byref(_hp()), None, 1 << 20, ctypes.byref(out)) == 1
    # launch of no graph; destroy of none is a no-op
    assert lib.muon_step_graph_launch(None, None) == 1
    assert lib.muon_step_graph_destroy(None) == 0


def test_graph_of_no_matrices_is_a_no_op(built):
    lib = built
    out = ctypes.c_void_p()
    assert lib.muon_step_graph_create(None, 0, ctypes.byref(_hp()), None, 0, ctypes.byref(out)) == 0
    assert out.value is not None
    assert lib.muon_step_graph_launch(out, None) == 0
    assert lib.muon_step_graph_destroy(out) == 0


@pytest.mark.skipif(cuda_available(), reason="checks the no-device path")
def test_graph_without_device_reports_no_device(built):
    arr = (m.MuonMatrix * 1)()
    arr[0].W = arr[0].G = arr[0].M = 1024
    arr[0].rows, arr[0].cols = 4, 4
    out = ctypes.c_void_p(12345)
    st = built.muon_step_graph_create(arr, 1, ctypes.byref(_hp()), ctypes.c_void_p(4096), 1 << 20,
                                      ctypes.byref(out))
    assert st == 7
    assert out.value is None


def test_library_never_loads_the_oracle(built):
    # the product path has no reference to the oracle
    for path in ("optimizer_muon_step_gb300/__init__.py", "optimizer_muon_step_gb300/build.py",
                 "optimizer_muon_step_gb300/optim.py"):
        src = open(os.path.join(ROOT, path)).read()
        assert "oracle" not in src.replace("no CPU or PyTorch fallback", "")
    for name in os.listdir(os.path.join(ROOT, "optimizer_muon_step_gb300", "csrc")):
        assert "oracle" not in open(os.path.join(ROOT, "optimizer_muon_step_gb300", "csrc", name)).read()


def test_optimizer_class_checks_its_parameters():
    """MuonAdamW takes fp32 CUDA parameters only and refuses an empty list
    (checked on the host, before any library call)."""
    with pytest.raises(TypeError):
        m.MuonAdamW([torch.zeros(4, 4)], [])            # a CPU tensor
    with pytest.raises(ValueError):
        m.MuonAdamW([], [])


def test_optimizer_refuses_parameters_on_several_devices():
    """The library reads every pointer on the current device, so one
    optimizer's parameters must share a device (checked on the host)."""
    from types import SimpleNamespace
    from optimizer_muon_step_gb300.optim import common_device

    on = lambda d: SimpleNamespace(device=torch.device(d))  # noqa: E731
    assert common_device([on("cuda:1"), on("cuda:1")]) == torch.device("cuda:1")
    with pytest.raises(ValueError):
        common_device([on("cuda:0"), on("cuda:1")])
    with pytest.raises(ValueError):
        common_device([])


@pytest.mark.skipif(cuda_available(), reason="checks the no-device path")
def test_fp16_gradient_dtype_rules(built):
    """MUON_F16 gradients need 2-byte alignment only (like bf16): a G at an
    odd 2-byte offset passes the host checks (the call then reports that no
    device is current), an odd address is MUON_ERR_MISALIGNED, and an
    unknown dtype is MUON_ERR_UNSUPPORTED_DTYPE."""
    lib = built
    arr = (m.MuonMatrix * 1)()
    arr[0].W, arr[0].M = 1024, 4096
    arr[0].rows, arr[0].cols = 4, 4
    arr[0].g_dtype = m.MUON_F16
    ws = ctypes.c_void_p(1 << 20)
    arr[0].G = 8194                       # 2-byte aligned only
    assert lib.muon_step_batched(arr, 1, ctypes.byref(_hp()), ws, 1 << 20, None) == 7
    arr[0].G = 8195
    assert lib.muon_step_batched(arr, 1, ctypes.byref(_hp()), ws, 1 << 20, None) == 3
    arr[0].g_dtype = 3
    assert lib.muon_step_batched(arr, 1, ctypes.byref(_hp()), ws, 1 << 20, None) == 2
