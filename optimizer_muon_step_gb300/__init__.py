"""Muon + AdamW optimizer step for GB300 (sm_103a): Python binding.

Thin ctypes marshalling over ``libmuonstep.so`` (C ABI in
``include/muon_step.h``).  Every step of the computation runs in the
library's CUDA kernels; PyTorch only supplies device memory and streams.
There is no CPU or PyTorch fallback: if the library is missing the calls
raise.

Functions keep the C names:
    muon_step_batched(W, G, M, hp, workspace=None, stream=None)
    muon_newton_schulz(X, steps, coeffs, out=None, workspace=None, stream=None)
    adamw_step(p, g, m, v, hp, step, stream=None)
    adamw_step_batched([(p, g, m, v), ...], hp, step, stream=None)
    muon_plan(shapes, ws_bytes)
    muon_workspace_bytes_per_matrix(rows, cols)
    muon_workspace_size(shapes, budget_bytes)
    muon_query_status(workspace, stream=None)
    MuonAdamW(muon_params, adamw_params, muon_hp, adamw_hp): a torch.optim.Optimizer
    muon_step_graph_create / _launch / _destroy (through MuonBatch.capture)
"""
from __future__ import annotations

import ctypes
import os
import threading
from dataclasses import dataclass
from typing import Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmuonstep.so")
_lock = threading.Lock()
_lib = None

MUON_F32, MUON_BF16, MUON_F16 = 0, 1, 2
STATUS = {0: "MUON_OK", 1: "MUON_ERR_INVALID_ARG", 2: "MUON_ERR_UNSUPPORTED_DTYPE",
          3: "MUON_ERR_MISALIGNED", 4: "MUON_ERR_WORKSPACE_TOO_SMALL", 5: "MUON_ERR_CUDA",
          6: "MUON_ERR_TIMEOUT", 7: "MUON_ERR_NO_DEVICE", 8: "MUON_STEP_SKIPPED"}
MUON_STEP_SKIPPED = 8

# Every symbol include/muon_step.h declares.
EXPORTS = ("muon_workspace_bytes_per_matrix", "muon_workspace_size", "muon_plan",
           "muon_step_batched", "muon_newton_schulz", "adamw_step", "muon_query_status",
           "muon_status_string", "muon_version", "muon_launch_count", "muon_set_timing",
           "muon_timing_read", "muon_kernel_name", "muon_step_batched_noalloc",
           "muon_check_bounded_wait", "muon_step_graph_create", "muon_step_graph_launch",
           "muon_step_graph_destroy", "muon_step_batched_stats", "adamw_step_batched")
KERNEL_KINDS = ("momentum_norm", "norm_finalize", "x0_rescale", "ns_syrk", "ns_poly",
                "ns_update", "final_update", "adamw", "grad_guard", "desc_upload", "stats")


class MuonError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {STATUS.get(status, status)} ({status})")


class MuonMatrix(ctypes.Structure):
    _fields_ = [("W", ctypes.c_void_p), ("G", ctypes.c_void_p), ("M", ctypes.c_void_p),
                ("rows", ctypes.c_int64), ("cols", ctypes.c_int64),
                ("g_dtype", ctypes.c_int32), ("reserved", ctypes.c_int32)]


class _MuonHparamsC(ctypes.Structure):
    _fields_ = [("lr", ctypes.c_float), ("weight_decay", ctypes.c_float),
                ("momentum", ctypes.c_float), ("nesterov", ctypes.c_int32),
                ("ns_steps", ctypes.c_int32), ("ns_a", ctypes.c_float),
                ("ns_b", ctypes.c_float), ("ns_c", ctypes.c_float),
                ("norm_eps", ctypes.c_float), ("rms_scale", ctypes.c_float),
                ("scale_mode", ctypes.c_int32), ("skip_nonfinite", ctypes.c_int32),
                ("max_grad_norm", ctypes.c_float), ("reserved0", ctypes.c_int32),
                ("ns_coeffs", ctypes.c_void_p)]


class _AdamwHparamsC(ctypes.Structure):
    _fields_ = [("lr", ctypes.c_float), ("beta1", ctypes.c_float), ("beta2", ctypes.c_float),
                ("eps", ctypes.c_float), ("weight_decay", ctypes.c_float)]


class PlanEntry(ctypes.Structure):
    _fields_ = [("mat_idx", ctypes.c_int32), ("transposed", ctypes.c_int32),
                ("group_id", ctypes.c_int32), ("slot", ctypes.c_int32),
                ("chunk_id", ctypes.c_int32), ("reserved", ctypes.c_int32),
                ("mp", ctypes.c_int64), ("np", ctypes.c_int64)]


PLAN_DTYPE = np.dtype([("mat_idx", np.int32), ("transposed", np.int32), ("group_id", np.int32),
                       ("slot", np.int32), ("chunk_id", np.int32), ("reserved", np.int32),
                       ("mp", np.int64), ("np", np.int64)])


@dataclass
class MuonHparams:
    lr: float = 0.02
    weight_decay: float = 0.1
    momentum: float = 0.95
    nesterov: bool = True
    ns_steps: int = 5
    ns_a: float = 3.4445
    ns_b: float = -4.7750
    ns_c: float = 2.0315
    norm_eps: float = 1e-7
    rms_scale: float = 0.2
    scale_mode: int = 0            # 0: rms_scale*sqrt(max(m,n)); 1: max(1, sqrt(rows/cols))
    skip_nonfinite: bool = False   # skip the whole call when any gradient is non-finite
    max_grad_norm: float = 0.0     # > 0: clip all gradients of the call by their global norm
    ns_coeffs: object = None       # None, or ns_steps (a, b, c) triples

    def _c(self):
        h = _MuonHparamsC(self.lr, self.weight_decay, self.momentum, int(bool(self.nesterov)),
                          int(self.ns_steps), self.ns_a, self.ns_b, self.ns_c, self.norm_eps,
                          self.rms_scale, int(self.scale_mode), int(bool(self.skip_nonfinite)),
                          self.max_grad_norm, 0, None)
        if self.ns_coeffs is not None:
            table = _coeff_array(self.ns_coeffs, self.ns_steps)
            h.ns_coeffs = ctypes.cast(table, ctypes.c_void_p)
            h._keep = table  # alive as long as the struct
        return h


def _coeff_array(coeffs, steps):
    """(ctypes float array, count of triples) from one triple or a list of them."""
    flat = [float(x) for x in np.asarray(coeffs, dtype=np.float64).reshape(-1)]
    if len(flat) % 3:
        raise ValueError("NS coefficients come in (a, b, c) triples")
    if len(flat) // 3 not in (1, max(int(steps), 1)) and steps:
        raise ValueError("give one (a, b, c) triple or one per NS step")
    return (ctypes.c_float * len(flat))(*flat)


@dataclass
class AdamwHparams:
    lr: float = 3e-4
    beta1: float = 0.9
    beta2: float = 0.95
    eps: float = 1e-8
    weight_decay: float = 0.1

    def _c(self):
        return _AdamwHparamsC(self.lr, self.beta1, self.beta2, self.eps, self.weight_decay)


def load_library(path: str = LIB_PATH):
    """Loads libmuonstep.so; raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is missing: build it with "
                               "`python -m optimizer_muon_step_gb300.build` (needs nvcc)")
        lib = ctypes.CDLL(path)
        P, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32
        lib.muon_workspace_bytes_per_matrix.argtypes = [i64, i64]
        lib.muon_workspace_bytes_per_matrix.restype = ctypes.c_size_t
        lib.muon_workspace_size.argtypes = [P, i64, ctypes.c_size_t, ctypes.POINTER(ctypes.c_size_t)]
        lib.muon_workspace_size.restype = ctypes.c_int
        lib.muon_plan.argtypes = [P, i64, ctypes.c_size_t, P]
        lib.muon_plan.restype = ctypes.c_int
        lib.muon_step_batched.argtypes = [P, i64, P, P, ctypes.c_size_t, P]
        lib.muon_step_batched.restype = ctypes.c_int
        lib.muon_step_batched_stats.argtypes = [P, i64, P, P, ctypes.c_size_t, P, P]
        lib.muon_step_batched_stats.restype = ctypes.c_int
        lib.muon_step_batched_noalloc.argtypes = [P, i64, P, P]
        lib.muon_step_batched_noalloc.restype = ctypes.c_int
        lib.muon_newton_schulz.argtypes = [P, P, i64, i64, i64, i32, P, i32, P, ctypes.c_size_t, P]
        lib.muon_newton_schulz.restype = ctypes.c_int
        lib.adamw_step.argtypes = [P, P, P, P, i64, P, i64, P]
        lib.adamw_step_batched.argtypes = [P, i64, P, i64, P]
        lib.adamw_step_batched.restype = ctypes.c_int
        lib.adamw_step.restype = ctypes.c_int
        lib.muon_query_status.argtypes = [P, P]
        lib.muon_query_status.restype = ctypes.c_int
        lib.muon_check_bounded_wait.argtypes = [P, i64, P]
        lib.muon_check_bounded_wait.restype = ctypes.c_int
        lib.muon_status_string.argtypes = [ctypes.c_int]
        lib.muon_status_string.restype = ctypes.c_char_p
        lib.muon_version.argtypes = []
        lib.muon_version.restype = i32
        lib.muon_launch_count.argtypes = []
        lib.muon_launch_count.restype = i64
        lib.muon_set_timing.argtypes = [i32]
        lib.muon_set_timing.restype = ctypes.c_int
        lib.muon_timing_read.argtypes = [P, P, i32]
        lib.muon_timing_read.restype = ctypes.c_int
        lib.muon_kernel_name.argtypes = [i32]
        lib.muon_kernel_name.restype = ctypes.c_char_p
        lib.muon_step_graph_create.argtypes = [P, i64, P, P, ctypes.c_size_t, ctypes.POINTER(P)]
        lib.muon_step_graph_create.restype = ctypes.c_int
        lib.muon_step_graph_launch.argtypes = [P, P]
        lib.muon_step_graph_launch.restype = ctypes.c_int
        lib.muon_step_graph_destroy.argtypes = [P]
        lib.muon_step_graph_destroy.restype = ctypes.c_int
        _lib = lib
        return lib


def _check(status: int, where: str):
    if status != 0:
        raise MuonError(status, where)


def _stream(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _matrices(shapes_or_tensors):
    arr = (MuonMatrix * max(1, len(shapes_or_tensors)))()
    for i, s in enumerate(shapes_or_tensors):
        arr[i].rows, arr[i].cols = int(s[0]), int(s[1])
    return arr


# --------------------------------------------------------------------------
# Host-only calls
# --------------------------------------------------------------------------

def muon_workspace_bytes_per_matrix(rows: int, cols: int) -> int:
    return int(load_library().muon_workspace_bytes_per_matrix(int(rows), int(cols)))


def muon_workspace_size(shapes: Sequence, budget_bytes: int) -> int:
    shapes = list(shapes)
    out = ctypes.c_size_t(0)
    _check(load_library().muon_workspace_size(ctypes.cast(_matrices(shapes), ctypes.c_void_p),
                                              len(shapes), int(budget_bytes), ctypes.byref(out)),
           "muon_workspace_size")
    return int(out.value)


def muon_plan(shapes: Sequence, ws_bytes: int) -> np.ndarray:
    """Execution plan for a list of (rows, cols) as a structured array."""
    shapes = list(shapes)
    out = (PlanEntry * max(1, len(shapes)))()
    _check(load_library().muon_plan(ctypes.cast(_matrices(shapes), ctypes.c_void_p), len(shapes),
                                    int(ws_bytes), ctypes.cast(out, ctypes.c_void_p)), "muon_plan")
    return np.frombuffer(bytes(out), dtype=PLAN_DTYPE, count=max(1, len(shapes))).copy()[:len(shapes)]


# --------------------------------------------------------------------------
# Device calls
# --------------------------------------------------------------------------

def _dev_tensor(t, name, dtypes):
    import torch
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if t.dtype not in dtypes:
        raise TypeError(f"{name} has dtype {t.dtype}, expected one of {dtypes}")
    return t


def allocate_workspace(nbytes: int, device=None):
    """Device workspace (torch allocation, 256-byte aligned)."""
    import torch
    return torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device=device or "cuda")


def _g_dtype(g) -> int:
    import torch
    return {torch.float32: MUON_F32, torch.bfloat16: MUON_BF16, torch.float16: MUON_F16}[g.dtype]


def _stats_tensor(stats, n):
    import torch
    if not (isinstance(stats, torch.Tensor) and stats.is_cuda and stats.dtype == torch.float64
            and stats.is_contiguous() and tuple(stats.shape) == (n, 2)):
        raise ValueError(f"stats must be a contiguous CUDA float64 tensor of shape ({n}, 2)")
    return ctypes.c_void_p(stats.data_ptr())


def muon_step_batched(W, G, M, hp: MuonHparams = MuonHparams(), workspace=None, stream=None,
                      budget_bytes: int = 16 << 30, stats=None):
    """One Muon step on lists of matrices (in place on every W and M).

    W, M: fp32 CUDA tensors (rows x cols); G: fp32, bf16 or fp16 of the same shape.
    workspace: a uint8 CUDA tensor; allocated here (torch) when None.
    stats: optional CUDA float64 tensor (len(W), 2) that receives each
    matrix's (||u||_F, update RMS) (muon_step_batched_stats).
    Returns the workspace so callers can reuse it."""
    import torch
    n = len(W)
    if not (len(G) == n and len(M) == n):
        raise ValueError("W, G, M must have the same length")
    arr = (MuonMatrix * max(1, n))()
    for i in range(n):
        w = _dev_tensor(W[i], f"W[{i}]", (torch.float32,))
        g = _dev_tensor(G[i], f"G[{i}]", (torch.float32, torch.bfloat16, torch.float16))
        m = _dev_tensor(M[i], f"M[{i}]", (torch.float32,))
        if w.dim() != 2 or w.shape != g.shape or w.shape != m.shape:
            raise ValueError(f"matrix {i}: W, G, M must be equal-shaped 2-D tensors")
        arr[i].W, arr[i].G, arr[i].M = w.data_ptr(), g.data_ptr(), m.data_ptr()
        arr[i].rows, arr[i].cols = w.shape
        arr[i].g_dtype = _g_dtype(g)
    lib = load_library()
    if workspace is None:
        need = ctypes.c_size_t(0)
        _check(lib.muon_workspace_size(ctypes.cast(arr, ctypes.c_void_p), n, int(budget_bytes),
                                       ctypes.byref(need)), "muon_workspace_size")
        workspace = allocate_workspace(need.value, W[0].device if n else None)
    h = hp._c()
    if stats is None:
        _check(lib.muon_step_batched(ctypes.cast(arr, ctypes.c_void_p), n, ctypes.byref(h),
                                     ctypes.c_void_p(workspace.data_ptr()), workspace.numel(),
                                     _stream(stream)), "muon_step_batched")
    else:
        _check(lib.muon_step_batched_stats(ctypes.cast(arr, ctypes.c_void_p), n, ctypes.byref(h),
                                           ctypes.c_void_p(workspace.data_ptr()), workspace.numel(),
                                           _stats_tensor(stats, n), _stream(stream)),
               "muon_step_batched_stats")
    return workspace


def muon_step_batched_noalloc(W, G, M, hp: MuonHparams = MuonHparams(), stream=None):
    """The Muon step with the library's static device scratch as workspace:
    no device memory is allocated by this call or by the library.  For
    callers that cannot allocate; every matrix must fit the 64 MiB scratch
    on its own, and calls that overlap on the GPU race on that scratch."""
    import torch
    n = len(W)
    if not (len(G) == n and len(M) == n):
        raise ValueError("W, G, M must have the same length")
    arr = (MuonMatrix * max(1, n))()
    for i in range(n):
        w = _dev_tensor(W[i], f"W[{i}]", (torch.float32,))
        g = _dev_tensor(G[i], f"G[{i}]", (torch.float32, torch.bfloat16, torch.float16))
        m = _dev_tensor(M[i], f"M[{i}]", (torch.float32,))
        if w.dim() != 2 or w.shape != g.shape or w.shape != m.shape:
            raise ValueError(f"matrix {i}: W, G, M must be equal-shaped 2-D tensors")
        arr[i].W, arr[i].G, arr[i].M = w.data_ptr(), g.data_ptr(), m.data_ptr()
        arr[i].rows, arr[i].cols = w.shape
        arr[i].g_dtype = _g_dtype(g)
    h = hp._c()
    _check(load_library().muon_step_batched_noalloc(ctypes.cast(arr, ctypes.c_void_p), n,
                                                    ctypes.byref(h), _stream(stream)),
           "muon_step_batched_noalloc")


def muon_newton_schulz(X, steps: int = 5, coeffs=(3.4445, -4.7750, 2.0315), out=None,
                       workspace=None, stream=None):
    """Newton-Schulz on a bf16 CUDA tensor [count, m', n'] (or [m', n']).

    coeffs: one (a, b, c) triple for every step, or `steps` triples."""
    import torch
    _dev_tensor(X, "X", (torch.bfloat16,))
    squeeze = X.dim() == 2
    X3 = X.unsqueeze(0) if squeeze else X
    if X3.dim() != 3 or X3.shape[1] > X3.shape[2]:
        raise ValueError("X must be [count, m', n'] with m' <= n'")
    count, mp, np_ = X3.shape
    if out is None:
        out = torch.empty_like(X3)
    out3 = out.view(count, mp, np_)
    _dev_tensor(out3, "out", (torch.bfloat16,))
    lib = load_library()
    if workspace is None:
        workspace = allocate_workspace(count * muon_workspace_bytes_per_matrix(mp, np_), X.device)
    table = _coeff_array(coeffs, steps)
    _check(lib.muon_newton_schulz(ctypes.c_void_p(X3.data_ptr()), ctypes.c_void_p(out3.data_ptr()),
                                  count, mp, np_, int(steps), ctypes.cast(table, ctypes.c_void_p),
                                  len(table) // 3, ctypes.c_void_p(workspace.data_ptr()),
                                  workspace.numel(), _stream(stream)), "muon_newton_schulz")
    return out3[0] if squeeze else out3


def adamw_step(p, g, m, v, hp: AdamwHparams = AdamwHparams(), step: int = 1, stream=None):
    """AdamW in place on flat fp32 CUDA tensors p, m, v with gradient g."""
    import torch
    for name, t in (("p", p), ("g", g), ("m", m), ("v", v)):
        _dev_tensor(t, name, (torch.float32,))
    n = p.numel()
    if not (g.numel() == m.numel() == v.numel() == n):
        raise ValueError("p, g, m, v must have the same number of elements")
    h = hp._c()
    _check(load_library().adamw_step(ctypes.c_void_p(p.data_ptr()), ctypes.c_void_p(g.data_ptr()),
                                     ctypes.c_void_p(m.data_ptr()), ctypes.c_void_p(v.data_ptr()),
                                     n, ctypes.byref(h), int(step), _stream(stream)), "adamw_step")


class AdamwTensor(ctypes.Structure):
    _fields_ = [("p", ctypes.c_void_p), ("g", ctypes.c_void_p), ("m", ctypes.c_void_p),
                ("v", ctypes.c_void_p), ("n", ctypes.c_int64)]


def adamw_step_batched(tensors, hp: AdamwHparams = AdamwHparams(), step: int = 1, stream=None):
    """AdamW in place on many tensors in few launches: `tensors` is a list of
    (p, g, m, v) contiguous fp32 CUDA tensors, the four of a tuple with equal
    element counts (any shapes)."""
    import torch
    arr = (AdamwTensor * max(1, len(tensors)))()
    for i, quad in enumerate(tensors):
        p, g, m, v = quad
        for name, x in (("p", p), ("g", g), ("m", m), ("v", v)):
            _dev_tensor(x, f"{name}[{i}]", (torch.float32,))
        n = p.numel()
        if not (g.numel() == m.numel() == v.numel() == n):
            raise ValueError(f"tensor {i}: p, g, m, v must have the same number of elements")
        arr[i].p, arr[i].g, arr[i].m, arr[i].v = p.data_ptr(), g.data_ptr(), m.data_ptr(), v.data_ptr()
        arr[i].n = n
    h = hp._c()
    _check(load_library().adamw_step_batched(ctypes.cast(arr, ctypes.c_void_p), len(tensors), ctypes.byref(h),
                                             int(step), _stream(stream)), "adamw_step_batched")


def muon_query_status(workspace, stream=None) -> int:
    """Synchronises the stream and returns (and clears) the device status:
    0, MUON_ERR_TIMEOUT (6) or MUON_STEP_SKIPPED (8)."""
    return int(load_library().muon_query_status(ctypes.c_void_p(workspace.data_ptr()), _stream(stream)))


def muon_check_bounded_wait(workspace, limit_us: int = 20000, stream=None) -> None:
    """Enqueues the failure-detection self-check: a bounded wait that nothing
    satisfies runs out after limit_us and records MUON_ERR_TIMEOUT (6) in the
    workspace status; read it with muon_query_status."""
    _check(load_library().muon_check_bounded_wait(ctypes.c_void_p(workspace.data_ptr()), int(limit_us),
                                                  _stream(stream)), "muon_check_bounded_wait")


def version() -> int:
    return int(load_library().muon_version())


# --------------------------------------------------------------------------
# Instrumentation
# --------------------------------------------------------------------------

def muon_launch_count() -> int:
    """Kernels this library has launched in this process."""
    return int(load_library().muon_launch_count())


def muon_set_timing(enable: bool) -> None:
    _check(load_library().muon_set_timing(1 if enable else 0), "muon_set_timing")


def muon_timing_read() -> dict:
    """{kernel name: (total ms, launches)} since timing was enabled."""
    n = len(KERNEL_KINDS)
    ms = (ctypes.c_double * n)()
    cnt = (ctypes.c_int64 * n)()
    _check(load_library().muon_timing_read(ms, cnt, n), "muon_timing_read")
    return {KERNEL_KINDS[i]: (float(ms[i]), int(cnt[i])) for i in range(n)}


class MuonBatch:
    """A fixed list of (W, G, M) matrices marshalled once for repeated steps.

    The tensors must stay alive and keep their storage while the batch is
    used; ``step`` then only passes the prepared array to the library."""

    def __init__(self, W, G, M, budget_bytes: int = 16 << 30, workspace=None):
        import torch
        n = len(W)
        if not (len(G) == n and len(M) == n):
            raise ValueError("W, G, M must have the same length")
        self._keep = (list(W), list(G), list(M))
        self.count = n
        self.arr = (MuonMatrix * max(1, n))()
        for i in range(n):
            w = _dev_tensor(W[i], f"W[{i}]", (torch.float32,))
            g = _dev_tensor(G[i], f"G[{i}]", (torch.float32, torch.bfloat16, torch.float16))
            m = _dev_tensor(M[i], f"M[{i}]", (torch.float32,))
            if w.dim() != 2 or w.shape != g.shape or w.shape != m.shape:
                raise ValueError(f"matrix {i}: W, G, M must be equal-shaped 2-D tensors")
            self.arr[i].W, self.arr[i].G, self.arr[i].M = w.data_ptr(), g.data_ptr(), m.data_ptr()
            self.arr[i].rows, self.arr[i].cols = w.shape
            self.arr[i].g_dtype = _g_dtype(g)
        lib = load_library()
        if workspace is None:
            need = ctypes.c_size_t(0)
            _check(lib.muon_workspace_size(ctypes.cast(self.arr, ctypes.c_void_p), n, int(budget_bytes),
                                           ctypes.byref(need)), "muon_workspace_size")
            workspace = allocate_workspace(need.value, W[0].device if n else None)
        self.workspace = workspace

    def step(self, hp: MuonHparams = MuonHparams(), stream=None):
        h = hp._c()
        _check(load_library().muon_step_batched(ctypes.cast(self.arr, ctypes.c_void_p), self.count,
                                                ctypes.byref(h),
                                                ctypes.c_void_p(self.workspace.data_ptr()),
                                                self.workspace.numel(), _stream(stream)),
               "muon_step_batched")

    def step_with_stats(self, hp: MuonHparams = MuonHparams(), stream=None, out=None):
        """The step plus each matrix's (||u||_F, update RMS): returns a CUDA
        float64 tensor (count, 2), `out` when given (muon_step_batched_stats)."""
        import torch
        if out is None:
            out = torch.empty((self.count, 2), dtype=torch.float64, device=self.workspace.device)
        h = hp._c()
        _check(load_library().muon_step_batched_stats(ctypes.cast(self.arr, ctypes.c_void_p), self.count,
                                                      ctypes.byref(h),
                                                      ctypes.c_void_p(self.workspace.data_ptr()),
                                                      self.workspace.numel(), _stats_tensor(out, self.count),
                                                      _stream(stream)),
               "muon_step_batched_stats")
        return out

    def capture(self, hp: MuonHparams = MuonHparams()) -> "MuonGraph":
        """The step with these hyper-parameters captured once as a CUDA
        graph (muon_step_graph_create); replay it with ``MuonGraph.launch``."""
        return MuonGraph(self, hp)


class MuonGraph:
    """A captured Muon step over a MuonBatch's matrices and workspace.

    Every replay runs the same kernels as ``MuonBatch.step(hp)`` with the
    hyper-parameters fixed at capture, reading the current gradients."""

    def __init__(self, batch: MuonBatch, hp: MuonHparams):
        self._batch = batch  # keeps the tensors and the workspace alive
        self._lib = load_library()
        h = hp._c()
        handle = ctypes.c_void_p()
        _check(self._lib.muon_step_graph_create(ctypes.cast(batch.arr, ctypes.c_void_p), batch.count,
                                                ctypes.byref(h),
                                                ctypes.c_void_p(batch.workspace.data_ptr()),
                                                batch.workspace.numel(), ctypes.byref(handle)),
               "muon_step_graph_create")
        self._handle = handle

    def launch(self, stream=None):
        if self._handle is None:
            raise RuntimeError("the graph has been destroyed")
        _check(self._lib.muon_step_graph_launch(self._handle, _stream(stream)), "muon_step_graph_launch")

    def destroy(self):
        if getattr(self, "_handle", None) is not None:
            _check(self._lib.muon_step_graph_destroy(self._handle), "muon_step_graph_destroy")
            self._handle = None

    def __del__(self):
        try:
            self.destroy()
        except Exception:
            pass


def __getattr__(name):
    # the torch.optim.Optimizer over this library (imports torch)
    if name == "MuonAdamW":
        from .optim import MuonAdamW
        return MuonAdamW
    raise AttributeError(f"module {__name__!r} has no attribute {name!r}")
