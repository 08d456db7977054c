"""Oracle: a plain CPU restatement of the Muon step and AdamW.

TEST INFRASTRUCTURE ONLY.  Only the test suite, ``__graft_entry__.smoke()``
and the CPU-baseline leg of ``bench.py`` may import this package.  The GPU
library never imports it, links it or runs it, and nothing here reads any
value the GPU library produced.

The arithmetic lives in ``muon_oracle.c`` (plain loops, fp64 accumulation,
explicit bf16 round-to-nearest-even).  This module compiles it with gcc on
first use and wraps it with ctypes over numpy arrays.

Sources are cited by page title and section:
  [OPT] "LLM training series, part 2: optimizers" (mhpq.cn article)
  [K2]  "Kimi K2 ... what is worth noting" (Zhihu answer by toothacher17)
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "muon_oracle.c")
# MUON_ORACLE_LIB names a prebuilt variant of the library to load instead
# (the test that plants mistakes in copies of muon_oracle.c uses it); it is
# loaded as given and never rebuilt.
_PREBUILT = os.environ.get("MUON_ORACLE_LIB")
_LIB_PATH = _PREBUILT or os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

CFLAGS = ["-O3", "-std=c11", "-fPIC", "-shared", "-fopenmp",
          "-ffp-contract=off", "-fno-fast-math"]


def build(force: bool = False) -> str:
    """Compile muon_oracle.c into liboracle.so (gcc, no GPU involved)."""
    if _PREBUILT:
        return _LIB_PATH
    stale = (not os.path.exists(_LIB_PATH)
             or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
    if force or stale:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.run(["gcc", *CFLAGS, "-o", tmp, _SRC, "-lm"], check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class MuonHparams(ctypes.Structure):
    _fields_ = [("lr", ctypes.c_float), ("weight_decay", ctypes.c_float),
                ("momentum", ctypes.c_float), ("nesterov", ctypes.c_int),
                ("ns_steps", ctypes.c_int), ("ns_a", ctypes.c_float),
                ("ns_b", ctypes.c_float), ("ns_c", ctypes.c_float),
                ("norm_eps", ctypes.c_float), ("rms_scale", ctypes.c_float),
                ("scale_mode", ctypes.c_int), ("skip_nonfinite", ctypes.c_int),
                ("max_grad_norm", ctypes.c_float), ("reserved", ctypes.c_int),
                ("ns_coeffs", ctypes.c_void_p)]


class AdamwHparams(ctypes.Structure):
    _fields_ = [("lr", ctypes.c_float), ("beta1", ctypes.c_float),
                ("beta2", ctypes.c_float), ("eps", ctypes.c_float),
                ("weight_decay", ctypes.c_float)]


class PlanEntry(ctypes.Structure):
    _fields_ = [("mat_idx", ctypes.c_int32), ("transposed", ctypes.c_int32),
                ("group_id", ctypes.c_int32), ("slot", ctypes.c_int32),
                ("chunk_id", ctypes.c_int32), ("pad_", ctypes.c_int32),
                ("mp", ctypes.c_int64), ("np", ctypes.c_int64)]


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            i64 = ctypes.c_int64
            lib.oracle_bf16_from_f32.argtypes = [ctypes.c_float]
            lib.oracle_bf16_from_f32.restype = ctypes.c_uint16
            lib.oracle_bf16_encode.argtypes = [P, P, i64]
            lib.oracle_bf16_encode.restype = None
            lib.oracle_newton_schulz.argtypes = [P, i64, i64, ctypes.c_int,
                                                 ctypes.c_float, ctypes.c_float,
                                                 ctypes.c_float, ctypes.c_int]
            lib.oracle_newton_schulz.restype = ctypes.c_int
            lib.oracle_momentum.argtypes = [P, P, P, i64, ctypes.c_float, ctypes.c_int]
            lib.oracle_momentum.restype = None
            lib.oracle_normalize.argtypes = [P, i64, i64, ctypes.c_float, P]
            lib.oracle_normalize.restype = ctypes.c_float
            lib.oracle_final_update.argtypes = [P, P, i64, i64, ctypes.c_float, ctypes.c_float,
                                                ctypes.c_float, ctypes.c_int]
            lib.oracle_final_update.restype = None
            lib.oracle_step_stats.argtypes = [P, P, i64, i64, ctypes.c_float, ctypes.c_int, P, P]
            lib.oracle_step_stats.restype = None
            lib.oracle_muon_step_matrix.argtypes = [P, P, P, i64, i64, P, P, P]
            lib.oracle_muon_step_matrix.restype = ctypes.c_int
            lib.oracle_muon_step_matrix_scaled.argtypes = [P, P, P, i64, i64, P, ctypes.c_float,
                                                           ctypes.c_int, P, P]
            lib.oracle_muon_step_matrix_scaled.restype = ctypes.c_int
            lib.oracle_newton_schulz_table.argtypes = [P, i64, i64, ctypes.c_int, P, ctypes.c_int]
            lib.oracle_newton_schulz_table.restype = ctypes.c_int
            lib.oracle_newton_schulz_scaled.argtypes = [P, i64, i64, ctypes.c_int, P, ctypes.c_int, ctypes.c_float]
            lib.oracle_newton_schulz_scaled.restype = ctypes.c_int
            lib.oracle_newton_schulz_ex.argtypes = [P, i64, i64, ctypes.c_int, P, ctypes.c_int, ctypes.c_float,
                                                    ctypes.c_int]
            lib.oracle_newton_schulz_ex.restype = ctypes.c_int
            lib.oracle_matmul.argtypes = [P, P, P, i64, i64, i64, ctypes.c_int]
            lib.oracle_matmul.restype = None
            lib.oracle_normalize_cast_after.argtypes = [P, i64, i64, ctypes.c_float, P]
            lib.oracle_normalize_cast_after.restype = ctypes.c_float
            lib.oracle_muon_step_matrix_ex.argtypes = [P, P, P, i64, i64, P, ctypes.c_float, ctypes.c_int,
                                                       ctypes.c_int, ctypes.c_int, P, P]
            lib.oracle_muon_step_matrix_ex.restype = ctypes.c_int
            lib.oracle_update_scale.argtypes = [i64, i64, ctypes.c_float, ctypes.c_int]
            lib.oracle_update_scale.restype = ctypes.c_float
            lib.oracle_adamw_step.argtypes = [P, P, P, P, i64, P, i64]
            lib.oracle_adamw_step.restype = ctypes.c_int
            lib.oracle_ws_bytes_per_matrix.argtypes = [i64, i64]
            lib.oracle_ws_bytes_per_matrix.restype = i64
            lib.oracle_plan.argtypes = [P, P, i64, i64, P]
            lib.oracle_plan.restype = ctypes.c_int
            lib.oracle_grad_stats.argtypes = [P, P, i64, P, P]
            lib.oracle_grad_stats.restype = None
            lib.oracle_clip_factor.argtypes = [ctypes.c_double, ctypes.c_float]
            lib.oracle_clip_factor.restype = ctypes.c_float
            lib.oracle_num_threads.argtypes = []
            lib.oracle_num_threads.restype = ctypes.c_int
            _lib = lib
    return _lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def num_threads() -> int:
    """OpenMP threads the oracle's parallel loops use."""
    return int(_load().oracle_num_threads())


# --------------------------------------------------------------------------
# bf16
# --------------------------------------------------------------------------

def bf16_bits(x) -> np.ndarray:
    """fp32 -> bf16 bit patterns, round-to-nearest-even (uint16 array)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, dtype=np.uint16)
    _load().oracle_bf16_encode(_ptr(x), _ptr(out), x.size)
    return out


def bf16_values(bits) -> np.ndarray:
    """bf16 bit patterns -> the fp32 values they encode (exact widening)."""
    bits = np.ascontiguousarray(bits, dtype=np.uint16)
    return (bits.astype(np.uint32) << 16).view(np.float32)


def bf16_round(x) -> np.ndarray:
    return bf16_values(bf16_bits(x))


# --------------------------------------------------------------------------
# Newton-Schulz
# --------------------------------------------------------------------------

# How the NS products accumulate (the spread variants; ACC_FP64 is the
# reference evaluation): fp64; fp32 with one rounding per addition; fp32 with
# blocks of 16 products each added with one round-toward-zero.
ACC_FP64, ACC_FP32, ACC_FP32_RZ16 = 0, 1, 2

QUINTIC = (3.4445, -4.7750, 2.0315)
CUBIC = (1.5, -0.5, 0.0)  # [OPT] section 4.2: X <- (3X - X X^T X) / 2


def matmul(A, B, accum=ACC_FP64) -> np.ndarray:
    """A @ B with every element summed in ascending k: in fp64 (ACC_FP64), in
    fp32 with each product and each partial sum rounded to nearest
    (ACC_FP32), or in fp32 with each block of 16 products summed in fp64 and
    added with one rounding toward zero (ACC_FP32_RZ16)."""
    A = np.ascontiguousarray(A, dtype=np.float64)
    B = np.ascontiguousarray(B, dtype=np.float64)
    if A.ndim != 2 or B.ndim != 2 or A.shape[1] != B.shape[0]:
        raise ValueError("matmul expects M x K and K x N arrays")
    C = np.empty((A.shape[0], B.shape[1]), dtype=np.float64)
    _load().oracle_matmul(_ptr(A), _ptr(B), _ptr(C), A.shape[0], A.shape[1], B.shape[1], _accum(accum))
    return C


def _accum(accum) -> int:
    if accum not in (ACC_FP64, ACC_FP32, ACC_FP32_RZ16):
        raise ValueError("accum must be ACC_FP64, ACC_FP32 or ACC_FP32_RZ16")
    return int(accum)


def newton_schulz(X, steps=5, coeffs=QUINTIC, emulate_bf16=True, x_scale=1.0, accum=ACC_FP64) -> np.ndarray:
    """Run the NS iteration on the wide matrix x_scale * X (rows <= cols).

    coeffs: one (a, b, c) for every step, or a sequence of `steps` triples.
    emulate_bf16=True: X must hold bf16 values; A, B and each new X are
    rounded to bf16 at the GPU's storage points, and x_scale is applied in
    fp32 inside the first step.  emulate_bf16=False: pure fp64, for the
    closed-form checks.  accum (with emulate_bf16): how the products
    accumulate (see matmul); the fp32 modes are equally faithful
    evaluations, used to measure how far such evaluations lie apart."""
    X = np.array(X, dtype=np.float64, order="C", copy=True)
    if X.ndim != 2 or X.shape[0] > X.shape[1]:
        raise ValueError("newton_schulz expects a wide 2-D matrix")
    if _accum(accum) != ACC_FP64 and not emulate_bf16:
        raise ValueError("fp32 accumulation applies to the bf16-emulating iteration only")
    table = coeff_table(coeffs, steps)
    rc = _load().oracle_newton_schulz_ex(_ptr(X), X.shape[0], X.shape[1], int(steps),
                                         _ptr(table), 1 if emulate_bf16 else 0, float(x_scale),
                                         _accum(accum))
    if rc:
        raise RuntimeError(f"oracle_newton_schulz failed ({rc})")
    return X


def coeff_table(coeffs, steps) -> np.ndarray:
    """fp32 table of `steps` (a, b, c) triples from one triple or a list."""
    arr = np.asarray(coeffs, dtype=np.float64)
    if arr.ndim == 1:
        arr = np.tile(arr, (max(int(steps), 1), 1))
    if arr.shape != (max(int(steps), 1), 3) and not (steps == 0):
        raise ValueError("coeffs must be (a, b, c) or `steps` triples")
    return np.ascontiguousarray(arr.astype(np.float32).reshape(-1))


def update_scale(rows, cols, rms_scale=0.2, scale_mode=0) -> float:
    return float(_load().oracle_update_scale(int(rows), int(cols), float(rms_scale), int(scale_mode)))


# --------------------------------------------------------------------------
# Muon step
# --------------------------------------------------------------------------

@dataclass
class MuonConfig:
    lr: float = 0.02
    weight_decay: float = 0.1
    momentum: float = 0.95
    nesterov: bool = True
    ns_steps: int = 5
    ns_a: float = QUINTIC[0]
    ns_b: float = QUINTIC[1]
    ns_c: float = QUINTIC[2]
    norm_eps: float = 1e-7
    rms_scale: float = 0.2
    scale_mode: int = 0            # 0: rms_scale*sqrt(max(m,n)); 1: max(1, sqrt(rows/cols))
    skip_nonfinite: bool = False   # multi-matrix step: skip when any gradient is non-finite
    max_grad_norm: float = 0.0     # multi-matrix step: global-norm clip (<= 0: off)
    ns_coeffs: tuple = None        # None, or ns_steps (a, b, c) triples

    def c_struct(self):
        h = MuonHparams(self.lr, self.weight_decay, self.momentum,
                        int(bool(self.nesterov)), int(self.ns_steps),
                        self.ns_a, self.ns_b, self.ns_c, self.norm_eps,
                        self.rms_scale, int(self.scale_mode), int(bool(self.skip_nonfinite)),
                        self.max_grad_norm, 0, None)
        keep = None
        if self.ns_coeffs is not None:
            keep = coeff_table(self.ns_coeffs, self.ns_steps)
            h.ns_coeffs = keep.ctypes.data_as(ctypes.c_void_p)
        h._keep = keep  # the table must outlive the call
        return h


def muon_step_matrix(W, G, M, hp: MuonConfig = MuonConfig(), g_scale: float = 1.0, scale_g: bool = False,
                     accum: int = ACC_FP64, cast_after_scale: bool = False):
    """One Muon step on one matrix.

    W, M: fp32 (rows x cols).  G: fp32 values (a bf16 gradient is passed as
    its exact fp32 widening).  Returns (W_new, M_new, X0, O) with X0 and O in
    the wide orientation (min(rows,cols) x max(rows,cols)); inputs are not
    modified.  accum / cast_after_scale select the spread variants: NS
    products accumulated in fp32 (see matmul), and X0 = bf16(u * s) run
    unscaled instead of X0 = bf16(u) with s applied inside the first NS
    step."""
    W = np.array(W, dtype=np.float32, order="C", copy=True)
    M = np.array(M, dtype=np.float32, order="C", copy=True)
    G = np.ascontiguousarray(G, dtype=np.float32)
    if W.ndim != 2 or W.shape != G.shape or W.shape != M.shape:
        raise ValueError("W, G, M must be equal-shaped 2-D arrays")
    rows, cols = W.shape
    mp, np_ = min(rows, cols), max(rows, cols)
    X0 = np.empty((mp, np_), dtype=np.float32)
    O = np.empty((mp, np_), dtype=np.float32)
    h = hp.c_struct()
    rc = _load().oracle_muon_step_matrix_ex(_ptr(W), _ptr(G), _ptr(M), rows, cols,
                                            ctypes.byref(h), float(g_scale),
                                            1 if g_scale is not None and scale_g else 0,
                                            _accum(accum), 1 if cast_after_scale else 0,
                                            _ptr(X0), _ptr(O))
    if rc:
        raise RuntimeError(f"oracle_muon_step_matrix failed ({rc})")
    return W, M, X0, O


def momentum(G, M, mu=0.95, nesterov=True):
    """Steps 1-2 of the Muon step: returns (M_new, u), inputs untouched."""
    G = np.ascontiguousarray(G, dtype=np.float32)
    M = np.array(M, dtype=np.float32, order="C", copy=True)
    if G.shape != M.shape:
        raise ValueError("G and M must have the same shape")
    u = np.empty_like(M)
    _load().oracle_momentum(_ptr(G), _ptr(M), _ptr(u), M.size, float(mu), int(bool(nesterov)))
    return M, u


def normalize(u, eps=1e-7, cast_after_scale=False):
    """Steps 3-4: returns (X0 = bf16(u) wide as float values, s); the
    normalised NS input is s * X0, s applied inside the first NS step.
    cast_after_scale: X0 = bf16(u * s) instead, the NS input itself."""
    u = np.ascontiguousarray(u, dtype=np.float32)
    rows, cols = u.shape
    X0 = np.empty((min(rows, cols), max(rows, cols)), dtype=np.float64)
    fn = _load().oracle_normalize_cast_after if cast_after_scale else _load().oracle_normalize
    s = fn(_ptr(u), rows, cols, float(eps), _ptr(X0))
    return X0.astype(np.float32), float(s)


def final_update(W, O, lr=0.02, weight_decay=0.1, rms_scale=0.2, scale_mode=0):
    """Step 7 on W (rows x cols) with the wide NS output O; returns new W."""
    W = np.array(W, dtype=np.float32, order="C", copy=True)
    O = np.ascontiguousarray(O, dtype=np.float32)
    rows, cols = W.shape
    if O.shape != (min(rows, cols), max(rows, cols)):
        raise ValueError("O must be the wide (min x max) NS output")
    _load().oracle_final_update(_ptr(W), _ptr(O), rows, cols, float(lr), float(weight_decay),
                                float(rms_scale), int(scale_mode))
    return W


def step_stats(u, O, rms_scale=0.2, scale_mode=0):
    """(||u||_F, update RMS) of one matrix: u the look-ahead (rows x cols),
    O the wide NS output; the update RMS is that of fl(scale * O)."""
    u = np.ascontiguousarray(u, dtype=np.float32)
    O = np.ascontiguousarray(O, dtype=np.float32)
    rows, cols = u.shape
    if O.shape != (min(rows, cols), max(rows, cols)):
        raise ValueError("O must be the wide (min x max) NS output")
    un = ctypes.c_double(0.0)
    ur = ctypes.c_double(0.0)
    _load().oracle_step_stats(_ptr(u), _ptr(O), rows, cols, float(rms_scale), int(scale_mode),
                              ctypes.byref(un), ctypes.byref(ur))
    return float(un.value), float(ur.value)


def grad_stats(Gs):
    """(sum of g^2 over all gradients in fp64, count of non-finite elements)."""
    arrs = [np.ascontiguousarray(g, dtype=np.float32).reshape(-1) for g in Gs]
    ptrs = (ctypes.c_void_p * max(1, len(arrs)))(*[a.ctypes.data for a in arrs])
    ns = np.array([a.size for a in arrs] or [0], dtype=np.int64)
    sumsq = ctypes.c_double(0.0)
    bad = ctypes.c_int64(0)
    _load().oracle_grad_stats(ctypes.cast(ptrs, ctypes.c_void_p), _ptr(ns), len(arrs),
                              ctypes.byref(sumsq), ctypes.byref(bad))
    return float(sumsq.value), int(bad.value)


def clip_factor(sumsq: float, max_norm: float) -> float:
    return float(_load().oracle_clip_factor(float(sumsq), float(max_norm)))


def muon_step_list(Ws, Gs, Ms, hp: MuonConfig = MuonConfig()):
    """One Muon step over several matrices, with the call-wide gradient
    guard ([OPT] section 5.4): with skip_nonfinite, any NaN/inf gradient
    element leaves every matrix unchanged; with max_grad_norm > 0 every
    gradient is scaled by the global clip factor before the momentum.
    Returns (list of (W_new, M_new), skipped)."""
    clip_on = hp.max_grad_norm > 0
    clip = 1.0
    if clip_on or hp.skip_nonfinite:
        sumsq, bad = grad_stats(Gs)
        if hp.skip_nonfinite and bad > 0:
            return [(np.array(W, np.float32), np.array(M, np.float32)) for W, M in zip(Ws, Ms)], True
        if clip_on:
            clip = clip_factor(sumsq, hp.max_grad_norm)
    out = []
    for W, G, M in zip(Ws, Gs, Ms):
        W1, M1, _, _ = muon_step_matrix(W, G, M, hp, g_scale=clip, scale_g=clip_on)
        out.append((W1, M1))
    return out, False


# --------------------------------------------------------------------------
# AdamW
# --------------------------------------------------------------------------

@dataclass
class AdamwConfig:
    lr: float = 3e-4
    beta1: float = 0.9
    beta2: float = 0.95
    eps: float = 1e-8
    weight_decay: float = 0.1

    def c_struct(self) -> AdamwHparams:
        return AdamwHparams(self.lr, self.beta1, self.beta2, self.eps,
                            self.weight_decay)


def adamw_step(p, g, m, v, hp: AdamwConfig = AdamwConfig(), t: int = 1):
    """AdamW on flat fp32 buffers; returns new (p, m, v), inputs untouched."""
    p = np.array(p, dtype=np.float32, order="C", copy=True).reshape(-1)
    m = np.array(m, dtype=np.float32, order="C", copy=True).reshape(-1)
    v = np.array(v, dtype=np.float32, order="C", copy=True).reshape(-1)
    g = np.ascontiguousarray(g, dtype=np.float32).reshape(-1)
    if not (p.size == g.size == m.size == v.size):
        raise ValueError("p, g, m, v must have the same size")
    h = hp.c_struct()
    rc = _load().oracle_adamw_step(_ptr(p), _ptr(g), _ptr(m), _ptr(v), p.size,
                                   ctypes.byref(h), int(t))
    if rc:
        raise RuntimeError(f"oracle_adamw_step failed ({rc})")
    return p, m, v


# --------------------------------------------------------------------------
# Plan
# --------------------------------------------------------------------------

def ws_bytes_per_matrix(mp: int, np_: int) -> int:
    return int(_load().oracle_ws_bytes_per_matrix(int(mp), int(np_)))


def plan(shapes, ws_bytes: int) -> np.ndarray:
    """Plan for a list of (rows, cols): structured array with fields
    mat_idx, transposed, group_id, slot, chunk_id, mp, np (plan order)."""
    shapes = list(shapes)
    n = len(shapes)
    rows = np.array([s[0] for s in shapes] or [0], dtype=np.int64)
    cols = np.array([s[1] for s in shapes] or [0], dtype=np.int64)
    out = (PlanEntry * max(n, 1))()
    rc = _load().oracle_plan(_ptr(rows), _ptr(cols), n, int(ws_bytes),
                             ctypes.cast(out, ctypes.c_void_p))
    if rc:
        raise ValueError(f"oracle_plan failed ({rc})")
    dt = np.dtype([("mat_idx", np.int32), ("transposed", np.int32),
                   ("group_id", np.int32), ("slot", np.int32),
                   ("chunk_id", np.int32), ("pad_", np.int32),
                   ("mp", np.int64), ("np", np.int64)])
    arr = np.frombuffer(bytes(out), dtype=dt, count=max(n, 1)).copy()
    return arr[:n]
