"""Seeded synthetic inputs for the Muon and AdamW steps.

This module only draws random tensors of the right shapes, dtypes and value
distributions; it contains none of the optimizer's arithmetic, so both the
GPU library's tests and the oracle can be fed from it.

The five workloads (weights are (out, in) = (rows, cols); 'T' marks a tall
matrix, rows > cols, which the step orthogonalises in its transposed,
wide orientation):

  c1  one 256x512 weight; W~N(0,0.02), G fp32~N(0,1e-2), M~N(0,1e-2); seed 0
  c2  dense 24-layer decoder, hidden 2048, FFN 5632: per layer Wq,Wk,Wv,Wo
      2048x2048, gate/up 5632x2048 (T), down 2048x5632 -> 168 matrices.
      W~N(0,0.02); G bf16~N(0,s) with s log-uniform in [1e-4,1e-1] per
      matrix; M is a momentum after one prior step from zero, i.e.
      M~N(0,(1-mu)*s) in fp32; seed 1
  c3  fine-grained MoE: 8 layers x (Wq,Wk,Wv,Wo 2048x2048 + 64 experts x
      {gate 1408x2048, up 1408x2048, down 2048x1408 (T)}) -> 1568 matrices;
      distributions as c1; seed 2
  c4  large layer: gate, up 18432x7168 (T), down 7168x18432, Wq,Wk,Wv,Wo
      7168x7168; G bf16~N(0,1e-3), M~N(0,1e-3), W~N(0,0.02); seed 3
  c5  c3's expert set scaled to 16 layers x 128 experts (6144 matrices,
      distributions as c1) plus AdamW on an embedding and an LM head,
      163840x7168 fp32 each: p~N(0,0.02), g~N(0,1e-3), m~N(0,1e-3),
      v=|N(0,1e-6)|; step t=100; seed 4

"N(0,s)" means standard deviation s.
"""
from __future__ import annotations

import math
import random
from dataclasses import dataclass, field
from typing import List, Optional, Sequence, Tuple

import torch

MUON_HPARAMS = dict(lr=0.02, weight_decay=0.1, momentum=0.95, nesterov=True,
                    ns_steps=5, ns_a=3.4445, ns_b=-4.7750, ns_c=2.0315,
                    norm_eps=1e-7, rms_scale=0.2)
ADAMW_HPARAMS = dict(lr=3e-4, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1)
ADAMW_STEP = 100


@dataclass
class MatrixSpec:
    name: str
    rows: int
    cols: int
    g_dtype: torch.dtype     # torch.float32 or torch.bfloat16
    w_std: float
    g_std: Optional[float]   # None: drawn per matrix (log-uniform)
    m_std: Optional[float]   # None: (1 - mu) * g_std


@dataclass
class Workload:
    name: str
    description: str
    seed: int
    matrices: List[MatrixSpec]
    adamw_shapes: List[Tuple[int, int]] = field(default_factory=list)
    parity_sample: Optional[Sequence[int]] = None  # filled lazily

    @property
    def muon_params(self) -> int:
        return sum(m.rows * m.cols for m in self.matrices)

    @property
    def adamw_params(self) -> int:
        return sum(r * c for r, c in self.adamw_shapes)


def _c1():
    return Workload("c1", "single 256x512 Muon matrix", 0,
                    [MatrixSpec("w", 256, 512, torch.float32, 0.02, 1e-2, 1e-2)])


def _c2():
    mats = []
    for layer in range(24):
        for nm in ("q", "k", "v", "o"):
            mats.append(MatrixSpec(f"l{layer}.{nm}", 2048, 2048, torch.bfloat16,
                                   0.02, None, None))
        mats.append(MatrixSpec(f"l{layer}.gate", 5632, 2048, torch.bfloat16, 0.02, None, None))
        mats.append(MatrixSpec(f"l{layer}.up", 5632, 2048, torch.bfloat16, 0.02, None, None))
        mats.append(MatrixSpec(f"l{layer}.down", 2048, 5632, torch.bfloat16, 0.02, None, None))
    return Workload("c2", "dense 24-layer decoder (hidden 2048, FFN 5632), 168 matrices",
                    1, mats)


def _moe(name, layers, experts, seed, desc, attention=True, adamw=()):
    mats = []
    for layer in range(layers):
        if attention:
            for nm in ("q", "k", "v", "o"):
                mats.append(MatrixSpec(f"l{layer}.{nm}", 2048, 2048, torch.float32,
                                       0.02, 1e-2, 1e-2))
        for e in range(experts):
            mats.append(MatrixSpec(f"l{layer}.e{e}.gate", 1408, 2048, torch.float32, 0.02, 1e-2, 1e-2))
            mats.append(MatrixSpec(f"l{layer}.e{e}.up", 1408, 2048, torch.float32, 0.02, 1e-2, 1e-2))
            mats.append(MatrixSpec(f"l{layer}.e{e}.down", 2048, 1408, torch.float32, 0.02, 1e-2, 1e-2))
    return Workload(name, desc, seed, mats, list(adamw))


def _c3():
    return _moe("c3", 8, 64, 2,
                "fine-grained MoE, 8 layers x 64 experts + attention, 1568 matrices")


def _c4():
    mats = [MatrixSpec("gate", 18432, 7168, torch.bfloat16, 0.02, 1e-3, 1e-3),
            MatrixSpec("up", 18432, 7168, torch.bfloat16, 0.02, 1e-3, 1e-3),
            MatrixSpec("down", 7168, 18432, torch.bfloat16, 0.02, 1e-3, 1e-3)]
    for nm in ("q", "k", "v", "o"):
        mats.append(MatrixSpec(nm, 7168, 7168, torch.bfloat16, 0.02, 1e-3, 1e-3))
    return Workload("c4", "large layer, hidden 7168, FFN 18432, 7 matrices", 3, mats)


def _c5():
    return _moe("c5", 16, 128, 4,
                "full mixed step: 16 layers x 128 experts under Muon (6144 matrices) "
                "+ AdamW on embedding and LM head (163840x7168 each)",
                attention=False, adamw=[(163840, 7168), (163840, 7168)])


WORKLOADS = {"c1": _c1, "c2": _c2, "c3": _c3, "c4": _c4, "c5": _c5}


def get(name: str) -> Workload:
    return WORKLOADS[name]()


# Matrices whose outputs are compared against the oracle, chosen with
# random.Random(seed + 100) so the choice itself is reproducible.
def parity_sample(w: Workload) -> List[int]:
    rng = random.Random(w.seed + 100)
    idx = list(range(len(w.matrices)))
    if w.name == "c1":
        return [0]
    if w.name == "c2":
        return [i for i in idx if w.matrices[i].name.startswith(("l0.", "l23."))]
    if w.name in ("c3", "c5"):
        by_kind = {}
        for i in idx:
            kind = w.matrices[i].name.split(".")[-1]
            by_kind.setdefault(kind, []).append(i)
        pick = []
        for kind in ("gate", "up", "down"):
            pick += rng.sample(by_kind[kind], 2)
        if w.name == "c3":
            att = [i for i in idx if w.matrices[i].name.split(".")[-1] in "qkvo"]
            pick += rng.sample(att, 2)
        return sorted(pick)
    if w.name == "c4":
        return [0, 2, 3]
    return idx


# --------------------------------------------------------------------------
# Tensor generation
# --------------------------------------------------------------------------

@dataclass
class MuonTensors:
    W: List[torch.Tensor]
    G: List[torch.Tensor]
    M: List[torch.Tensor]
    storage: Tuple[torch.Tensor, ...]   # flat buffers the views live in


def _flat_views(flat: torch.Tensor, shapes):
    views, off = [], 0
    for r, c in shapes:
        views.append(flat[off:off + r * c].view(r, c))
        off += r * c
    return views


def make_muon(w: Workload, device="cpu", indices: Optional[Sequence[int]] = None,
              mu: float = MUON_HPARAMS["momentum"]) -> MuonTensors:
    """Draw W, G, M for the workload's matrices (all, or a subset).

    Draws happen in matrix order from one generator seeded with the
    workload's seed, so a subset reproduces the same values as the full set
    only when generated as the full set; use ``indices`` for small tests."""
    specs = w.matrices if indices is None else [w.matrices[i] for i in indices]
    gen = torch.Generator(device=device)
    gen.manual_seed(w.seed)
    shapes = [(s.rows, s.cols) for s in specs]
    total = sum(r * c for r, c in shapes)
    Wf = torch.empty(total, dtype=torch.float32, device=device)
    Mf = torch.empty(total, dtype=torch.float32, device=device)
    g_dtypes = {s.g_dtype for s in specs}
    if len(g_dtypes) != 1:
        raise ValueError("mixed gradient dtypes in one workload")
    Gf = torch.empty(total, dtype=g_dtypes.pop(), device=device)
    Ws, Gs, Ms = _flat_views(Wf, shapes), _flat_views(Gf, shapes), _flat_views(Mf, shapes)
    for s, Wv, Gv, Mv in zip(specs, Ws, Gs, Ms):
        g_std = s.g_std
        if g_std is None:
            u = torch.rand((), generator=gen, device=device, dtype=torch.float64).item()
            g_std = 10.0 ** (-4.0 + 3.0 * u)
        m_std = s.m_std if s.m_std is not None else (1.0 - mu) * g_std
        Wv.normal_(0.0, s.w_std, generator=gen)
        if Gv.dtype == torch.float32:
            Gv.normal_(0.0, g_std, generator=gen)
        else:
            tmp = torch.empty(Gv.shape, dtype=torch.float32, device=device)
            tmp.normal_(0.0, g_std, generator=gen)
            Gv.copy_(tmp)
            del tmp
        Mv.normal_(0.0, m_std, generator=gen)
    return MuonTensors(Ws, Gs, Ms, (Wf, Gf, Mf))


@dataclass
class AdamwTensors:
    p: torch.Tensor
    g: torch.Tensor
    m: torch.Tensor
    v: torch.Tensor


def make_adamw(n: int, seed: int, device="cpu") -> AdamwTensors:
    """p~N(0,0.02), g~N(0,1e-3), m~N(0,1e-3), v=|N(0,1e-6)|, fp32, flat."""
    gen = torch.Generator(device=device)
    gen.manual_seed(seed + 1000)
    out = []
    for std in (0.02, 1e-3, 1e-3, 1e-6):
        t = torch.empty(n, dtype=torch.float32, device=device)
        t.normal_(0.0, std, generator=gen)
        out.append(t)
    out[3].abs_()
    return AdamwTensors(*out)


def lowrank(rows: int, cols: int, seed: int, std: float, rank: int = 8, noise: float = 1e-3,
            basis_seed: Optional[int] = None) -> torch.Tensor:
    """An fp32 CPU matrix of rank `rank` plus i.i.d. noise, the shape real
    gradients tend to take: L R with L (rows x rank) and R (rank x cols) of
    i.i.d. normal draws, scaled to element standard deviation `std`, plus
    noise * std * N(0, 1) per element.  `basis_seed` (default: `seed`)
    draws L, so matrices that share it share their dominant column space."""
    g_basis = torch.Generator().manual_seed(seed if basis_seed is None else basis_seed)
    g = torch.Generator().manual_seed(seed + 7919)
    r = min(rank, rows, cols)
    left = torch.randn(rows, r, generator=g_basis, dtype=torch.float64)
    right = torch.randn(r, cols, generator=g, dtype=torch.float64)
    x = (left @ right) * (std / math.sqrt(r))
    x += torch.randn(rows, cols, generator=g, dtype=torch.float64) * (noise * std)
    return x.float()


def ns_input(rows: int, cols: int, seed: int, kind: str = "gaussian") -> torch.Tensor:
    """A wide bf16 NS input of Frobenius norm close to 1 (CPU tensor).

    kind 'gaussian': i.i.d. normal entries of standard deviation
    1/sqrt(rows*cols); 'lowrank': a rank-8 product of such draws plus 1e-3
    noise (a wide spread of singular values)."""
    gen = torch.Generator().manual_seed(seed)
    std = 1.0 / math.sqrt(rows * cols)
    x = torch.randn(rows, cols, generator=gen, dtype=torch.float64) * std
    if kind == "lowrank":
        r = min(8, rows)
        left = torch.randn(rows, r, generator=gen, dtype=torch.float64)
        right = torch.randn(r, cols, generator=gen, dtype=torch.float64)
        x = (left @ right) * (std / math.sqrt(r)) + 1e-3 * x
    return x.to(torch.bfloat16)
