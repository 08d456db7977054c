"""A torch.optim.Optimizer over the library: Muon for the hidden weight
matrices, AdamW for every other parameter.

"LLM training series, part 2: optimizers" (section 4.3) uses Muon on the
2-D hidden matrices and AdamW on the rest (embedding, LM head, norm gains,
biases); the caller passes the two lists.  Everything here is bookkeeping:
the state buffers (Muon's momentum, AdamW's m and v and step count) live in
``self.state`` like any torch optimizer's, so ``state_dict`` /
``load_state_dict`` save and restore them (section 5.3: resuming without
the optimizer state is not resuming), and ``step`` hands every tensor to
muon_step_batched and adamw_step_batched.  No arithmetic runs in Python.
"""
from __future__ import annotations

import dataclasses

import torch

from . import (AdamwHparams, MuonHparams, adamw_step_batched, allocate_workspace, muon_step_batched,
               muon_workspace_size)

_MUON_GRAD_DTYPES = (torch.float32, torch.bfloat16, torch.float16)


def common_device(tensors):
    """The one device every tensor of `tensors` lives on.  The library
    launches on the current device's stream and reads every pointer there,
    so a list that spans devices is refused (ValueError)."""
    devices = {t.device for t in tensors}
    if len(devices) != 1:
        raise ValueError(f"all parameters must be on one CUDA device, got {sorted(map(str, devices))}")
    return devices.pop()


class MuonAdamW(torch.optim.Optimizer):
    """Muon on `muon_params` (fp32, 2-D; gradients fp32, bf16 or fp16, any
    strides) and AdamW on `adamw_params` (fp32, any shape, fp32 gradients).

    Each part's ``lr`` and ``weight_decay`` live in its param group (group 0
    Muon, group 1 AdamW, when both are given), so torch.optim.lr_scheduler
    schedules work as usual; they start from `muon_hp` / `adamw_hp`, which
    hold the other hyper-parameters.  Parameters without a gradient are
    skipped (their state is kept as it is).  AdamW's bias correction uses
    each parameter's own step count.  Every parameter must live on one CUDA
    device; ``step`` runs there, on that device's current stream, whatever
    device is current when it is called.  A ``step`` that raises (a
    gradient of the wrong dtype, shape or device) changes no state of the
    part it rejects."""

    def __init__(self, muon_params, adamw_params, muon_hp: MuonHparams | None = None,
                 adamw_hp: AdamwHparams | None = None, budget_bytes: int = 16 << 30):
        muon_hp = muon_hp if muon_hp is not None else MuonHparams()
        adamw_hp = adamw_hp if adamw_hp is not None else AdamwHparams()
        groups = [{"params": list(muon_params), "kind": "muon", "lr": muon_hp.lr,
                   "weight_decay": muon_hp.weight_decay},
                  {"params": list(adamw_params), "kind": "adamw", "lr": adamw_hp.lr,
                   "weight_decay": adamw_hp.weight_decay}]
        groups = [g for g in groups if g["params"]]
        if not groups:
            raise ValueError("no parameters")
        super().__init__(groups, defaults={})
        for g in self.param_groups:
            for p in g["params"]:
                if p.dtype != torch.float32 or not p.is_cuda:
                    raise TypeError("parameters must be fp32 CUDA tensors")
                if g["kind"] == "muon" and p.dim() != 2:
                    raise ValueError("Muon parameters must be 2-D matrices")
        self.device = common_device([p for g in self.param_groups for p in g["params"]])
        self.muon_hp = muon_hp
        self.adamw_hp = adamw_hp
        self.budget_bytes = int(budget_bytes)
        self._workspace = None

    @torch.no_grad()
    def step(self, closure=None):
        loss = None
        if closure is not None:
            with torch.enable_grad():
                loss = closure()
        with torch.cuda.device(self.device):
            stream = torch.cuda.current_stream(self.device)
            for group in self.param_groups:
                params = [p for p in group["params"] if p.grad is not None]
                if not params:
                    continue
                if group["kind"] == "muon":
                    hp = dataclasses.replace(self.muon_hp, lr=group["lr"], weight_decay=group["weight_decay"])
                    self._muon(params, hp, stream)
                else:
                    hp = dataclasses.replace(self.adamw_hp, lr=group["lr"], weight_decay=group["weight_decay"])
                    self._adamw(params, hp, stream)
        return loss

    def _check_grad(self, p, dtypes):
        g = p.grad
        if g.dtype not in dtypes:
            raise TypeError(f"gradient dtype {g.dtype} not one of {dtypes}")
        if g.shape != p.shape:
            raise ValueError(f"gradient shape {tuple(g.shape)} != parameter shape {tuple(p.shape)}")
        if g.device != self.device:
            raise ValueError(f"gradient on {g.device}, parameters on {self.device}")

    def _muon(self, params, hp, stream):
        for p in params:                      # every check before any state changes
            self._check_grad(p, _MUON_GRAD_DTYPES)
        W, G, M = [], [], []
        for p in params:
            st = self.state[p]
            if "momentum_buffer" not in st:
                st["momentum_buffer"] = torch.zeros_like(p, memory_format=torch.contiguous_format)
            W.append(p)
            G.append(p.grad.contiguous())
            M.append(st["momentum_buffer"])
        need = muon_workspace_size([tuple(w.shape) for w in W], self.budget_bytes)
        ws = self._workspace
        if ws is None or ws.numel() < need or ws.device != self.device:
            self._workspace = None
            self._workspace = allocate_workspace(need, self.device)
        muon_step_batched(W, G, M, hp, workspace=self._workspace, stream=stream)

    def _adamw(self, params, hp, stream):
        for p in params:                      # every check before any state changes
            self._check_grad(p, (torch.float32,))
        by_step = {}
        for p in params:
            st = self.state[p]
            if "step" not in st:
                st["step"] = 0
                st["exp_avg"] = torch.zeros_like(p, memory_format=torch.contiguous_format)
                st["exp_avg_sq"] = torch.zeros_like(p, memory_format=torch.contiguous_format)
            t = int(st["step"]) + 1
            by_step.setdefault(t, []).append(p)
        for t, ps in sorted(by_step.items()):
            quads = [(p.view(-1), p.grad.contiguous().view(-1), self.state[p]["exp_avg"].view(-1),
                      self.state[p]["exp_avg_sq"].view(-1)) for p in ps]
            adamw_step_batched(quads, hp, step=t, stream=stream)
            for p in ps:                      # counted once the update is enqueued
                self.state[p]["step"] = t
