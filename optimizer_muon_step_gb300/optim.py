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


class MuonAdamW(torch.optim.Optimizer):
    """Muon on `muon_params` (fp32, 2-D; gradients fp32, bf16 or fp16) and
    AdamW on `adamw_params` (fp32, any shape, fp32 gradients).

    Each part's ``lr`` and ``weight_decay`` live in its param group (group 0
    Muon, group 1 AdamW, when both are given), so torch.optim.lr_scheduler
    schedules work as usual; they start from `muon_hp` / `adamw_hp`, which
    hold the other hyper-parameters.  Parameters without a gradient are
    skipped.  AdamW's bias correction uses each parameter's own step count."""

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
        for group in self.param_groups:
            params = [p for p in group["params"] if p.grad is not None]
            if not params:
                continue
            if group["kind"] == "muon":
                hp = dataclasses.replace(self.muon_hp, lr=group["lr"], weight_decay=group["weight_decay"])
                self._muon(params, hp)
            else:
                hp = dataclasses.replace(self.adamw_hp, lr=group["lr"], weight_decay=group["weight_decay"])
                self._adamw(params, hp)
        return loss

    def _muon(self, params, hp):
        W, G, M = [], [], []
        for p in params:
            st = self.state[p]
            if "momentum_buffer" not in st:
                st["momentum_buffer"] = torch.zeros_like(p, memory_format=torch.contiguous_format)
            W.append(p)
            G.append(p.grad.contiguous())
            M.append(st["momentum_buffer"])
        need = muon_workspace_size([tuple(w.shape) for w in W], self.budget_bytes)
        if self._workspace is None or self._workspace.numel() < need:
            self._workspace = None
            self._workspace = allocate_workspace(need, W[0].device)
        muon_step_batched(W, G, M, hp, workspace=self._workspace)

    def _adamw(self, params, hp):
        by_step = {}
        for p in params:
            st = self.state[p]
            if "step" not in st:
                st["step"] = 0
                st["exp_avg"] = torch.zeros_like(p, memory_format=torch.contiguous_format)
                st["exp_avg_sq"] = torch.zeros_like(p, memory_format=torch.contiguous_format)
            st["step"] = int(st["step"]) + 1
            g = p.grad
            if g.dtype != torch.float32:
                raise TypeError("AdamW gradients must be fp32")
            by_step.setdefault(st["step"], []).append(
                (p.view(-1), g.contiguous().view(-1), st["exp_avg"].view(-1), st["exp_avg_sq"].view(-1)))
        for t, quads in sorted(by_step.items()):
            adamw_step_batched(quads, hp, step=t)
