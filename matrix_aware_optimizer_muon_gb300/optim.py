"""Stateful wrapper: momentum buffers, workspace and step counter around muon_periodic_step."""
from __future__ import annotations

from typing import Dict, List, Sequence

import torch

from . import _lib


class PeriodicMuon:
    """Periodic Row-wise Muon over a list of 2-D weight tensors (K = 1 is vanilla Muon).

    State is the fp32 momentum of every matrix and the integer step, which decides
    the branch (Newton-Schulz refresh when step % K == 0, RowNorm otherwise).
    """

    def __init__(self, params: Sequence[torch.Tensor], K: int = 3, gamma: float = 0.15, mu: float = 0.95,
                 eta: float = 0.02, lam: float = 0.01, ns5_mode: str = "bf16",
                 aux_params: Sequence[torch.Tensor] = (), aux_lr: float = 1e-4, betas=(0.9, 0.999),
                 eps: float = 1e-8):
        """aux_params: parameters Muon does not take (biases, norms, out-of-block weights);
        they are updated by AdamW with learning rate aux_lr and the shared weight decay lam."""
        self.params: List[torch.Tensor] = list(params)
        self.aux = list(aux_params)
        self.aux_lr, self.betas, self.eps = aux_lr, betas, eps
        self.aux_m = [torch.zeros(p.numel(), dtype=torch.float32, device=p.device) for p in self.aux]
        self.aux_v = [torch.zeros(p.numel(), dtype=torch.float32, device=p.device) for p in self.aux]
        if not self.params:
            raise ValueError("no parameters")
        self.K, self.gamma, self.mu, self.eta, self.lam, self.ns5_mode = K, gamma, mu, eta, lam, ns5_mode
        dev = self.params[0].device
        self.M = [torch.zeros(p.shape, dtype=torch.float32, device=dev) for p in self.params]
        self.ws = _lib.alloc_workspace([tuple(p.shape) for p in self.params], ns5_mode, device=dev)
        self.step_count = 0
        # W and M never move, so the C matrix array is built once; each step only
        # points it at that step's gradients (after checking them like the array build does).
        self._arr, self._n = _lib.make_matrices(self.M, self.params, self.params)
        self._gdt = None

    def step(self, grads: Sequence[torch.Tensor], aux_grads: Sequence[torch.Tensor] = (), stream=None) -> int:
        if len(grads) != self._n:
            raise ValueError("one gradient per matrix")
        for i, (g, p) in enumerate(zip(grads, self.params)):
            if g.shape != p.shape:
                raise ValueError("W, G and M must have the same shape")
            self._arr[i].G = _lib._ptr(g)
            self._arr[i].g_dtype = _lib._dt(g)
        br = _lib.periodic_step_prepared(self._arr, self._n, self.step_count, self.ws, self.K, self.gamma, self.mu,
                                         self.eta, self.lam, self.ns5_mode, stream=stream)
        if self.aux:
            if len(aux_grads) != len(self.aux):
                raise ValueError("one gradient per auxiliary parameter")
            _lib.muon_adamw_step([p.view(-1) for p in self.aux], [g.reshape(-1) for g in aux_grads], self.aux_m,
                                 self.aux_v, self.step_count + 1, self.aux_lr, self.betas[0], self.betas[1],
                                 self.eps, self.lam, stream=stream)
        self.step_count += 1
        return br

    def check(self, stream=None) -> int:
        return _lib.muon_check_status(self.ws, stream)

    def state_dict(self) -> Dict:
        return {"step": self.step_count, "M": [m.detach().clone() for m in self.M],
                "aux_m": [m.detach().clone() for m in self.aux_m], "aux_v": [v.detach().clone() for v in self.aux_v],
                "hyper": dict(K=self.K, gamma=self.gamma, mu=self.mu, eta=self.eta, lam=self.lam,
                              ns5_mode=self.ns5_mode)}

    def load_state_dict(self, sd: Dict) -> None:
        """Restores the momentum, the AdamW moments and the step.  The schedule period K
        and the NS5 mode must match the saved ones (they change which branch a step takes
        and its arithmetic); learning rate, weight decay and gamma may differ."""
        hyper = sd.get("hyper", {})
        for key in ("K", "ns5_mode"):
            if key in hyper and hyper[key] != getattr(self, key):
                raise ValueError(f"state was saved with {key}={hyper[key]!r}, this optimizer has {getattr(self, key)!r}")
        if len(sd["M"]) != len(self.M):
            raise ValueError("state has a different number of matrices")
        aux_m, aux_v = sd.get("aux_m", []), sd.get("aux_v", [])
        if len(aux_m) != len(self.aux_m) or len(aux_v) != len(self.aux_v):
            raise ValueError("state has a different number of auxiliary parameters")
        for dst, src in zip(self.M + self.aux_m + self.aux_v, list(sd["M"]) + list(aux_m) + list(aux_v)):
            if tuple(dst.shape) != tuple(src.shape):
                raise ValueError("state shape mismatch")
            dst.copy_(src)
        self.step_count = int(sd["step"])
