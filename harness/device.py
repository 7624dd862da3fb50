"""Upload generated layers to the GPU and bind them to a library plan (torch for memory only).

Test and benchmark infrastructure: moves the generator's byte arrays into
device tensors and builds the expert descriptor array the library binds.
"""
from __future__ import annotations

import numpy as np
import torch

import quantized_expert_ffn_bias_gb300 as coli

from . import Layer, ExpertBank, X_BF16


def to_dev(a: np.ndarray, device) -> torch.Tensor:
    """numpy -> device tensor with the same bytes (uint16 bf16/fp16 patterns travel as int16)."""
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        t = torch.from_numpy(a.view(np.int16))
    else:
        t = torch.from_numpy(a)
    return t.to(device, non_blocking=False)


class DeviceBank:
    """One expert bank resident on the device: q/s/z of gate, up, down with a leading expert axis."""

    def __init__(self, bank: ExpertBank, device):
        self.bank = bank
        self.E = bank.E
        self.t = {}
        for name in ("gate", "up", "down"):
            m = getattr(bank, name)
            self.t[name] = (to_dev(m.q, device), to_dev(m.s, device), to_dev(m.z, device))

    def expert(self, e: int) -> coli.coli_expert:
        def qm(name):
            q, s, z = self.t[name]
            return coli.qmat(q[e].data_ptr(), s[e].data_ptr(), z[e].data_ptr())
        return coli.coli_expert(qm("gate"), qm("up"), qm("down"))

    @property
    def nbytes(self) -> int:
        return sum(x.numel() * x.element_size() for v in self.t.values() for x in v)


class DeviceLayer:
    """A generated layer on the device with a bound plan and a workspace for up to T_max tokens."""

    def __init__(self, layer: Layer, T_max: int, xtype: int = X_BF16, device="cuda", workspace: bool = True):
        self.layer = layer
        self.device = torch.device(device)
        self.experts = DeviceBank(layer.experts, self.device)
        self.shared = DeviceBank(layer.shared, self.device) if layer.shared is not None else None
        self.router_w = to_dev(layer.router_w, self.device)
        self.bias = to_dev(layer.bias, self.device)
        self.plan = coli.Plan(T_max=T_max, d=layer.d, d_ff=layer.F, E=layer.E, k=layer.k,
                              routed_scale=float(layer.rho), qtype=layer.qtype, xtype=xtype,
                              has_shared=layer.shared is not None,
                              shared_d_ff=layer.shared.F if layer.shared is not None else 0)
        self.plan.bind_experts([self.experts.expert(e) for e in range(layer.E)],
                               self.shared.expert(0) if self.shared is not None else None)
        self.ws = torch.empty(self.plan.workspace_bytes, dtype=torch.uint8, device=self.device) if workspace else None

    def forward(self, x: torch.Tensor, out: torch.Tensor | None = None, residual: torch.Tensor | None = None,
                ws: torch.Tensor | None = None, stream=None) -> torch.Tensor:
        T = x.shape[0]
        if out is None:
            out = torch.empty((T, self.layer.d), dtype=torch.float32, device=self.device)
        ws = self.ws if ws is None else ws
        st = stream if stream is not None else torch.cuda.current_stream(self.device)
        self.plan.forward(T, x, self.router_w, self.bias, out, ws, ws.numel(), residual=residual, stream=st)
        return out

    def routing(self, T: int, ws: torch.Tensor | None = None):
        """(topk_idx, topk_w, near_tie, offsets, pair_token, pair_slot) of the last forward, as numpy."""
        ws = self.ws if ws is None else ws
        L = self.layer
        dev = self.device
        idx = torch.empty((T, L.k), dtype=torch.int32, device=dev)
        w = torch.empty((T, L.k), dtype=torch.float32, device=dev)
        nt = torch.empty(T, dtype=torch.int32, device=dev)
        off = torch.empty(L.E + 1, dtype=torch.int32, device=dev)
        pt = torch.empty(T * L.k, dtype=torch.int32, device=dev)
        ps = torch.empty(T * L.k, dtype=torch.int32, device=dev)
        self.plan.debug_routing(ws, T, idx, w, nt, off, pt, ps, stream=torch.cuda.current_stream(dev))
        torch.cuda.synchronize(dev)
        return tuple(t.cpu().numpy() for t in (idx, w, nt, off, pt, ps))

    def close(self):
        self.plan.close()
