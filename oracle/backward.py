"""fp64 CPU oracle of the selective scan's backward pass -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU legs may use this module.

The forward of the scan is written out here once more in plain PyTorch fp64 ops, sequential in time
(the recurrence of dpshk.com/news/3333417 sections 2.2, 2.3, 4.1, 5.1 and 5.2, as the C oracle computes
it), and PyTorch's autograd differentiates it: the gradient of <y, dy> + <h_L, dh_out> with respect to
every input.  Gradients are the ones training needs (pwwt.cn/news/5168881 section 3.2 notes that they
run back along time through the state recurrence).  The tests pin this against central finite
differences of the C forward oracle, which shares no code with it.

One reading: the zero-order-hold factor E = (exp(dt a) - 1) / a is written as dt * phi(dt a) with
phi(x) = expm1(x) / x (phi(0) = 1, by its series near 0), so that the a = 0 limit and its derivative
dE/da = dt^2 / 2 come out of the same smooth expression.
"""
from __future__ import annotations

from typing import Optional

import numpy as np
import torch


def _t(x, requires_grad=True):
    if x is None:
        return None
    t = torch.as_tensor(x.detach().to("cpu") if hasattr(x, "detach") else x).to(torch.float64).clone()
    return t.requires_grad_(requires_grad)


def _phi(x):
    """expm1(x) / x, with its Taylor series near 0 (smooth, exact derivative there)."""
    small = x.abs() < 1e-5
    xs = torch.where(small, torch.ones_like(x), x)
    return torch.where(small, 1.0 + x / 2.0 + x * x / 6.0, torch.expm1(xs) / xs)


def _softplus(s):
    return torch.where(s > 0, s + torch.log1p(torch.exp(-s.abs())), torch.log1p(torch.exp(-s.abs())))


def _silu(v):
    return v * torch.sigmoid(v)


def forward(u, delta, A, Bm, Cm, Dskip=None, delta_bias=None, z=None, conv_w=None, conv_b=None, h0=None,
            conv_init=None, zoh=True, delta_softplus=True):
    """The scan forward in plain fp64 torch ops; returns (y (B, D, L), h_L (B, D, N))."""
    Bsz, D, L = u.shape
    N = A.shape[1]
    if conv_w is not None:
        W = conv_w.shape[1]
        hist = conv_init if conv_init is not None else torch.zeros((Bsz, D, W - 1), dtype=u.dtype)
        xx = torch.cat([hist, u], dim=-1)  # x_{-W+1} .. x_{L-1}
        c = torch.zeros((Bsz, D, L), dtype=u.dtype) + (conv_b[None, :, None] if conv_b is not None else 0.0)
        for k in range(W):  # tap k multiplies x_{t-W+1+k}
            c = c + conv_w[None, :, k, None] * xx[..., k:k + L]
        v = _silu(c)
    else:
        v = u
    s = delta + (delta_bias[None, :, None] if delta_bias is not None else 0.0)
    dt = _softplus(s) if delta_softplus else s
    h = h0 if h0 is not None else torch.zeros((Bsz, D, N), dtype=u.dtype)
    ys = []
    for t in range(L):
        x = dt[:, :, t, None] * A[None]                     # (B, D, N)
        Abar = torch.exp(x)
        E = dt[:, :, t, None] * (_phi(x) if zoh else torch.ones_like(x))
        h = Abar * h + E * Bm[:, None, :, t] * v[:, :, t, None]
        yt = (h * Cm[:, None, :, t]).sum(-1)
        if Dskip is not None:
            yt = yt + Dskip[None, :] * v[:, :, t]
        ys.append(yt)
    y = torch.stack(ys, dim=-1)
    if z is not None:
        y = y * _silu(z)
    return y, h


def scan_bwd(inputs: dict, dy, dh_out=None, zoh: Optional[bool] = None,
             delta_softplus: Optional[bool] = None) -> dict:
    """Gradients of sum(y * dy) + sum(h_L * dh_out) with respect to every input of the workload dict
    (see ``workloads.make_scan_inputs``).  Returns fp64 numpy arrays keyed like the inputs ("u" is the
    gradient of the conv input x when a conv is given; "h0" the gradient of the initial state, zero-init
    when the call had none)."""
    names = ["u", "delta", "A", "Bm", "Cm", "Dskip", "delta_bias", "z", "conv_w", "conv_b", "h0", "conv_init"]
    T = {k: _t(inputs.get(k)) for k in names}
    Bsz, D, L = T["u"].shape
    N = T["A"].shape[1]
    if T["h0"] is None:
        T["h0"] = torch.zeros((Bsz, D, N), dtype=torch.float64, requires_grad=True)
    z_flag = inputs.get("zoh", True) if zoh is None else zoh
    sp_flag = inputs.get("delta_softplus", True) if delta_softplus is None else delta_softplus
    y, hL = forward(T["u"], T["delta"], T["A"], T["Bm"], T["Cm"], T["Dskip"], T["delta_bias"], T["z"], T["conv_w"],
                    T["conv_b"], T["h0"], T["conv_init"], zoh=z_flag, delta_softplus=sp_flag)
    loss = (y * _t(dy, False)).sum()
    if dh_out is not None:
        loss = loss + (hL * _t(dh_out, False)).sum()
    live = [k for k in names if T[k] is not None]
    grads = torch.autograd.grad(loss, [T[k] for k in live], allow_unused=True)
    out = {}
    for k, gk in zip(live, grads):
        out[k] = np.zeros(tuple(T[k].shape)) if gk is None else gk.numpy()
    out["y"] = y.detach().numpy()
    return out
