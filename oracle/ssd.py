"""CPU fp64 oracle for the Mamba-2 (SSD) scan -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg may import this module;
the product path never does and shares no code with it.

What it computes (dpshk.com/news/3333417 section 6.1, "SSD: SSM = another form of attention", and section
6.2; pwwt.cn/news/5168881 section 2.3, "Mamba-2: turning the SSM into matrix multiplication"): the
selective recurrence with ONE scalar A per head instead of a diagonal (D, N) matrix, run independently by
every channel p of every head h, with B and C shared by the heads of a group (the grouped SSM of section
6.2, like grouped-query attention):

    dt_t     = softplus(dt_raw[b,h,t] + dt_bias[h])          (or without softplus)
    a_t      = exp(dt_t A[h])
    w_t      = dt_t                      simplified input scale (the default here)
             = expm1(dt_t A[h]) / A[h]   zero-order hold (limit dt_t at A = 0)
    h_t[p,n] = a_t h_{t-1}[p,n] + w_t B[b,g,t,n] x[b,h*P+p,t],     g = h // (H / G)
    y[b,h*P+p,t] = (sum_n C[b,g,t,n] h_t[p,n] + Dskip[h] x[b,h*P+p,t]) * SiLU(z[b,h*P+p,t])

The recurrence is the plain definition; the pages' matrix ("dual", attention-like) form y = M x with
M[k,i] = (C_k . B_i) w_i prod_{j=i+1..k} a_j is what the chunked kernel computes, and it is NOT used here:
the tests pin this oracle against that matrix form written out by brute force.

Per channel this is exactly the Mamba-1 recurrence of ``oracle.c`` with A[d, :] = A[h] for every state,
dt and its bias shared by the head's channels, and B, C taken from the head's group, so the arithmetic
runs in that fp64 C code; this module only lays the arrays out (``ssd_scan``).
"""
from __future__ import annotations

from typing import Optional, Sequence

import numpy as np

from . import _iptr, _load, _ptr, f64


def _take_rows(t, idx0, idx1):
    """t[idx0, idx1] as fp64 numpy, gathering before widening."""
    if hasattr(t, "detach"):
        import torch
        t = t.detach()[torch.as_tensor(idx0, dtype=torch.long), torch.as_tensor(idx1, dtype=torch.long)]
        return np.ascontiguousarray(f64(t))
    return np.ascontiguousarray(np.asarray(t, dtype=np.float64)[idx0, idx1])


def ssd_scan(inputs: dict, rows: Optional[Sequence[tuple]] = None, nthreads: int = 0):
    """SSD scan of a workload dict (see ``workloads.make_ssd_inputs``).

    ``rows``: optional list of (b, h, p) triples; default every (b, h, p) in (b, h*P+p) order.
    Returns (y (R, L), h_out (R, N), threads_used) as fp64 numpy arrays; row r is channel
    d = h * P + p of batch row b, and h_out[r] is the final state h_L[p, :] of that channel.
    """
    lib = _load()
    x = inputs["x"]
    Bsz, Dm, L = tuple(x.shape)
    H = int(inputs["nheads"])
    G = int(inputs["ngroups"])
    if H % G or Dm % H:
        raise ValueError("heads must split into equal groups and d_inner into equal heads")
    P = Dm // H
    N = int(inputs["Bm"].shape[-1])
    if rows is None:
        rb = np.repeat(np.arange(Bsz), Dm)
        rd = np.tile(np.arange(Dm), Bsz)
    else:
        rb = np.asarray([r[0] for r in rows], dtype=np.int64)
        rd = np.asarray([r[1] * P + r[2] for r in rows], dtype=np.int64)
    rh = rd // P
    R = len(rb)

    ur = _take_rows(x, rb, rd)
    dr = _take_rows(inputs["dt"], rb, rh)                      # the head's step, for each of its channels
    zr = _take_rows(inputs["z"], rb, rd) if inputs.get("z") is not None else None
    h0 = inputs.get("h0")
    h0r = _take_rows(h0.reshape(Bsz, Dm, N) if hasattr(h0, "reshape") else h0, rb, rd) if h0 is not None else None

    # per-channel parameters: the head's scalar A for every state, its D skip and dt bias
    A = f64(inputs["A"])
    A_ch = np.ascontiguousarray(np.repeat(A[:, None], P, axis=0).repeat(N, axis=1))     # (Dm, N)
    Dsk = f64(inputs.get("Dskip"))
    D_ch = np.ascontiguousarray(np.repeat(Dsk, P)) if Dsk is not None else None
    bias = f64(inputs.get("dt_bias"))
    bias_ch = np.ascontiguousarray(np.repeat(bias, P)) if bias is not None else None

    # B and C of every (batch, group) as (B*G, N, L); a row reads entry b*G + g
    Bf = np.ascontiguousarray(f64(inputs["Bm"]).transpose(0, 1, 3, 2).reshape(Bsz * G, N, L))
    Cf = np.ascontiguousarray(f64(inputs["Cm"]).transpose(0, 1, 3, 2).reshape(Bsz * G, N, L))
    rbc = np.ascontiguousarray(rb * G + rh // (H // G), dtype=np.int32)
    rdi = np.ascontiguousarray(rd, dtype=np.int32)

    y = np.empty((R, L), dtype=np.float64)
    h_out = np.empty((R, N), dtype=np.float64)
    nt = lib.oracle_scan_rows(R, L, N, _iptr(rbc), _iptr(rdi), _ptr(ur), _ptr(dr), _ptr(zr), _ptr(A_ch),
                              _ptr(D_ch), _ptr(bias_ch), None, None, 0, None, None, _ptr(Bf), _ptr(Cf),
                              _ptr(h0r), _ptr(y), _ptr(h_out), None, int(bool(inputs.get("delta_softplus", True))),
                              int(bool(inputs.get("zoh", False))), int(nthreads))
    if nt < 0:
        raise ValueError("oracle_scan_rows rejected its arguments")
    return y, h_out, nt
