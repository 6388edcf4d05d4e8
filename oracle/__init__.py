"""CPU fp64 oracle for the selective scan -- TEST INFRASTRUCTURE ONLY.

(The backward pass's oracle is ``oracle.backward``: autograd of the same recurrence in fp64 torch ops.)

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg may import
this package.  The product path (``selective_state_space_156_b300``) never imports it and
shares no code with it: the arithmetic lives in ``oracle.c`` (plain C, fp64, libm), this
file only marshals arrays.

Every function returns fp64 numpy arrays computed from the exact fp64 widening of the
(bf16- or fp32-rounded) tensors it is given.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lib = None

_dp = ctypes.POINTER(ctypes.c_double)
_ip = ctypes.POINTER(ctypes.c_int)


def build(force: bool = False) -> str:
    """Compile ``oracle.c`` into ``liboracle.so`` next to it (gcc, -O2, no fast-math)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + ".tmp"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fno-fast-math", "-shared", "-fPIC",
                               "-o", tmp, _SRC, "-lm", "-lpthread"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        lib.oracle_scan_rows.restype = ctypes.c_int
        lib.oracle_scan_rows.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, _ip, _ip,
                                         _dp, _dp, _dp, _dp, _dp, _dp, _dp, _dp, ctypes.c_int, _dp, _dp,
                                         _dp, _dp, _dp, _dp, _dp, _dp, ctypes.c_int, ctypes.c_int, ctypes.c_int]
        lib.oracle_conv1d_rows.restype = ctypes.c_int
        lib.oracle_conv1d_rows.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, _ip, _dp, _dp, _dp,
                                           ctypes.c_int, _dp]
        lib.oracle_state_update.restype = ctypes.c_int
        lib.oracle_state_update.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, _dp, _dp, _dp, _dp,
                                            _dp, _dp, _dp, _dp, _dp, _dp, _dp, ctypes.c_int, _dp, _dp,
                                            ctypes.c_int, ctypes.c_int, ctypes.c_int]
        _lib = lib
    return _lib


def f64(t) -> Optional[np.ndarray]:
    """Exact fp64 widening of a torch tensor or array (bf16 and fp32 widen exactly)."""
    if t is None:
        return None
    if hasattr(t, "detach"):
        t = t.detach().to("cpu")
        import torch
        t = t.to(torch.float64).numpy()
    return np.ascontiguousarray(np.asarray(t, dtype=np.float64))


def _ptr(a: Optional[np.ndarray]):
    if a is None:
        return None
    return a.ctypes.data_as(_dp)


def _iptr(a: np.ndarray):
    return a.ctypes.data_as(_ip)


def scan(inputs: dict, rows: Optional[Sequence[tuple]] = None, nthreads: int = 0, zoh: Optional[bool] = None,
         delta_softplus: Optional[bool] = None, extra: Optional[dict] = None):
    """Selective scan of a workload dict (see ``workloads.make_scan_inputs``).

    ``rows``: optional list of (b, d) pairs to compute; default is every row in (b, d) order.
    ``inputs["conv_init"]`` (B, D, W-1), when present with a conv, is the x history before t = 0.
    Returns (y (R, L), h_out (R, N), threads_used) as fp64 numpy arrays; with a dict ``extra`` and a
    conv, also stores the last W-1 inputs of every row as ``extra["conv_final"]`` (R, W-1); with
    ``extra["h_all"] = True`` it also stores the state after every step as ``extra["h_all"]`` (R, L, N).
    """
    lib = _load()
    Bsz, D, L = tuple(inputs["u"].shape)
    N = inputs["A"].shape[1]
    if rows is None:
        rb = np.repeat(np.arange(Bsz, dtype=np.int32), D)
        rd = np.tile(np.arange(D, dtype=np.int32), Bsz)
    else:
        rb = np.ascontiguousarray([r[0] for r in rows], dtype=np.int32)
        rd = np.ascontiguousarray([r[1] for r in rows], dtype=np.int32)
    R = len(rb)

    def rows_of(t, width):
        if t is None:
            return None
        if rows is None:
            return np.ascontiguousarray(f64(t).reshape(R, width))
        # take the rows first, then widen: the full tensor is never converted
        if hasattr(t, "detach"):
            import torch
            t = t.detach()[torch.as_tensor(rb, dtype=torch.long, device=t.device),
                           torch.as_tensor(rd, dtype=torch.long, device=t.device)]
            return np.ascontiguousarray(f64(t))
        return np.ascontiguousarray(np.asarray(t, dtype=np.float64)[rb, rd])

    ur = rows_of(inputs["u"], L)
    dr = rows_of(inputs["delta"], L)
    zr = rows_of(inputs.get("z"), L)
    h0 = rows_of(inputs.get("h0"), N)
    A = f64(inputs["A"])
    Bm = f64(inputs["Bm"])
    Cm = f64(inputs["Cm"])
    Dskip = f64(inputs.get("Dskip"))
    bias = f64(inputs.get("delta_bias"))
    cw = f64(inputs.get("conv_w"))
    cb = f64(inputs.get("conv_b"))
    W = 0 if cw is None else cw.shape[1]
    if cw is not None and cb is None:
        cb = np.zeros(D)
    ci = rows_of(inputs.get("conv_init"), W - 1) if (cw is not None and W > 1) else None
    cf = np.zeros((R, max(W - 1, 1)), dtype=np.float64) if (cw is not None and extra is not None) else None
    y = np.empty((R, L), dtype=np.float64)
    h_out = np.empty((R, N), dtype=np.float64)
    h_all = np.empty((R, L, N), dtype=np.float64) if (extra is not None and extra.get("h_all")) else None
    z_flag = inputs.get("zoh", True) if zoh is None else zoh
    sp_flag = inputs.get("delta_softplus", True) if delta_softplus is None else delta_softplus
    nt = lib.oracle_scan_rows(R, L, N, _iptr(rb), _iptr(rd), _ptr(ur), _ptr(dr), _ptr(zr), _ptr(A), _ptr(Dskip),
                              _ptr(bias), _ptr(cw), _ptr(cb), W, _ptr(ci), _ptr(cf), _ptr(Bm), _ptr(Cm), _ptr(h0),
                              _ptr(y), _ptr(h_out), _ptr(h_all), int(bool(sp_flag)), int(bool(z_flag)), int(nthreads))
    if nt < 0:
        raise ValueError("oracle_scan_rows rejected its arguments")
    if cf is not None:
        extra["conv_final"] = cf[:, :W - 1]
    if h_all is not None:
        extra["h_all"] = h_all
    return y, h_out, nt


def conv1d(x, w, b=None, silu: bool = True, rows: Optional[Sequence[tuple]] = None):
    """Causal depthwise conv1d (+ optional SiLU) of x (B, D, L) with w (D, W), b (D,)."""
    lib = _load()
    Bsz, D, L = tuple(x.shape)
    wa = f64(w)
    ba = f64(b)
    if rows is None:
        rd = np.tile(np.arange(D, dtype=np.int32), Bsz)
        xr = np.ascontiguousarray(f64(x).reshape(Bsz * D, L))
    else:
        rb = np.asarray([r[0] for r in rows], dtype=np.int64)
        rd = np.ascontiguousarray([r[1] for r in rows], dtype=np.int32)
        if hasattr(x, "detach"):
            import torch
            xr = np.ascontiguousarray(f64(x.detach()[torch.as_tensor(rb), torch.as_tensor(rd, dtype=torch.long)]))
        else:
            xr = np.ascontiguousarray(np.asarray(x, dtype=np.float64)[rb, rd])
    R = len(rd)
    out = np.empty((R, L), dtype=np.float64)
    rc = lib.oracle_conv1d_rows(R, L, wa.shape[1], _iptr(rd), _ptr(xr), _ptr(wa), _ptr(ba), int(bool(silu)),
                                _ptr(out))
    if rc < 0:
        raise ValueError("oracle_conv1d_rows rejected its arguments")
    return out


def state_update(state, u, delta, A, Bm, Cm, Dskip=None, delta_bias=None, z=None, zoh: bool = True,
                 delta_softplus: bool = True, nthreads: int = 0, conv_w=None, conv_b=None, conv_state=None):
    """One decode step.  ``state`` (B, D, N) is widened to fp64 and returned updated (not in place)
    together with y (B, D).  With ``conv_w`` (D, W), u is the conv input x and ``conv_state``
    (B, D, W-1) the previous W-1 inputs; the updated conv state is returned third."""
    lib = _load()
    st = f64(state).copy()
    ua = f64(u)
    Bsz, D = ua.shape
    N = st.shape[2]
    y = np.empty((Bsz, D), dtype=np.float64)
    cw = f64(conv_w)
    W = 0 if cw is None else cw.shape[1]
    cs = None
    if cw is not None:
        cs = (f64(conv_state).copy() if conv_state is not None and W > 1
              else np.zeros((Bsz, D, max(W - 1, 1)), dtype=np.float64))
    rc = lib.oracle_state_update(Bsz, D, N, _ptr(st), _ptr(ua), _ptr(f64(delta)), _ptr(f64(A)), _ptr(f64(Bm)),
                                 _ptr(f64(Cm)), _ptr(f64(Dskip)), _ptr(f64(delta_bias)), _ptr(f64(z)), _ptr(cw),
                                 _ptr(f64(conv_b)), W, _ptr(cs), _ptr(y), int(bool(delta_softplus)), int(bool(zoh)),
                                 int(nthreads))
    if rc < 0:
        raise ValueError("oracle_state_update rejected its arguments")
    if cw is not None:
        return st, y, cs[..., :W - 1]
    return st, y
