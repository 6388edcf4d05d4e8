"""B300 (sm_103a) selective state-space scan: Python binding of libssm_b300.so.

This module only marshals arguments: it checks that tensors live on the GPU with the expected
dtype and layout, passes their device pointers and sizes to the C ABI (include/ssm_scan.h), and
raises if a call fails.  Every step of the computation runs in the library's CUDA kernels.  There
is no CPU fallback: importing works without the library, but any call raises if it is missing.

Entry points (same names as the C ABI):
  ssm_scan_fwd(u, delta, A, Bm, Cm, ...)      -> y  (and the final state if requested)
  causal_conv1d_fwd(x, w, b=None, silu=True)  -> y
  ssm_state_update(state, u, delta, A, Bm, Cm, ...)  -> y  (state updated in place)
  ssm_scan_workspace_size(...)                -> bytes of optional scratch for the L split
  ssm_scan_bwd(u, delta, A, Bm, Cm, dy, h_ckpt, ...) -> gradients of every input
  ssd_scan_fwd(x, dt, A, Bm, Cm, nheads=..., ngroups=...) -> y (Mamba-2 / SSD layer, tensor cores)
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

__all__ = ["ssm_scan_fwd", "ssm_scan_fwd_static", "causal_conv1d_fwd", "ssm_state_update", "ssm_scan_workspace_size",
           "ssm_scan_bwd", "ssd_scan_fwd", "lib", "SsmError", "ScanParams", "SsdParams", "LIB_PATH"]

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libssm_b300.so")

SSM_OK, SSM_ERR_INVALID_ARG, SSM_ERR_UNSUPPORTED, SSM_ERR_CUDA = 0, 1, 2, 3
SSM_F32, SSM_BF16 = 0, 1


class SsmError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"[status {status}] {msg}")
        self.status = status


class ScanParams(ctypes.Structure):
    """Mirror of ssm_scan_params in include/ssm_scan.h (same field order and types)."""
    _fields_ = [
        ("batch", ctypes.c_int), ("dim", ctypes.c_int), ("dstate", ctypes.c_int), ("seqlen", ctypes.c_int),
        ("in_dtype", ctypes.c_int), ("out_dtype", ctypes.c_int),
        ("u", ctypes.c_void_p), ("delta", ctypes.c_void_p), ("A", ctypes.c_void_p),
        ("Bm", ctypes.c_void_p), ("Cm", ctypes.c_void_p), ("Dskip", ctypes.c_void_p),
        ("delta_bias", ctypes.c_void_p), ("z", ctypes.c_void_p), ("conv_w", ctypes.c_void_p),
        ("conv_b", ctypes.c_void_p), ("conv_width", ctypes.c_int), ("h0", ctypes.c_void_p),
        ("h_out", ctypes.c_void_p), ("y", ctypes.c_void_p), ("delta_softplus", ctypes.c_int),
        ("zoh", ctypes.c_int), ("workspace", ctypes.c_void_p), ("workspace_bytes", ctypes.c_size_t),
        ("conv_init", ctypes.c_void_p), ("conv_final", ctypes.c_void_p),
        ("state_indices", ctypes.c_void_p), ("h_all", ctypes.c_void_p), ("h_ckpt", ctypes.c_void_p),
    ]


class ScanBwdParams(ctypes.Structure):
    """Mirror of ssm_scan_bwd_params in include/ssm_scan.h (same field order and types)."""
    _fields_ = [
        ("batch", ctypes.c_int), ("dim", ctypes.c_int), ("dstate", ctypes.c_int), ("seqlen", ctypes.c_int),
        ("in_dtype", ctypes.c_int),
        ("u", ctypes.c_void_p), ("delta", ctypes.c_void_p), ("A", ctypes.c_void_p), ("Bm", ctypes.c_void_p),
        ("Cm", ctypes.c_void_p), ("Dskip", ctypes.c_void_p), ("delta_bias", ctypes.c_void_p), ("z", ctypes.c_void_p),
        ("conv_w", ctypes.c_void_p), ("conv_b", ctypes.c_void_p), ("conv_width", ctypes.c_int),
        ("conv_init", ctypes.c_void_p), ("h0", ctypes.c_void_p), ("delta_softplus", ctypes.c_int),
        ("zoh", ctypes.c_int), ("h_ckpt", ctypes.c_void_p), ("dy", ctypes.c_void_p), ("dh_out", ctypes.c_void_p),
        ("du", ctypes.c_void_p), ("ddelta", ctypes.c_void_p), ("dz", ctypes.c_void_p), ("dA", ctypes.c_void_p),
        ("dB", ctypes.c_void_p), ("dC", ctypes.c_void_p), ("dDskip", ctypes.c_void_p),
        ("ddelta_bias", ctypes.c_void_p), ("dconv_w", ctypes.c_void_p), ("dconv_b", ctypes.c_void_p),
        ("dconv_init", ctypes.c_void_p), ("dh0", ctypes.c_void_p), ("workspace", ctypes.c_void_p),
        ("workspace_bytes", ctypes.c_size_t),
    ]


class StepParams(ctypes.Structure):
    """Mirror of ssm_step_params in include/ssm_scan.h (same field order and types)."""
    _fields_ = [
        ("batch", ctypes.c_int), ("dim", ctypes.c_int), ("dstate", ctypes.c_int), ("dtype", ctypes.c_int),
        ("state", ctypes.c_void_p), ("x", ctypes.c_void_p), ("delta", ctypes.c_void_p), ("A", ctypes.c_void_p),
        ("Bm", ctypes.c_void_p), ("Cm", ctypes.c_void_p), ("Dskip", ctypes.c_void_p),
        ("delta_bias", ctypes.c_void_p), ("z", ctypes.c_void_p), ("conv_w", ctypes.c_void_p),
        ("conv_b", ctypes.c_void_p), ("conv_width", ctypes.c_int), ("conv_state", ctypes.c_void_p),
        ("y", ctypes.c_void_p), ("delta_softplus", ctypes.c_int), ("zoh", ctypes.c_int),
        ("state_indices", ctypes.c_void_p),
    ]


_lib = None


def lib() -> ctypes.CDLL:
    """The loaded C library (ctypes).  Raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"{LIB_PATH} is missing: build it with `python -m selective_state_space_156_b300.build`"
                              " (there is no CPU fallback)")
        L = ctypes.CDLL(LIB_PATH)
        vp, i, st = ctypes.c_void_p, ctypes.c_int, ctypes.c_int
        L.ssm_scan_fwd.restype = st
        L.ssm_scan_fwd.argtypes = [ctypes.POINTER(ScanParams), vp]
        L.ssm_scan_fwd_static.restype = st
        L.ssm_scan_fwd_static.argtypes = [ctypes.POINTER(ScanParams), vp]
        L.ssm_scan_workspace_size.restype = ctypes.c_size_t
        L.ssm_scan_workspace_size.argtypes = [ctypes.POINTER(ScanParams)]
        L.causal_conv1d_fwd.restype = st
        L.causal_conv1d_fwd.argtypes = [vp, vp, vp, vp, i, i, i, i, i, i, vp]
        L.ssm_state_update.restype = st
        L.ssm_state_update.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, vp]
        L.ssm_scan_bwd.restype = st
        L.ssm_scan_bwd.argtypes = [ctypes.POINTER(ScanBwdParams), vp]
        L.ssm_scan_bwd_workspace_size.restype = ctypes.c_size_t
        L.ssm_scan_bwd_workspace_size.argtypes = [ctypes.POINTER(ScanBwdParams)]
        L.ssm_state_update_conv.restype = st
        L.ssm_state_update_conv.argtypes = [ctypes.POINTER(StepParams), vp]
        L.ssd_scan_fwd.restype = st
        L.ssd_scan_fwd.argtypes = [ctypes.POINTER(SsdParams), vp]
        L.ssm_device_error.restype = st
        L.ssm_device_error.argtypes = [ctypes.POINTER(ctypes.c_uint)]
        L.ssm_test_withhold_first_copy.restype = None
        L.ssm_test_withhold_first_copy.argtypes = [i]
        L.ssm_last_error.restype = ctypes.c_char_p
        L.ssm_last_error.argtypes = []
        L.ssm_version.restype = ctypes.c_char_p
        L.ssm_version.argtypes = []
        _lib = L
    return _lib


def _check(status: int):
    if status != SSM_OK:
        raise SsmError(status, lib().ssm_last_error().decode())


_DT = {torch.float32: SSM_F32, torch.bfloat16: SSM_BF16}


def _ptr(t: Optional[torch.Tensor], name: str, dtype=None, shape=None) -> Optional[int]:
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    return t.data_ptr()


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _slots_shape(t, name, Bsz, tail, state_indices):
    """Shape check of a tensor that is per batch row, or a slot cache (S, *tail) with state_indices."""
    if t is None:
        return None
    if state_indices is None:
        return (Bsz,) + tuple(tail)
    if t.dim() != 1 + len(tail) or tuple(t.shape[1:]) != tuple(tail):
        raise ValueError(f"{name} must be a slot cache (slots, {', '.join(map(str, tail))})")
    return tuple(t.shape)


CKPT_STEPS = 8  # SSM_CKPT_STEPS: steps between the forward's state checkpoints


def ckpt_count(seqlen: int) -> int:
    """Entries of the checkpoint tensor h_ckpt for a sequence of seqlen steps: ceil(seqlen / 8)."""
    return (seqlen + CKPT_STEPS - 1) // CKPT_STEPS


def _scan_params(u, delta, A, Bm, Cm, Dskip, delta_bias, z, conv_w, conv_b, h0, h_out, y, delta_softplus, zoh,
                 workspace, conv_init=None, conv_final=None, state_indices=None, h_all=None,
                 h_ckpt=None) -> ScanParams:
    if u.dim() != 3:
        raise ValueError("u must be (batch, dim, seqlen)")
    Bsz, D, L = u.shape
    N = A.shape[1]
    idt = u.dtype
    if idt not in _DT:
        raise ValueError(f"unsupported input dtype {idt}")
    p = ScanParams()
    p.batch, p.dim, p.dstate, p.seqlen = Bsz, D, N, L
    p.in_dtype = _DT[idt]
    p.out_dtype = _DT[y.dtype] if y is not None else _DT[idt]
    p.u = _ptr(u, "u", idt)
    p.delta = _ptr(delta, "delta", idt, (Bsz, D, L))
    p.A = _ptr(A, "A", torch.float32, (D, N))
    p.Bm = _ptr(Bm, "Bm", idt, (Bsz, N, L))
    p.Cm = _ptr(Cm, "Cm", idt, (Bsz, N, L))
    p.Dskip = _ptr(Dskip, "Dskip", torch.float32, (D,))
    p.delta_bias = _ptr(delta_bias, "delta_bias", torch.float32, (D,))
    p.z = _ptr(z, "z", idt, (Bsz, D, L))
    if conv_w is not None:
        if conv_w.dim() != 2 or conv_w.shape[0] != D:
            raise ValueError("conv_w must be (dim, width)")
        p.conv_w = _ptr(conv_w, "conv_w", torch.float32)
        p.conv_width = conv_w.shape[1]
        p.conv_b = _ptr(conv_b, "conv_b", torch.float32, (D,))
        W1 = conv_w.shape[1] - 1
        if W1 > 0:
            p.conv_init = _ptr(conv_init, "conv_init", idt, _slots_shape(conv_init, "conv_init", Bsz, (D, W1),
                                                                          state_indices))
            p.conv_final = _ptr(conv_final, "conv_final", idt, _slots_shape(conv_final, "conv_final", Bsz, (D, W1),
                                                                             state_indices))
    p.h0 = _ptr(h0, "h0", torch.float32, _slots_shape(h0, "h0", Bsz, (D, N), state_indices))
    p.h_out = _ptr(h_out, "h_out", torch.float32, _slots_shape(h_out, "h_out", Bsz, (D, N), state_indices))
    p.state_indices = _ptr(state_indices, "state_indices", torch.int32, (Bsz,))
    p.h_all = _ptr(h_all, "h_all", torch.float32, (Bsz, L, D, N))
    p.h_ckpt = _ptr(h_ckpt, "h_ckpt", torch.float32, (Bsz, ckpt_count(L), D, N))
    p.y = _ptr(y, "y", None, (Bsz, D, L)) if y is not None else None
    p.delta_softplus = int(bool(delta_softplus))
    p.zoh = int(bool(zoh))
    if workspace is not None:
        p.workspace = _ptr(workspace, "workspace", torch.uint8)
        p.workspace_bytes = workspace.numel()
    return p


def ssm_scan_workspace_size(u, delta, A, Bm, Cm, **kw) -> int:
    """Bytes of scratch that let ssm_scan_fwd split L for this problem (0 = no split needed)."""
    y = kw.pop("y", None)
    if y is None:
        y = torch.empty_like(u, dtype=kw.pop("out_dtype", None) or u.dtype)
    p = _scan_params(u, delta, A, Bm, Cm, kw.get("Dskip"), kw.get("delta_bias"), kw.get("z"), kw.get("conv_w"),
                     kw.get("conv_b"), kw.get("h0"), kw.get("h_out"), y, kw.get("delta_softplus", True),
                     kw.get("zoh", True), None, kw.get("conv_init"), kw.get("conv_final"), kw.get("state_indices"),
                     kw.get("h_all"), kw.get("h_ckpt"))
    return int(lib().ssm_scan_workspace_size(ctypes.byref(p)))


def ssm_scan_fwd(u: torch.Tensor, delta: torch.Tensor, A: torch.Tensor, Bm: torch.Tensor, Cm: torch.Tensor,
                 Dskip: Optional[torch.Tensor] = None, delta_bias: Optional[torch.Tensor] = None,
                 z: Optional[torch.Tensor] = None, conv_w: Optional[torch.Tensor] = None,
                 conv_b: Optional[torch.Tensor] = None, h0: Optional[torch.Tensor] = None,
                 h_out: Optional[torch.Tensor] = None, y: Optional[torch.Tensor] = None,
                 delta_softplus: bool = True, zoh: bool = True, out_dtype: Optional[torch.dtype] = None,
                 workspace="auto", return_state: bool = False, stream=None,
                 conv_init: Optional[torch.Tensor] = None, conv_final: Optional[torch.Tensor] = None,
                 state_indices: Optional[torch.Tensor] = None, h_all: Optional[torch.Tensor] = None,
                 h_ckpt: Optional[torch.Tensor] = None):
    """Selective scan forward on the GPU.  Layouts as in include/ssm_scan.h: u/delta/z/y (B, D, L),
    Bm/Cm (B, N, L), A (D, N) fp32, Dskip/delta_bias/conv_b (D,) fp32, conv_w (D, W) fp32,
    h0/h_out (B, D, N) fp32, conv_init/conv_final (B, D, W-1) of u's dtype (the conv history before
    and after this call; conv_final may be conv_init).  ``state_indices`` (B,) int32 makes h0, h_out,
    conv_init and conv_final slot caches indexed per batch row (negative: padding row, y = 0);
    ``h_all`` (B, L, D, N) fp32 receives the state after every step; ``h_ckpt`` (B, ckpt_count(L), D, N) fp32
    the state after every 8th step (and after the last), the checkpoints ssm_scan_bwd recomputes from.
    ``workspace``: "auto" (default)
    allocates, through torch's allocator, the scratch that lets the library split L when the (b, d) rows
    alone would leave the GPU idle; a uint8 CUDA tensor of at least ssm_scan_workspace_size bytes; or
    None (no split).  Returns y, or (y, h_out) with return_state."""
    if y is None:
        y = torch.empty(u.shape, dtype=out_dtype or u.dtype, device=u.device)
    if return_state and h_out is None:
        if state_indices is not None:
            raise ValueError("with state_indices, pass the slot cache as h_out")
        h_out = torch.empty((u.shape[0], u.shape[1], A.shape[1]), dtype=torch.float32, device=u.device)
    if isinstance(workspace, str) and workspace == "auto":
        n = ssm_scan_workspace_size(u, delta, A, Bm, Cm, Dskip=Dskip, delta_bias=delta_bias, z=z, conv_w=conv_w,
                                    conv_b=conv_b, h0=h0, h_out=h_out, y=y, delta_softplus=delta_softplus, zoh=zoh,
                                    conv_init=conv_init, conv_final=conv_final, state_indices=state_indices,
                                    h_all=h_all, h_ckpt=h_ckpt)
        workspace = torch.empty(n, dtype=torch.uint8, device=u.device) if n > 0 else None
    p = _scan_params(u, delta, A, Bm, Cm, Dskip, delta_bias, z, conv_w, conv_b, h0, h_out, y, delta_softplus, zoh,
                     workspace, conv_init, conv_final, state_indices, h_all, h_ckpt)
    _check(lib().ssm_scan_fwd(ctypes.byref(p), _stream(stream)))
    return (y, h_out) if return_state else y


def ssm_scan_fwd_static(u: torch.Tensor, delta: torch.Tensor, A: torch.Tensor, Bm: torch.Tensor, Cm: torch.Tensor,
                        Dskip: Optional[torch.Tensor] = None, delta_bias: Optional[torch.Tensor] = None,
                        z: Optional[torch.Tensor] = None, conv_w: Optional[torch.Tensor] = None,
                        conv_b: Optional[torch.Tensor] = None, h0: Optional[torch.Tensor] = None,
                        h_out: Optional[torch.Tensor] = None, y: Optional[torch.Tensor] = None,
                        delta_softplus: bool = True, zoh: bool = True, out_dtype: Optional[torch.dtype] = None,
                        return_state: bool = False, stream=None, conv_init: Optional[torch.Tensor] = None,
                        conv_final: Optional[torch.Tensor] = None, state_indices: Optional[torch.Tensor] = None,
                        h_all: Optional[torch.Tensor] = None):
    """ssm_scan_fwd for callers that cannot allocate scratch: the L split uses the library's fixed
    4 MiB device buffer instead of a workspace.  Calls that may overlap on the GPU share that buffer and
    must be serialised.  Output tensors are allocated here only when not given (pass y / h_out to keep
    the call allocation-free)."""
    if y is None:
        y = torch.empty(u.shape, dtype=out_dtype or u.dtype, device=u.device)
    if return_state and h_out is None:
        h_out = torch.empty((u.shape[0], u.shape[1], A.shape[1]), dtype=torch.float32, device=u.device)
    p = _scan_params(u, delta, A, Bm, Cm, Dskip, delta_bias, z, conv_w, conv_b, h0, h_out, y, delta_softplus, zoh,
                     None, conv_init, conv_final, state_indices, h_all)
    _check(lib().ssm_scan_fwd_static(ctypes.byref(p), _stream(stream)))
    return (y, h_out) if return_state else y


def causal_conv1d_fwd(x: torch.Tensor, w: torch.Tensor, b: Optional[torch.Tensor] = None, silu: bool = True,
                      y: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """Causal depthwise conv1d (+ SiLU) of x (B, D, L) with taps w (D, W) fp32 and bias b (D,) fp32."""
    if x.dim() != 3:
        raise ValueError("x must be (batch, dim, seqlen)")
    Bsz, D, L = x.shape
    if x.dtype not in _DT:
        raise ValueError(f"unsupported dtype {x.dtype}")
    if y is None:
        y = torch.empty_like(x)
    if w.dim() != 2 or w.shape[0] != D:
        raise ValueError("w must be (dim, width)")
    _check(lib().causal_conv1d_fwd(_ptr(x, "x"), _ptr(w, "w", torch.float32), _ptr(b, "b", torch.float32, (D,)),
                                   _ptr(y, "y", x.dtype, (Bsz, D, L)), Bsz, D, L, w.shape[1], int(bool(silu)),
                                   _DT[x.dtype], _stream(stream)))
    return y


def ssm_state_update(state: torch.Tensor, u: torch.Tensor, delta: torch.Tensor, A: torch.Tensor, Bm: torch.Tensor,
                     Cm: torch.Tensor, Dskip: Optional[torch.Tensor] = None,
                     delta_bias: Optional[torch.Tensor] = None, z: Optional[torch.Tensor] = None,
                     y: Optional[torch.Tensor] = None, delta_softplus: bool = True, zoh: bool = True,
                     stream=None, conv_w: Optional[torch.Tensor] = None, conv_b: Optional[torch.Tensor] = None,
                     conv_state: Optional[torch.Tensor] = None,
                     state_indices: Optional[torch.Tensor] = None) -> torch.Tensor:
    """One decode step: state (B, D, N) fp32 updated in place; u/delta/z (B, D), Bm/Cm (B, N).  Returns y (B, D).
    With ``conv_w`` (D, W) fp32 the conv front end is fused (ssm_state_update_conv): u is the conv input x,
    ``conv_state`` (B, D, W-1) of u's dtype holds the previous W-1 inputs and is updated in place.
    With ``state_indices`` (B,) int32, state and conv_state are slot caches (S, D, N), (S, D, W-1) and
    batch row b uses slot state_indices[b] (negative: padding row, y = 0)."""
    _, D, N = state.shape
    Bsz = u.shape[0]
    dt = u.dtype
    if dt not in _DT:
        raise ValueError(f"unsupported dtype {dt}")
    if y is None:
        y = torch.empty_like(u)
    if conv_w is not None or state_indices is not None:
        if conv_w is not None and (conv_w.dim() != 2 or conv_w.shape[0] != D):
            raise ValueError("conv_w must be (dim, width)")
        W = conv_w.shape[1] if conv_w is not None else 1
        p = StepParams()
        p.batch, p.dim, p.dstate, p.dtype = Bsz, D, N, _DT[dt]
        p.state = _ptr(state, "state", torch.float32, _slots_shape(state, "state", Bsz, (D, N), state_indices))
        p.x = _ptr(u, "u", dt, (Bsz, D))
        p.delta = _ptr(delta, "delta", dt, (Bsz, D))
        p.A = _ptr(A, "A", torch.float32, (D, N))
        p.Bm = _ptr(Bm, "Bm", dt, (Bsz, N))
        p.Cm = _ptr(Cm, "Cm", dt, (Bsz, N))
        p.Dskip = _ptr(Dskip, "Dskip", torch.float32, (D,))
        p.delta_bias = _ptr(delta_bias, "delta_bias", torch.float32, (D,))
        p.z = _ptr(z, "z", dt, (Bsz, D))
        p.conv_w = _ptr(conv_w, "conv_w", torch.float32)
        p.conv_b = _ptr(conv_b, "conv_b", torch.float32, (D,)) if conv_w is not None else None
        p.conv_width = W
        p.conv_state = (_ptr(conv_state, "conv_state", dt,
                             _slots_shape(conv_state, "conv_state", Bsz, (D, W - 1), state_indices))
                        if W > 1 else None)
        p.state_indices = _ptr(state_indices, "state_indices", torch.int32, (Bsz,))
        p.y = _ptr(y, "y", dt, (Bsz, D))
        p.delta_softplus = int(bool(delta_softplus))
        p.zoh = int(bool(zoh))
        _check(lib().ssm_state_update_conv(ctypes.byref(p), _stream(stream)))
        return y
    _check(lib().ssm_state_update(_ptr(state, "state", torch.float32, (Bsz, D, N)), _ptr(u, "u", dt, (Bsz, D)),
                                  _ptr(delta, "delta", dt, (Bsz, D)), _ptr(A, "A", torch.float32, (D, N)),
                                  _ptr(Bm, "Bm", dt, (Bsz, N)), _ptr(Cm, "Cm", dt, (Bsz, N)),
                                  _ptr(Dskip, "Dskip", torch.float32, (D,)),
                                  _ptr(delta_bias, "delta_bias", torch.float32, (D,)), _ptr(z, "z", dt, (Bsz, D)),
                                  _ptr(y, "y", dt, (Bsz, D)), Bsz, D, N, int(bool(delta_softplus)), int(bool(zoh)),
                                  _DT[dt], _stream(stream)))
    return y


def ssm_device_error() -> int:
    """Synchronises the current device and returns (and clears) the flags that kernels record when a
    bounded wait runs out: 0 when nothing was recorded, bit 0 for a decode-kernel wait, bit 1 for a scan
    kernel's wait for its staged chunk, bit 2 for an SSD kernel's wait for its copies or products."""
    flags = ctypes.c_uint(0)
    _check(lib().ssm_device_error(ctypes.byref(flags)))
    return int(flags.value)


def ssm_test_withhold_first_copy(on: bool) -> None:
    """Test hook: while on, the packed scan, streamed decode and SSD kernels leave out their first staged
    copy so that their bounded waits run out (see ssm_device_error).  Never for production use."""
    lib().ssm_test_withhold_first_copy(1 if on else 0)


def ssm_scan_bwd(u: torch.Tensor, delta: torch.Tensor, A: torch.Tensor, Bm: torch.Tensor, Cm: torch.Tensor,
                 dy: torch.Tensor, h_ckpt: torch.Tensor, Dskip: Optional[torch.Tensor] = None,
                 delta_bias: Optional[torch.Tensor] = None, z: Optional[torch.Tensor] = None,
                 conv_w: Optional[torch.Tensor] = None, conv_b: Optional[torch.Tensor] = None,
                 conv_init: Optional[torch.Tensor] = None, h0: Optional[torch.Tensor] = None,
                 dh_out: Optional[torch.Tensor] = None, delta_softplus: bool = True, zoh: bool = True,
                 stream=None, workspace="auto") -> dict:
    """Backward pass of ssm_scan_fwd: gradients of sum(y * dy) + sum(h_L * dh_out) for every input, keyed
    like the inputs (``u`` is the gradient of x with a conv; ``h0`` that of the initial state).  ``h_ckpt``
    (B, ckpt_count(L), D, N) fp32 holds the forward call's state checkpoints (ssm_scan_fwd with h_ckpt=...);
    the pass recomputes the other states from them.
    ``workspace``: "auto" (allocated here when the L split pays), None (no split) or a uint8 tensor."""
    if u.dim() != 3:
        raise ValueError("u must be (batch, dim, seqlen)")
    Bsz, D, L = u.shape
    N = A.shape[1]
    idt = u.dtype
    if idt not in _DT:
        raise ValueError(f"unsupported dtype {idt}")
    dev = u.device
    g = {
        "u": torch.empty_like(u), "delta": torch.empty_like(u), "z": torch.empty_like(u) if z is not None else None,
        "A": torch.empty((D, N), dtype=torch.float32, device=dev),
        "Bm": torch.empty((Bsz, N, L), dtype=torch.float32, device=dev),
        "Cm": torch.empty((Bsz, N, L), dtype=torch.float32, device=dev),
        "Dskip": torch.empty(D, dtype=torch.float32, device=dev) if Dskip is not None else None,
        "delta_bias": torch.empty(D, dtype=torch.float32, device=dev) if delta_bias is not None else None,
        "conv_w": torch.empty_like(conv_w) if conv_w is not None else None,
        "conv_b": torch.empty(D, dtype=torch.float32, device=dev) if (conv_w is not None and conv_b is not None)
        else None,
        "conv_init": (torch.empty((Bsz, D, conv_w.shape[1] - 1), dtype=idt, device=dev)
                      if (conv_w is not None and conv_w.shape[1] > 1) else None),
        "h0": torch.empty((Bsz, D, N), dtype=torch.float32, device=dev),
    }
    p = ScanBwdParams()
    p.batch, p.dim, p.dstate, p.seqlen = Bsz, D, N, L
    p.in_dtype = _DT[idt]
    p.u = _ptr(u, "u", idt)
    p.delta = _ptr(delta, "delta", idt, (Bsz, D, L))
    p.A = _ptr(A, "A", torch.float32, (D, N))
    p.Bm = _ptr(Bm, "Bm", idt, (Bsz, N, L))
    p.Cm = _ptr(Cm, "Cm", idt, (Bsz, N, L))
    p.Dskip = _ptr(Dskip, "Dskip", torch.float32, (D,))
    p.delta_bias = _ptr(delta_bias, "delta_bias", torch.float32, (D,))
    p.z = _ptr(z, "z", idt, (Bsz, D, L))
    if conv_w is not None:
        p.conv_w = _ptr(conv_w, "conv_w", torch.float32)
        p.conv_b = _ptr(conv_b, "conv_b", torch.float32, (D,))
        p.conv_width = conv_w.shape[1]
        if conv_w.shape[1] > 1:
            p.conv_init = _ptr(conv_init, "conv_init", idt, (Bsz, D, conv_w.shape[1] - 1))
    p.h0 = _ptr(h0, "h0", torch.float32, (Bsz, D, N))
    p.delta_softplus = int(bool(delta_softplus))
    p.zoh = int(bool(zoh))
    p.h_ckpt = _ptr(h_ckpt, "h_ckpt", torch.float32, (Bsz, ckpt_count(L), D, N))
    p.dy = _ptr(dy, "dy", idt, (Bsz, D, L))
    p.dh_out = _ptr(dh_out, "dh_out", torch.float32, (Bsz, D, N))
    p.du, p.ddelta, p.dz = _ptr(g["u"], "du"), _ptr(g["delta"], "ddelta"), _ptr(g["z"], "dz")
    p.dA, p.dB, p.dC = _ptr(g["A"], "dA"), _ptr(g["Bm"], "dB"), _ptr(g["Cm"], "dC")
    p.dDskip, p.ddelta_bias = _ptr(g["Dskip"], "dDskip"), _ptr(g["delta_bias"], "ddelta_bias")
    p.dconv_w, p.dconv_b = _ptr(g["conv_w"], "dconv_w"), _ptr(g["conv_b"], "dconv_b")
    p.dconv_init, p.dh0 = _ptr(g["conv_init"], "dconv_init"), _ptr(g["h0"], "dh0")
    if isinstance(workspace, str) and workspace == "auto":
        n = int(lib().ssm_scan_bwd_workspace_size(ctypes.byref(p)))
        workspace = torch.empty(n, dtype=torch.uint8, device=dev) if n > 0 else None
    if workspace is not None:
        p.workspace = _ptr(workspace, "workspace", torch.uint8)
        p.workspace_bytes = workspace.numel()
    _check(lib().ssm_scan_bwd(ctypes.byref(p), _stream(stream)))
    return {k: v for k, v in g.items() if v is not None}


class SsdParams(ctypes.Structure):
    """Mirror of ``ssd_scan_params`` in include/ssm_scan.h."""
    _fields_ = [("batch", ctypes.c_int), ("nheads", ctypes.c_int), ("headdim", ctypes.c_int),
                ("ngroups", ctypes.c_int), ("dstate", ctypes.c_int), ("seqlen", ctypes.c_int),
                ("x", ctypes.c_void_p), ("dt", ctypes.c_void_p), ("A", ctypes.c_void_p), ("Bm", ctypes.c_void_p),
                ("Cm", ctypes.c_void_p), ("Dskip", ctypes.c_void_p), ("dt_bias", ctypes.c_void_p),
                ("z", ctypes.c_void_p), ("h0", ctypes.c_void_p), ("h_out", ctypes.c_void_p), ("y", ctypes.c_void_p),
                ("delta_softplus", ctypes.c_int), ("zoh", ctypes.c_int)]


def ssd_scan_fwd(x: torch.Tensor, dt: torch.Tensor, A: torch.Tensor, Bm: torch.Tensor, Cm: torch.Tensor, *,
                 nheads: int, ngroups: int = 1, Dskip: Optional[torch.Tensor] = None,
                 dt_bias: Optional[torch.Tensor] = None, z: Optional[torch.Tensor] = None,
                 h0: Optional[torch.Tensor] = None, return_state: bool = False, h_out: Optional[torch.Tensor] = None,
                 y: Optional[torch.Tensor] = None, delta_softplus: bool = True, zoh: bool = False, stream=None):
    """Mamba-2 (SSD) layer scan: x, z (B, H*P, L) bf16; dt (B, H, L) bf16; A, Dskip, dt_bias (H,) fp32;
    Bm, Cm (B, G, L, N) bf16; h0 / h_out (B, H, P, N) fp32.  Returns y (and the final state with
    ``return_state``).  Head h reads group h // (H / G)."""
    if x.dim() != 3:
        raise ValueError("x must be (batch, nheads * headdim, seqlen)")
    Bsz, D, L = x.shape
    H, G = int(nheads), int(ngroups)
    if H <= 0 or G <= 0 or D % H:
        raise ValueError("x's channel count must be a multiple of nheads")
    P = D // H
    if Bm.dim() != 4:
        raise ValueError("Bm must be (batch, ngroups, seqlen, dstate)")
    N = Bm.shape[3]
    bf = torch.bfloat16
    if y is None:
        y = torch.empty_like(x)
    if return_state and h_out is None:
        h_out = torch.empty((Bsz, H, P, N), dtype=torch.float32, device=x.device)
    p = SsdParams()
    p.batch, p.nheads, p.headdim, p.ngroups, p.dstate, p.seqlen = Bsz, H, P, G, N, L
    p.x = _ptr(x, "x", bf)
    p.dt = _ptr(dt, "dt", bf, (Bsz, H, L))
    p.A = _ptr(A, "A", torch.float32, (H,))
    p.Bm = _ptr(Bm, "Bm", bf, (Bsz, G, L, N))
    p.Cm = _ptr(Cm, "Cm", bf, (Bsz, G, L, N))
    p.Dskip = _ptr(Dskip, "Dskip", torch.float32, (H,))
    p.dt_bias = _ptr(dt_bias, "dt_bias", torch.float32, (H,))
    p.z = _ptr(z, "z", bf, (Bsz, D, L))
    p.h0 = _ptr(h0, "h0", torch.float32, (Bsz, H, P, N))
    p.h_out = _ptr(h_out, "h_out", torch.float32, (Bsz, H, P, N))
    p.y = _ptr(y, "y", bf, (Bsz, D, L))
    p.delta_softplus = int(bool(delta_softplus))
    p.zoh = int(bool(zoh))
    _check(lib().ssd_scan_fwd(ctypes.byref(p), _stream(stream)))
    return (y, h_out) if return_state else y
