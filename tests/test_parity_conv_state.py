"""Parity of the conv history carried across calls, through the C ABI, against the oracle.

ssm_scan_fwd with conv_init / conv_final (a chunked prefill carries the last W-1 conv inputs from one
call to the next, dpshk.com/news/5205047 section 1.3) on each kernel path: the packed bf16 kernel
(N <= 16), the lane-group kernel (N = 32, 64) and the element-wise kernel (fp32, ragged L); with and
without the L split.  ssm_state_update with the conv front end fused (the decode cache holds a conv
state beside the SSM state, lshu.cn/news/79586 section 6.5) on the streamed kernel (D % 8 == 0) and the
row kernel, and a run of decode steps against one fused scan."""
import numpy as np
import pytest
import torch

import oracle
import selective_state_space_156_b300 as ssm
import workloads
from gpu_helpers import Guarded, assert_close, h_tolerance, to_dev, y_tolerance

pytestmark = pytest.mark.gpu


def _inputs(Bsz, D, N, L, W, dtype, seed, h0=True):
    cfg = workloads.SCAN_CONFIGS["mamba1.4b_conv"]
    d = workloads.make_scan_inputs(cfg, batch=Bsz, dim=D, seqlen=L, dstate=N, dtype=dtype, with_h0=h0, seed=seed)
    d["conv_w"] = d["conv_w"][:, :W].contiguous()
    g = torch.Generator().manual_seed(seed + 1)
    d["conv_init"] = torch.randn((Bsz, D, W - 1), generator=g).to(d["u"].dtype) if W > 1 else None
    return d


def _kw(g):
    return dict(Dskip=g["Dskip"], delta_bias=g["delta_bias"], z=g["z"], conv_w=g["conv_w"], conv_b=g["conv_b"])


@pytest.mark.parametrize("W", [2, 3, 4])
@pytest.mark.parametrize("case", [
    ("bf16", 16, 2, 128, 96),     # packed bf16 kernel
    ("bf16", 64, 2, 64, 96),      # lane-group kernel
    ("f32", 16, 2, 64, 61),       # element-wise kernel, ragged L
    ("bf16", 16, 1, 64, 8192),    # packed kernel with the L split
    ("f32", 8, 1, 32, 4099),      # element-wise kernel with the L split
])
def test_scan_with_conv_history_matches_oracle(W, case):
    dt, N, Bsz, D, L = case
    d = _inputs(Bsz, D, N, L, W, dt, seed=3000 + W + N + L)
    g = to_dev(d)
    fin = Guarded((Bsz, D, W - 1), g["u"].dtype)
    # output in the input dtype: bf16 in and out is what the packed and lane-group kernels take
    y, h = ssm.ssm_scan_fwd(g["u"], g["delta"], g["A"], g["Bm"], g["Cm"], h0=g["h0"], workspace="auto",
                            return_state=True, conv_init=g["conv_init"], conv_final=fin.t, **_kw(g))
    torch.cuda.synchronize()
    fin.check_bands()
    extra = {}
    y_ref, h_ref, _ = oracle.scan(d, extra=extra)
    y_ref = y_ref.reshape(Bsz, D, L)
    h_ref = h_ref.reshape(Bsz, D, N)
    assert_close(y, y_ref, y_tolerance(y_ref, y.dtype), "y")
    assert_close(h, h_ref, h_tolerance(h_ref, g["u"].dtype), "h_out")
    assert torch.equal(fin.t.cpu().double(), torch.tensor(extra["conv_final"]).reshape(Bsz, D, W - 1)), "conv_final"


@pytest.mark.parametrize("dt,N,L,cuts", [
    ("bf16", 16, 256, [64, 200]),
    ("bf16", 32, 256, [128, 136]),
    ("f32", 16, 101, [1, 2, 50]),      # calls shorter than the history
])
def test_chunked_prefill_with_history_in_place_equals_one_call(dt, N, L, cuts):
    """Calls over consecutive pieces of the sequence, each taking the history and state of the one before
    (conv_final written over its own conv_init), reproduce one call over the whole sequence."""
    Bsz, D, W = 2, 64, 4
    d = _inputs(Bsz, D, N, L, W, dt, seed=4000 + N + L, h0=False)
    g = to_dev(d)
    kw = _kw(g)
    y_one, h_one = ssm.ssm_scan_fwd(g["u"], g["delta"], g["A"], g["Bm"], g["Cm"], return_state=True, **kw)
    hist = torch.zeros((Bsz, D, W - 1), dtype=g["u"].dtype, device="cuda")
    h = torch.zeros((Bsz, D, N), dtype=torch.float32, device="cuda")
    ys = []
    edges = [0] + cuts + [L]
    for a, b in zip(edges[:-1], edges[1:]):
        piece = {k: g[k][..., a:b].contiguous() for k in ("u", "delta", "z", "Bm", "Cm")}
        yp = ssm.ssm_scan_fwd(piece["u"], piece["delta"], g["A"], piece["Bm"], piece["Cm"], h0=h, h_out=h,
                              conv_init=hist, conv_final=hist, **dict(kw, z=piece["z"]))
        ys.append(yp)
    torch.cuda.synchronize()
    y_cat = torch.cat(ys, dim=-1)
    # the pieces run the same per-step arithmetic as the one call; only the rounding of y to bf16 of
    # values that differ in the last fp32 bits could separate them
    tol = 2e-5 if dt == "f32" else 8e-3
    torch.testing.assert_close(y_cat.float(), y_one.float(), rtol=tol, atol=tol)
    torch.testing.assert_close(h, h_one, rtol=2e-5, atol=2e-5)
    assert torch.equal(hist, g["u"][..., -(W - 1):])


@pytest.mark.parametrize("W", [1, 2, 3, 4])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("shape", [(3, 64, 16), (5, 200, 8), (2, 150, 16), (4, 64, 64)])
def test_decode_step_with_conv_state(W, dtype, shape):
    """(3, 64, 16), (5, 200, 8), (4, 64, 64): the streamed kernel; (2, 150, 16): the row kernel."""
    Bsz, D, N = shape
    gen = torch.Generator().manual_seed(5000 + W + D + N)
    s = {
        "state": torch.randn((Bsz, D, N), generator=gen) * 0.5,
        "x": torch.randn((Bsz, D), generator=gen).to(dtype),
        "delta": (torch.randn((Bsz, D), generator=gen) * 0.5).to(dtype),
        "A": -torch.arange(1, N + 1, dtype=torch.float32).repeat(D, 1),
        "Bm": torch.randn((Bsz, N), generator=gen).to(dtype),
        "Cm": torch.randn((Bsz, N), generator=gen).to(dtype),
        "Dskip": torch.randn(D, generator=gen),
        "delta_bias": torch.log(torch.expm1(1e-3 + 0.099 * torch.rand(D, generator=gen))),
        "z": torch.randn((Bsz, D), generator=gen).to(dtype),
        "conv_w": torch.randn((D, W), generator=gen) * 0.5,
        "conv_b": torch.randn(D, generator=gen) * 0.1,
        "conv_state": torch.randn((Bsz, D, max(W - 1, 1)), generator=gen).to(dtype)[..., :W - 1].contiguous(),
    }
    g = to_dev(s)
    st = g["state"].clone()
    cs = g["conv_state"].clone()
    y = Guarded((Bsz, D), dtype)
    ssm.ssm_state_update(st, g["x"], g["delta"], g["A"], g["Bm"], g["Cm"], Dskip=g["Dskip"],
                         delta_bias=g["delta_bias"], z=g["z"], y=y.t, conv_w=g["conv_w"], conv_b=g["conv_b"],
                         conv_state=cs if W > 1 else None)
    assert ssm.ssm_device_error() == 0
    y.check_bands()
    st_ref, y_ref, cs_ref = oracle.state_update(s["state"], s["x"], s["delta"], s["A"], s["Bm"], s["Cm"], s["Dskip"],
                                                s["delta_bias"], s["z"], conv_w=s["conv_w"], conv_b=s["conv_b"],
                                                conv_state=s["conv_state"] if W > 1 else None)
    assert_close(y.t, y_ref, y_tolerance(y_ref, dtype), "y")
    assert_close(st, st_ref, h_tolerance(st_ref, dtype), "state")
    if W > 1:
        assert torch.equal(cs.cpu().double(), torch.tensor(np.ascontiguousarray(cs_ref))), "conv state"


@pytest.mark.parametrize("D", [256, 100])
def test_decode_steps_with_conv_equal_one_fused_scan(D):
    """128 fused decode steps (conv state + SSM state carried) against one fused scan of length 128, both on
    the GPU and both against the oracle; D = 256 takes the streamed kernel, D = 100 the row kernel."""
    Bsz, N, L, W = 4, 16, 128, 4
    d = _inputs(Bsz, D, N, L, W, "bf16", seed=6000 + D)
    g = to_dev(d)
    kw = _kw(g)
    y_scan, h_scan = ssm.ssm_scan_fwd(g["u"], g["delta"], g["A"], g["Bm"], g["Cm"], h0=g["h0"], return_state=True,
                                      conv_init=g["conv_init"], out_dtype=torch.float32, **kw)
    st = g["h0"].clone()
    cs = g["conv_init"].clone()
    ys = []
    for t in range(L):
        ys.append(ssm.ssm_state_update(st, g["u"][..., t].contiguous(), g["delta"][..., t].contiguous(), g["A"],
                                       g["Bm"][..., t].contiguous(), g["Cm"][..., t].contiguous(), Dskip=g["Dskip"],
                                       delta_bias=g["delta_bias"], z=g["z"][..., t].contiguous(),
                                       conv_w=g["conv_w"], conv_b=g["conv_b"], conv_state=cs,
                                       y=torch.empty((Bsz, D), dtype=torch.bfloat16, device="cuda")))
    assert ssm.ssm_device_error() == 0
    y_dec = torch.stack(ys, dim=-1).float()
    y_ref, h_ref, _ = oracle.scan(d)
    y_ref = y_ref.reshape(Bsz, D, L)
    assert_close(y_dec, y_ref, y_tolerance(y_ref, torch.bfloat16), "decode y")
    assert_close(y_scan, y_ref, y_tolerance(y_ref, torch.bfloat16), "scan y")
    h_ref = h_ref.reshape(Bsz, D, N)
    assert_close(st, h_ref, h_tolerance(h_ref, torch.bfloat16), "decode state")
    torch.testing.assert_close(st, h_scan, rtol=1e-3, atol=1e-4)
    assert torch.equal(cs, g["u"][..., -(W - 1):])
