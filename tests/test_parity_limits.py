"""Edge sizes through the C ABI against the oracle: the largest batch the boundary accepts (65535, the
grid's y extent), a single channel, a single step, one state; each on the kernel its shape selects."""
import pytest
import torch

import oracle
import selective_state_space_156_b300 as ssm
import workloads
from gpu_helpers import assert_close, h_tolerance, to_dev, y_tolerance

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("dt,B,D,N,L", [
    ("bf16", 65535, 2, 4, 8),    # packed kernel, largest batch
    ("f32", 65535, 1, 1, 3),     # element-wise kernel, largest batch, one channel, one state
    ("bf16", 1, 1, 16, 4096),    # one channel, long: the L split over a single row
    ("bf16", 3, 128, 16, 8),     # a single 8-step group per row
    ("f32", 2, 33, 7, 1),        # a single step
])
def test_scan_at_edge_sizes(dt, B, D, N, L):
    d = workloads.make_scan_inputs(workloads.SCAN_CONFIGS["mamba1.4b_conv"], batch=B, dim=D, seqlen=L, dstate=N,
                                   dtype=dt, with_h0=True, seed=9500 + B + D + N + L)
    g = to_dev(d)
    y, h = ssm.ssm_scan_fwd(g["u"], g["delta"], g["A"], g["Bm"], g["Cm"], h0=g["h0"], Dskip=g["Dskip"],
                            delta_bias=g["delta_bias"], z=g["z"], conv_w=g["conv_w"], conv_b=g["conv_b"],
                            workspace="auto", return_state=True)
    assert ssm.ssm_device_error() == 0
    y_ref, h_ref, _ = oracle.scan(d)
    y_ref = y_ref.reshape(B, D, L)
    h_ref = h_ref.reshape(B, D, N)
    assert_close(y, y_ref, y_tolerance(y_ref, y.dtype), "y")
    assert_close(h, h_ref, h_tolerance(h_ref, g["u"].dtype), "h_out")


@pytest.mark.parametrize("B,D,N", [(65535, 8, 16), (65535, 3, 5), (1, 8, 8)])
def test_decode_at_edge_sizes(B, D, N):
    """(65535, 8, 16): the streamed kernel over 65535 one-tile rows; (65535, 3, 5): the row kernel."""
    gen = torch.Generator().manual_seed(9600 + B + D + N)
    s = {
        "state": torch.randn((B, D, N), generator=gen) * 0.5,
        "u": torch.randn((B, D), generator=gen).to(torch.bfloat16),
        "delta": (torch.randn((B, D), generator=gen) * 0.5).to(torch.bfloat16),
        "A": -torch.arange(1, N + 1, dtype=torch.float32).repeat(D, 1),
        "Bm": torch.randn((B, N), generator=gen).to(torch.bfloat16),
        "Cm": torch.randn((B, N), generator=gen).to(torch.bfloat16),
        "Dskip": torch.randn(D, generator=gen),
        "delta_bias": torch.log(torch.expm1(1e-3 + 0.099 * torch.rand(D, generator=gen))),
        "z": torch.randn((B, D), generator=gen).to(torch.bfloat16),
    }
    g = to_dev(s)
    st = g["state"].clone()
    y = ssm.ssm_state_update(st, g["u"], g["delta"], g["A"], g["Bm"], g["Cm"], Dskip=g["Dskip"],
                             delta_bias=g["delta_bias"], z=g["z"])
    assert ssm.ssm_device_error() == 0
    st_ref, y_ref = oracle.state_update(s["state"], s["u"], s["delta"], s["A"], s["Bm"], s["Cm"], s["Dskip"],
                                        s["delta_bias"], s["z"])
    assert_close(y, y_ref, y_tolerance(y_ref, torch.bfloat16), "y")
    assert_close(st, st_ref, h_tolerance(st_ref, torch.bfloat16), "state")
