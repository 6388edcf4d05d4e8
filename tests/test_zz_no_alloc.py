"""ssm_scan_fwd_static: the scan entry point for callers that cannot allocate device memory (a runtime
that plans every buffer at start-up, code in a stream callback, latency-critical paths where an
allocation may synchronise the device).  It takes the scratch of the L split from a fixed 4 MiB buffer
inside the library instead of a caller workspace.

Checked through the C ABI against ssm_scan_fwd with a workspace and against the fp64 oracle element by
element, on two calls in a row (the buffer keeps the previous call's contents), on two problems of
different shapes, and for the rejection of a problem whose split needs more than the buffer.  Collected last so that a run stopping at its first failure has
run every other test first; it also passes on its own in a fresh process."""
import numpy as np
import pytest
import torch

import oracle
import selective_state_space_156_b300 as ssm
import workloads
from gpu_helpers import assert_close, h_tolerance, to_dev, y_tolerance

pytestmark = pytest.mark.gpu

STATIC_BYTES = 4 << 20


def _args(g):
    return dict(Dskip=g.get("Dskip"), delta_bias=g.get("delta_bias"), z=g.get("z"), conv_w=g.get("conv_w"),
                conv_b=g.get("conv_b"), delta_softplus=g.get("delta_softplus", True), zoh=g.get("zoh", True))


@pytest.mark.parametrize("case", ["bf16_split_with_h0", "f32_split_without_h0"])
def test_static_scratch_matches_workspace_entry_point_twice(case):
    if case == "bf16_split_with_h0":
        d = workloads.make_scan_inputs(workloads.SCAN_CONFIGS["long2.8b"], batch=1, dim=200, seqlen=6144,
                                       with_h0=True)
    else:
        d = workloads.make_scan_inputs(workloads.SCAN_CONFIGS["tiny"], batch=2, dim=64, seqlen=4096, dstate=8)
    g = to_dev(d)
    kw = _args(g)
    need = ssm.ssm_scan_workspace_size(g["u"], g["delta"], g["A"], g["Bm"], g["Cm"], h0=g.get("h0"), **kw)
    assert 0 < need <= STATIC_BYTES, "the case must take the L split and fit the static buffer"

    h0 = g.get("h0")
    y_ref, h_ref = ssm.ssm_scan_fwd(g["u"], g["delta"], g["A"], g["Bm"], g["Cm"], h0=h0, workspace="auto",
                                    return_state=True, **kw)
    torch.cuda.synchronize()
    yr = y_ref.double().cpu().numpy()
    hr = h_ref.double().cpu().numpy()
    yo, ho, _ = oracle.scan(d)
    yo = yo.reshape(yr.shape)
    ho = ho.reshape(hr.shape)
    y = torch.empty_like(y_ref)
    h = torch.empty_like(h_ref)
    for call in range(2):
        y.fill_(float("nan"))
        h.fill_(float("nan"))
        ssm.ssm_scan_fwd_static(g["u"], g["delta"], g["A"], g["Bm"], g["Cm"], h0=h0, h_out=h, y=y, **kw)
        torch.cuda.synchronize()
        assert_close(y, yr, y_tolerance(yr, y.dtype), f"y, call {call}")
        assert_close(h, hr, h_tolerance(hr, g["u"].dtype), f"h_out, call {call}")
        assert_close(y, yo, y_tolerance(yo, y.dtype), f"y against the oracle, call {call}")
        assert_close(h, ho, h_tolerance(ho, g["u"].dtype), f"h_out against the oracle, call {call}")


def test_static_scratch_rejects_a_split_beyond_the_buffer():
    # 8288 channels with N = 64: the split plan needs about 6.5 MB of scratch
    d = workloads.make_scan_inputs(workloads.SCAN_CONFIGS["mamba130m"], batch=1, dim=8288, seqlen=2048, dstate=64)
    g = to_dev(d)
    kw = _args(g)
    need = ssm.ssm_scan_workspace_size(g["u"], g["delta"], g["A"], g["Bm"], g["Cm"], **kw)
    assert need > STATIC_BYTES
    y = torch.full_like(g["u"], float("nan"))
    with pytest.raises(ssm.SsmError) as err:
        ssm.ssm_scan_fwd_static(g["u"], g["delta"], g["A"], g["Bm"], g["Cm"], y=y, **kw)
    assert err.value.status == ssm.SSM_ERR_UNSUPPORTED
    assert "static" in str(err.value)
    torch.cuda.synchronize()
    assert bool(torch.isnan(y.float()).all()), "a rejected call must launch nothing"
