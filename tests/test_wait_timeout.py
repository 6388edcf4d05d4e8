"""The bounded waits, made to run out on a GPU: with the library's test hook ssm_test_withhold_first_copy on, the
packed scan (its TMA-staged pass), the streamed decode kernel and the SSD kernel leave out their first copy,
so that the waits for it give up after about a second.  Nothing faults or hangs: the kernel records the failure, lets its other copies and
products end, frees its tensor memory and returns; ssm_device_error reports the bit and clears it, and
the same call without the switch is then correct, so the context stayed usable."""
import numpy as np
import pytest
import torch

import oracle
import selective_state_space_156_b300 as ssm
import workloads
from gpu_helpers import assert_close, h_tolerance, to_dev, y_tolerance
from oracle.ssd import ssd_scan

pytestmark = pytest.mark.gpu

def _withheld(call):
    assert ssm.ssm_device_error() == 0
    ssm.ssm_test_withhold_first_copy(True)
    try:
        call()
        flags = ssm.ssm_device_error()   # synchronises the device
    finally:
        ssm.ssm_test_withhold_first_copy(False)
    return flags


def test_scan_wait_runs_out_and_is_reported():
    d = workloads.make_scan_inputs(workloads.SCAN_CONFIGS["mamba1.4b_conv"], batch=2, dim=256, seqlen=304,
                                   with_h0=True)
    g = to_dev(d)

    def run():
        return ssm.ssm_scan_fwd(g["u"], g["delta"], g["A"], g["Bm"], g["Cm"], Dskip=g["Dskip"],
                                delta_bias=g["delta_bias"], z=g["z"], conv_w=g["conv_w"], conv_b=g["conv_b"],
                                h0=g["h0"], return_state=True, workspace=None)

    flags = _withheld(run)
    assert flags & 2, f"scan timeout not reported (flags {flags})"
    y, h = run()
    torch.cuda.synchronize()
    assert ssm.ssm_device_error() == 0
    ref_y, ref_h, _ = oracle.scan(d)
    ref_y = ref_y.reshape(y.shape)
    assert_close(y, ref_y, y_tolerance(ref_y, torch.bfloat16), "scan y after the timeout")
    assert_close(h, ref_h.reshape(h.shape), h_tolerance(ref_h.reshape(h.shape), torch.bfloat16),
                 "scan state after the timeout")


def test_decode_wait_runs_out_and_is_reported():
    cfg = workloads.DECODE_CONFIG
    layer = workloads.make_decode_layer(cfg, 0, batch=4)
    pool = workloads.make_decode_pool(cfg, 1, batch=4)
    g = {k: v.cuda() for k, v in layer.items()}
    x = {k: v[0].cuda().contiguous() for k, v in pool.items()}

    def step(state):
        return ssm.ssm_state_update(state, x["u"], x["delta"], g["A"], x["Bm"], x["Cm"], Dskip=g["Dskip"],
                                    delta_bias=g["delta_bias"], z=x["z"])

    flags = _withheld(lambda: step(g["state"].clone()))
    assert flags & 1, f"decode timeout not reported (flags {flags})"
    st = g["state"].clone()
    y = step(st)
    torch.cuda.synchronize()
    assert ssm.ssm_device_error() == 0
    st_ref, y_ref = oracle.state_update(layer["state"], pool["u"][0], pool["delta"][0], layer["A"], pool["Bm"][0],
                                        pool["Cm"][0], layer["Dskip"], layer["delta_bias"], pool["z"][0])
    assert_close(y, y_ref, y_tolerance(y_ref, torch.bfloat16), "decode y after the timeout")
    assert_close(st, st_ref, h_tolerance(st_ref, torch.bfloat16), "decode state after the timeout")


def test_ssd_wait_runs_out_and_is_reported():
    d = workloads.make_ssd_inputs(workloads.SSD_CONFIGS["ssd_small"], batch=1, nheads=2, ngroups=1, seqlen=256,
                                  with_h0=True)
    g = to_dev(d)

    def run():
        return ssm.ssd_scan_fwd(g["x"], g["dt"], g["A"], g["Bm"], g["Cm"], nheads=2, ngroups=1, Dskip=g["Dskip"],
                                dt_bias=g["dt_bias"], z=g["z"], h0=g["h0"], return_state=True)

    flags = _withheld(run)
    assert flags & 4, f"SSD timeout not reported (flags {flags})"
    y, h = run()
    torch.cuda.synchronize()
    assert ssm.ssm_device_error() == 0
    ref_y, ref_h, _ = ssd_scan(d)
    ref_y = ref_y.reshape(y.shape)
    assert_close(y, ref_y, y_tolerance(ref_y, torch.bfloat16), "SSD y after the timeout")
    assert_close(h, ref_h.reshape(h.shape), h_tolerance(ref_h.reshape(h.shape), torch.bfloat16),
                 "SSD state after the timeout")
