"""GPU parity of causal_conv1d_fwd and ssm_state_update (through the C ABI) against the fp64 oracle,
plus the decode workload at full size (256 x 5120 x 16 state per layer, 64 layers, 128 tokens) checked
on sampled layers and batch rows over every step."""
import numpy as np
import pytest
import torch

import oracle
import selective_state_space_156_b300 as ssm
import workloads
from gpu_helpers import Guarded, assert_close, h_tolerance, sample_rows, to_dev, y_tolerance

pytestmark = pytest.mark.gpu


# ------------------------------------------------------------------------------------------------
# causal conv1d
# ------------------------------------------------------------------------------------------------
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("width", [1, 2, 3, 4])
@pytest.mark.parametrize("silu", [True, False])
@pytest.mark.parametrize("L", [1, 5, 64, 600, 1027])
def test_conv1d(dtype, width, silu, L):
    g = torch.Generator().manual_seed(width * 1000 + L)
    x = torch.randn((2, 70, L), generator=g).to(dtype)
    w = torch.randn((70, width), generator=g) * 0.5
    b = torch.randn(70, generator=g) * 0.1
    out = Guarded((2, 70, L), dtype)
    ssm.causal_conv1d_fwd(x.cuda(), w.cuda(), b.cuda(), silu=silu, y=out.t)
    torch.cuda.synchronize()
    out.check_bands()
    ref = oracle.conv1d(x, w, b, silu=silu).reshape(2, 70, L)
    assert_close(out.t, ref, y_tolerance(ref, dtype), "conv y")


def test_conv1d_no_bias_unaligned():
    x = torch.randn((1, 33, 41))
    w = torch.randn((33, 4)) * 0.5
    xd = torch.empty(x.numel() + 1, device="cuda")[1:].view(x.shape)
    xd.copy_(x)
    y = ssm.causal_conv1d_fwd(xd, w.cuda(), None, silu=True)
    ref = oracle.conv1d(x, w, None, silu=True).reshape(x.shape)
    assert_close(y, ref, y_tolerance(ref, torch.float32), "conv y")


def test_conv1d_full_size_sampled():
    cfg = workloads.SCAN_CONFIGS["mamba1.4b_conv"]
    d = workloads.make_scan_inputs(cfg)
    y = ssm.causal_conv1d_fwd(d["u"].cuda(), d["conv_w"].cuda(), d["conv_b"].cuda(), silu=True)
    torch.cuda.synchronize()
    rows = sample_rows(cfg.batch, cfg.dim, 128, 7)
    ref = oracle.conv1d(d["u"], d["conv_w"], d["conv_b"], silu=True, rows=rows)
    bi = torch.tensor([r[0] for r in rows], device="cuda")
    di = torch.tensor([r[1] for r in rows], device="cuda")
    assert_close(y[bi, di], ref, y_tolerance(ref, torch.bfloat16), "conv y (sampled rows)")


# ------------------------------------------------------------------------------------------------
# single-token state update
# ------------------------------------------------------------------------------------------------
def _step_inputs(Bsz, D, N, dtype, seed, with_z=True, with_D=True):
    g = torch.Generator().manual_seed(seed)
    return {
        "state": torch.randn((Bsz, D, N), generator=g) * 0.5,
        "u": torch.randn((Bsz, D), generator=g).to(dtype),
        "delta": (torch.randn((Bsz, D), generator=g) * 0.5).to(dtype),
        "A": -torch.arange(1, N + 1, dtype=torch.float32).repeat(D, 1) * (0.5 + torch.rand((D, 1), generator=g)),
        "Bm": torch.randn((Bsz, N), generator=g).to(dtype),
        "Cm": torch.randn((Bsz, N), generator=g).to(dtype),
        "Dskip": torch.randn(D, generator=g) if with_D else None,
        "delta_bias": torch.log(torch.expm1(1e-3 + 0.099 * torch.rand(D, generator=g))),
        "z": torch.randn((Bsz, D), generator=g).to(dtype) if with_z else None,
    }


@pytest.mark.parametrize("N", [1, 3, 4, 8, 16, 32, 64])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("zoh", [True, False])
def test_state_update(N, dtype, zoh):
    s = _step_inputs(3, 150, N, dtype, N * 7 + int(zoh))
    g = to_dev(s)
    st = g["state"].clone()
    y = Guarded((3, 150), dtype)
    ssm.ssm_state_update(st, g["u"], g["delta"], g["A"], g["Bm"], g["Cm"], Dskip=g["Dskip"],
                         delta_bias=g["delta_bias"], z=g["z"], y=y.t, zoh=zoh)
    torch.cuda.synchronize()
    y.check_bands()
    st_ref, y_ref = oracle.state_update(s["state"], s["u"], s["delta"], s["A"], s["Bm"], s["Cm"], s["Dskip"],
                                        s["delta_bias"], s["z"], zoh=zoh)
    assert_close(y.t, y_ref, y_tolerance(y_ref, dtype), "y")
    assert_close(st, st_ref, h_tolerance(st_ref, torch.float32), "state")


@pytest.mark.parametrize("N", [8, 16, 32, 64])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("shape", [(2, 8), (5, 200), (128, 3584)])
def test_state_update_streamed(N, dtype, shape):
    """The streamed (bulk-copy) decode kernel: D % 8 == 0 and aligned tensors.  (5, 200) ends every batch
    row with a partial tile of 8 rows; (128, 3584) gives every block more tiles than its stage ring holds,
    so the ring wraps several times."""
    Bsz, D = shape
    s = _step_inputs(Bsz, D, N, dtype, 1000 + N + D)
    g = to_dev(s)
    st = g["state"].clone()
    y = Guarded((Bsz, D), dtype)
    ssm.ssm_state_update(st, g["u"], g["delta"], g["A"], g["Bm"], g["Cm"], Dskip=g["Dskip"],
                         delta_bias=g["delta_bias"], z=g["z"], y=y.t)
    assert ssm.ssm_device_error() == 0
    y.check_bands()
    st_ref, y_ref = oracle.state_update(s["state"], s["u"], s["delta"], s["A"], s["Bm"], s["Cm"], s["Dskip"],
                                        s["delta_bias"], s["z"])
    assert_close(y.t, y_ref, y_tolerance(y_ref, dtype), "y")
    assert_close(st, st_ref, h_tolerance(st_ref, torch.float32), "state")


def test_state_update_streamed_without_optional_inputs_and_zero_A():
    s = _step_inputs(4, 128, 16, torch.bfloat16, 17, with_z=False, with_D=False)
    s["A"][70, 5] = 0.0
    s["delta_bias"] = None
    g = to_dev(s)
    st = g["state"].clone()
    y = ssm.ssm_state_update(st, g["u"], g["delta"], g["A"], g["Bm"], g["Cm"], zoh=True)
    assert ssm.ssm_device_error() == 0
    st_ref, y_ref = oracle.state_update(s["state"], s["u"], s["delta"], s["A"], s["Bm"], s["Cm"])
    assert_close(y, y_ref, y_tolerance(y_ref, torch.bfloat16), "y")
    assert_close(st, st_ref, h_tolerance(st_ref, torch.float32), "state")


def test_state_update_optional_inputs_and_zero_A():
    s = _step_inputs(2, 64, 16, torch.float32, 5, with_z=False, with_D=False)
    s["A"][7, 3] = 0.0
    s["delta_bias"] = None
    g = to_dev(s)
    st = g["state"].clone()
    y = ssm.ssm_state_update(st, g["u"], g["delta"], g["A"], g["Bm"], g["Cm"])
    st_ref, y_ref = oracle.state_update(s["state"], s["u"], s["delta"], s["A"], s["Bm"], s["Cm"])
    assert_close(y, y_ref, y_tolerance(y_ref, torch.float32), "y")
    assert_close(st, st_ref, h_tolerance(st_ref, torch.float32), "state")


def test_decode_steps_equal_scan_on_gpu():
    """128 single-token updates must reproduce one scan of length 128 (both CUDA paths)."""
    d = workloads.make_scan_inputs(workloads.SCAN_CONFIGS["mamba130m"], batch=4, dim=256, seqlen=128, with_h0=True)
    g = to_dev(d)
    y_scan, h_scan = ssm.ssm_scan_fwd(g["u"], g["delta"], g["A"], g["Bm"], g["Cm"], Dskip=g["Dskip"],
                                      delta_bias=g["delta_bias"], z=g["z"], h0=g["h0"], return_state=True,
                                      out_dtype=torch.float32)
    st = g["h0"].clone()
    ys = []
    for t in range(128):
        ys.append(ssm.ssm_state_update(st, g["u"][..., t].contiguous(), g["delta"][..., t].contiguous(), g["A"],
                                       g["Bm"][..., t].contiguous(), g["Cm"][..., t].contiguous(), Dskip=g["Dskip"],
                                       delta_bias=g["delta_bias"], z=g["z"][..., t].contiguous(),
                                       y=torch.empty((4, 256), dtype=torch.bfloat16, device="cuda")))
    y_dec = torch.stack(ys, dim=-1).float()
    y_ref, h_ref, _ = oracle.scan(d)
    assert_close(y_dec, y_ref.reshape(4, 256, 128), y_tolerance(y_ref.reshape(4, 256, 128), torch.bfloat16), "decode y")
    torch.testing.assert_close(st, h_scan, rtol=1e-4, atol=1e-5)


def test_decode_workload_full_size_sampled():
    """The decode workload exactly as bench.py runs it: 64 layers x 128 tokens, layer-major per token,
    inputs from a pool of 64 per-token sets; sampled layers {0, 63} and 16 batch rows checked every step."""
    cfg = workloads.DECODE_CONFIG
    P = 64
    pool = workloads.make_decode_pool(cfg, P, device="cuda")
    layers = [workloads.make_decode_layer(cfg, l, device="cuda") for l in range(cfg.layers)]
    check_layers = (0, cfg.layers - 1)
    rng = np.random.default_rng(11)
    brow = np.sort(rng.choice(cfg.batch, 16, replace=False))
    bsel = torch.tensor(brow, device="cuda")
    init = {l: layers[l]["state"][bsel].cpu() for l in check_layers}
    ys = {l: [] for l in check_layers}
    ins = {l: [] for l in check_layers}
    y = torch.empty((cfg.batch, cfg.dim), dtype=torch.bfloat16, device="cuda")
    for step in range(cfg.steps):
        for l in range(cfg.layers):
            k = workloads.decode_pool_index(l, step, P)
            L_ = layers[l]
            ssm.ssm_state_update(L_["state"], pool["u"][k], pool["delta"][k], L_["A"], pool["Bm"][k], pool["Cm"][k],
                                 Dskip=L_["Dskip"], delta_bias=L_["delta_bias"], z=pool["z"][k], y=y)
            if l in check_layers:
                ys[l].append(y[bsel].cpu())
                ins[l].append(k)
    torch.cuda.synchronize()
    for l in check_layers:
        L_ = layers[l]
        st = init[l]
        for step, k in enumerate(ins[l]):
            st_np, y_ref = oracle.state_update(st, pool["u"][k][bsel].cpu(), pool["delta"][k][bsel].cpu(),
                                               L_["A"].cpu(), pool["Bm"][k][bsel].cpu(), pool["Cm"][k][bsel].cpu(),
                                               L_["Dskip"].cpu(), L_["delta_bias"].cpu(), pool["z"][k][bsel].cpu())
            assert_close(ys[l][step], y_ref, y_tolerance(y_ref, torch.bfloat16), f"layer {l} step {step} y")
            st = torch.from_numpy(st_np)
        assert_close(L_["state"][bsel], st.numpy(), h_tolerance(st.numpy(), torch.bfloat16), f"layer {l} state")
