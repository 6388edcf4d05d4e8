"""GPU parity in the regime where the zero-order hold's input factor E = (exp(dt a) - 1) / a cancels:
small |A| (-1e-4, -1e-3, -1e-2 per state) and small steps dt (1e-4, 1e-3, 1e-2), against the fp64 oracle
element by element at the stated tolerances.

Every kernel that discretises is covered: the element-wise scan (fp32 I/O and bf16 with L % 8 != 0), the
packed bf16 scan (N <= 16) with and without the L split, the four-lanes-per-channel scan (N = 32, 64),
both decode kernels (streamed and per-row) and the backward pass (dA and d(delta) included).  The ZOH
definition is that of dpshk.com/news/3333417 section 2.2 and lshu.cn/news/79586 section 2.2; trained
models reach small |A| because A = -exp(A_log) with A_log learned."""
import numpy as np
import pytest
import torch

import oracle
import selective_state_space_156_b300 as ssm
import workloads
from gpu_helpers import Guarded, assert_close, h_tolerance, to_dev, y_tolerance
from oracle import backward as obwd

pytestmark = pytest.mark.gpu

SMALL_A = (-1e-4, -1e-3, -1e-2)
DTS = (1e-4, 1e-3, 1e-2)


def _small_a(D, N, seed, ordinary=True):
    """A[d, n] cycles through the small values; with `ordinary`, every fourth state keeps the S4D-real
    -(n+1), so blocks mix both regimes."""
    g = torch.Generator().manual_seed(seed)
    A = torch.empty((D, N), dtype=torch.float32)
    for d in range(D):
        for n in range(N):
            if ordinary and n % 4 == 3:
                A[d, n] = -(n + 1.0)
            else:
                A[d, n] = SMALL_A[(d + n) % 3]
    return A * (0.75 + 0.5 * torch.rand((D, 1), generator=g))


def _scan_inputs(cfg_name, Bsz, D, N, L, dtype, dt, seed, conv=False):
    cfg = workloads.SCAN_CONFIGS[cfg_name]
    d = workloads.make_scan_inputs(cfg, batch=Bsz, dim=D, seqlen=L, dstate=N, dtype=dtype, with_h0=True, seed=seed)
    g = torch.Generator().manual_seed(seed + 11)
    # softplus off, no bias: the step is exactly the (rounded) input, dt (0.75 .. 1.25)
    raw = dt * (0.75 + 0.5 * torch.rand((Bsz, D, L), generator=g))
    d["delta"] = raw.to(d["u"].dtype)
    d["delta_bias"] = None
    d["delta_softplus"] = False
    d["A"] = _small_a(D, N, seed)
    if not conv:
        d["conv_w"] = None
        d["conv_b"] = None
    return d


def _check_scan(d, workspace="auto"):
    g = to_dev(d)
    Bsz, D, L = g["u"].shape
    N = g["A"].shape[1]
    y = Guarded((Bsz, D, L), g["u"].dtype)
    h = Guarded((Bsz, D, N), torch.float32)
    ssm.ssm_scan_fwd(g["u"], g["delta"], g["A"], g["Bm"], g["Cm"], Dskip=g.get("Dskip"), z=g.get("z"),
                     conv_w=g.get("conv_w"), conv_b=g.get("conv_b"), h0=g["h0"], h_out=h.t, y=y.t,
                     delta_softplus=False, zoh=True, workspace=workspace)
    torch.cuda.synchronize()
    y.check_bands()
    h.check_bands()
    y_ref, h_ref, _ = oracle.scan(d)
    y_ref = y_ref.reshape(Bsz, D, L)
    h_ref = h_ref.reshape(Bsz, D, N)
    assert_close(y.t, y_ref, y_tolerance(y_ref, g["u"].dtype), "y")
    assert_close(h.t, h_ref, h_tolerance(h_ref, d["u"].dtype), "h_out")


@pytest.mark.parametrize("dt", DTS)
@pytest.mark.parametrize("L", [61, 2048])
def test_element_scan_fp32(dt, L):
    _check_scan(_scan_inputs("tiny", 2, 70, 16, L, "f32", dt, 31))


@pytest.mark.parametrize("dt", DTS)
def test_element_scan_bf16_ragged_length(dt):
    _check_scan(_scan_inputs("mamba130m", 2, 70, 16, 1021, "bf16", dt, 37))


@pytest.mark.parametrize("dt", DTS)
@pytest.mark.parametrize("split", [True, False])
@pytest.mark.parametrize("conv", [False, True])
def test_packed_scan(dt, split, conv):
    _check_scan(_scan_inputs("mamba1.4b_conv" if conv else "mamba130m", 2, 136, 16, 2048, "bf16", dt, 41,
                             conv=conv), workspace="auto" if split else None)


@pytest.mark.parametrize("dt", DTS)
@pytest.mark.parametrize("N", [32, 64])
def test_four_lane_scan(dt, N):
    _check_scan(_scan_inputs("mamba130m", 2, 72, N, 1024, "bf16", dt, 43))


@pytest.mark.parametrize("zoh", [True, False])
def test_long_memory_equilibrium_fp32(zoh):
    """A constant input into states that forget slowly (|dt a| 5e-4 .. 5e-3, 8192 steps) drives each
    state to its equilibrium E B v / (1 - Abar), about 1 / |a|, where 1 - Abar decides the level: an
    error of k ulp in Abar moves the state by about k 6e-8 / |dt a| relative.  Checked per state."""
    Bsz, D, N, L = 1, 32, 16, 8192
    cfg = workloads.SCAN_CONFIGS["tiny"]
    d = workloads.make_scan_inputs(cfg, batch=Bsz, dim=D, seqlen=L, dstate=N, dtype="f32", seed=61)
    g = torch.Generator().manual_seed(67)
    d["u"] = torch.ones((Bsz, D, L), dtype=torch.float32)
    d["Bm"] = torch.ones((Bsz, N, L), dtype=torch.float32)
    d["Cm"] = (1.0 + torch.rand((Bsz, N, 1), generator=g)).expand(Bsz, N, L).contiguous()
    d["z"] = None
    d["Dskip"] = None
    d["delta"] = torch.full((Bsz, D, L), 0.5, dtype=torch.float32)
    d["delta_bias"] = None
    d["delta_softplus"] = False
    d["A"] = -1e-3 * torch.exp(torch.rand((D, N), generator=g) * 2.3)
    d["conv_w"] = d["conv_b"] = None
    d["zoh"] = zoh
    gd = to_dev(d)
    y, h = ssm.ssm_scan_fwd(gd["u"], gd["delta"], gd["A"], gd["Bm"], gd["Cm"], delta_softplus=False, zoh=zoh,
                            return_state=True)
    torch.cuda.synchronize()
    y_ref, h_ref, _ = oracle.scan(d)
    assert_close(y, y_ref.reshape(Bsz, D, L), y_tolerance(y_ref.reshape(Bsz, D, L), torch.float32), "y")
    assert_close(h, h_ref.reshape(Bsz, D, N), h_tolerance(h_ref.reshape(Bsz, D, N), torch.float32), "h_out")


# Cases of a randomised sweep of the fp32-output scan (seed, batch, channels, states, length, bf16 inputs, zoh,
# z, D skip, h0, A drawn small or around zero) that missed the 1e-4 (1 + |y|) bound by 2.4 and 3.1 times
# while the decay came from the hardware exp2, and meet it with the series decay (every row checked).
SWEEP_CASES = [
    (437883965, 2, 62, 4, 6512, False, False, True, True, True, "small"),
    (577547123, 2, 57, 16, 256, False, True, False, True, False, "near_zero"),
]


@pytest.mark.parametrize("case", SWEEP_CASES, ids=lambda c: str(c[0]))
def test_fp32_output_sweep_cases(case):
    seed, Bsz, D, N, L, in_bf16, zoh, has_z, has_d, with_h0, a_kind = case
    cfg = workloads.ScanConfig("sweep", Bsz, D, N, L, "bf16" if in_bf16 else "f32", seed=seed % 100000)
    d = workloads.make_scan_inputs(cfg, with_h0=with_h0)
    g = torch.Generator().manual_seed(seed)
    if a_kind == "small":   # |A| log-uniform in [1e-4, 1]
        d["A"] = -torch.exp(torch.empty(D, N).uniform_(-9.2, 0.0, generator=g))
    else:                   # A uniform in [-1, 0.02]: a few states grow slowly
        d["A"] = torch.empty(D, N).uniform_(-1.0, 0.02, generator=g)
    if not has_z:
        d["z"] = None
    if not has_d:
        d["Dskip"] = None
    d["delta_bias"] = None   # dt = softplus(delta) about 0.5 .. 1: long memory where |A| is small
    d["zoh"] = zoh
    gd = to_dev(d)
    y, h = ssm.ssm_scan_fwd(gd["u"], gd["delta"], gd["A"], gd["Bm"], gd["Cm"], Dskip=gd.get("Dskip"), z=gd.get("z"),
                            h0=gd.get("h0"), zoh=zoh, out_dtype=torch.float32, return_state=True)
    torch.cuda.synchronize()
    y_ref, h_ref, _ = oracle.scan(d)
    assert_close(y, y_ref.reshape(Bsz, D, L), y_tolerance(y_ref, torch.float32).reshape(Bsz, D, L), "y")
    assert_close(h, h_ref.reshape(Bsz, D, N), h_tolerance(h_ref, d["u"].dtype).reshape(Bsz, D, N), "h_out")


def test_packed_scan_fast_form_still_used_for_ordinary_A():
    """|A| >= 1/4 everywhere keeps the fast form; the result matches as before."""
    d = _scan_inputs("mamba130m", 2, 136, 16, 2048, "bf16", 1e-2, 47)
    d["A"] = -torch.arange(1, 17, dtype=torch.float32).repeat(136, 1) * 0.26
    _check_scan(d, workspace=None)


# ------------------------------------------------------------------------------------------------
# decode
# ------------------------------------------------------------------------------------------------
def _decode_inputs(Bsz, D, N, dtype, dt, seed):
    g = torch.Generator().manual_seed(seed)
    return {
        "state": torch.randn((Bsz, D, N), generator=g) * 0.5,
        "u": torch.randn((Bsz, D), generator=g).to(dtype),
        "delta": (dt * (0.75 + 0.5 * torch.rand((Bsz, D), generator=g))).to(dtype),
        "A": _small_a(D, N, seed),
        "Bm": torch.randn((Bsz, N), generator=g).to(dtype),
        "Cm": torch.randn((Bsz, N), generator=g).to(dtype),
        "Dskip": torch.randn(D, generator=g),
        "z": torch.randn((Bsz, D), generator=g).to(dtype),
    }


@pytest.mark.parametrize("dt", DTS)
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("kernel,N,D", [("streamed", 16, 200), ("streamed", 64, 64), ("row", 4, 150),
                                        ("row", 16, 75)])
def test_decode_steps(dt, dtype, kernel, N, D):
    """64 decode steps in a row (the error of each step is carried in the state), against the oracle's
    step applied as many times."""
    s = _decode_inputs(3, D, N, dtype, dt, 53 + N + D)
    g = to_dev(s)
    st = g["state"].clone()
    st_ref = s["state"].clone().to(torch.float64)
    gen = torch.Generator().manual_seed(59)
    for k in range(64):
        u = torch.randn(s["u"].shape, generator=gen).to(dtype)
        y = ssm.ssm_state_update(st, u.cuda(), g["delta"], g["A"], g["Bm"], g["Cm"], Dskip=g["Dskip"], z=g["z"],
                                 delta_softplus=False, zoh=True)
        st_ref, y_ref = oracle.state_update(st_ref, u, s["delta"], s["A"], s["Bm"], s["Cm"], s["Dskip"], None,
                                            s["z"], zoh=True, delta_softplus=False)
        st_ref = torch.as_tensor(np.asarray(st_ref)).reshape(s["state"].shape)
        y_ref = np.asarray(y_ref).reshape(s["u"].shape)
        assert_close(y, y_ref, y_tolerance(y_ref, dtype), f"y (step {k})")
    assert ssm.ssm_device_error() == 0
    ref = st_ref.numpy()
    assert_close(st, ref, h_tolerance(ref, torch.float32), "state after 64 steps")


# ------------------------------------------------------------------------------------------------
# backward
# ------------------------------------------------------------------------------------------------
def _bwd_tol(ref, stored_dtype, in_dtype):
    rms = float(np.sqrt(np.mean(ref * ref))) if ref.size else 0.0
    k = 2e-2 if stored_dtype == torch.bfloat16 else (2e-3 if in_dtype == torch.bfloat16 else 2e-4)
    return k * (np.abs(ref) + rms) + 1e-30


@pytest.mark.parametrize("dt", DTS)
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_backward(dt, dtype):
    d = _scan_inputs("mamba130m", 2, 66, 16, 256, dtype, dt, 61)
    g = to_dev(d)
    Bsz, D, L = g["u"].shape
    N = 16
    h_ckpt = torch.empty((Bsz, ssm.ckpt_count(L), D, N), dtype=torch.float32, device="cuda")
    kw = dict(Dskip=g["Dskip"], z=g["z"], delta_softplus=False, zoh=True)
    ssm.ssm_scan_fwd(g["u"], g["delta"], g["A"], g["Bm"], g["Cm"], h0=g["h0"], h_ckpt=h_ckpt, **kw)
    gen = torch.Generator().manual_seed(67)
    dy = torch.randn((Bsz, D, L), generator=gen).to(g["u"].dtype)
    dh = torch.randn((Bsz, D, N), generator=gen) * 0.3
    grads = ssm.ssm_scan_bwd(g["u"], g["delta"], g["A"], g["Bm"], g["Cm"], dy.cuda(), h_ckpt, h0=g["h0"],
                             dh_out=dh.cuda(), **kw)
    torch.cuda.synchronize()
    ref = obwd.scan_bwd(d, dy.cpu(), dh)
    for k in ("u", "delta", "A", "Bm", "Cm", "Dskip", "z", "h0"):
        assert_close(grads[k], ref[k], _bwd_tol(ref[k], grads[k].dtype, g["u"].dtype), f"d{k}")
