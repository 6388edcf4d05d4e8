"""Parity of the Mamba-2 (SSD) scan on the tensor cores (ssd_scan_fwd) against the fp64 oracle, through
the C ABI.

Small problems cover the flags (softplus on or off, zero-order hold or the simplified input scale, gate,
initial state), one to four groups, a ragged last chunk, the shortest accepted sequence, d_state 64 and
an A = 0 head;
the Mamba-2 2.7B layer (8 x 80 heads x 64 x 128 states x 2048 steps) is checked on sampled channels.
Tolerances: y (bf16) |err| <= 2e-2 (|y_ref| + rms(y_ref)) per element and, across all elements,
rms(err) <= 5e-3 rms(y_ref); the final state (fp32) |err| <= 1e-3 (1 + |h_ref|)."""
import numpy as np
import pytest
import torch

import selective_state_space_156_b300 as ssm
import workloads
from gpu_helpers import Guarded, assert_close, h_tolerance, to_dev, y_tolerance
from oracle.ssd import ssd_scan

pytestmark = pytest.mark.gpu


def _run(d, return_state=True):
    g = to_dev(d)
    Bsz, D, L = g["x"].shape
    out = Guarded((Bsz, D, L), torch.bfloat16)
    r = ssm.ssd_scan_fwd(g["x"], g["dt"], g["A"], g["Bm"], g["Cm"], nheads=d["nheads"], ngroups=d["ngroups"],
                         Dskip=g.get("Dskip"), dt_bias=g.get("dt_bias"), z=g.get("z"), h0=g.get("h0"),
                         return_state=return_state, y=out.t, delta_softplus=d["delta_softplus"], zoh=d["zoh"])
    torch.cuda.synchronize()
    out.check_bands()
    return r if return_state else (r, None)


def _check_y(y, ref, what):
    assert_close(y, ref, y_tolerance(ref, torch.bfloat16), what)
    g = y.detach().float().cpu().double().numpy().reshape(ref.shape)
    rms = float(np.sqrt(np.mean(ref * ref)))
    agg = float(np.sqrt(np.mean((g - ref) ** 2)))
    assert agg <= 5e-3 * rms, f"{what}: rms error {agg:.3e} above 5e-3 of rms(y) {rms:.3e}"


def _small(L, G, seed, *, z=True, h0=True, zoh=False, softplus=True, H=4, Bsz=2, N=128):
    d = workloads.make_ssd_inputs(workloads.SSD_CONFIGS["ssd_small"], batch=Bsz, nheads=H, ngroups=G, seqlen=L,
                                  dstate=N, with_h0=h0, has_z=z, seed=seed)
    d["zoh"] = zoh
    d["delta_softplus"] = softplus
    if not softplus:  # dt = raw + bias directly: a positive step
        d["dt"] = (0.01 + 0.05 * d["dt"].float().abs()).to(torch.bfloat16)
        d["dt_bias"] = torch.full((H,), 0.01)
    return d


FLAGS = [dict(), dict(zoh=True), dict(z=False, h0=False), dict(softplus=False, zoh=True, h0=False)]


@pytest.mark.parametrize("L", [8, 128, 200, 384])
@pytest.mark.parametrize("flags", range(len(FLAGS)))
def test_ssd_matches_oracle(L, flags):
    d = _small(L, 2, 3000 + L + 17 * flags, **FLAGS[flags])
    y, h = _run(d)
    ref_y, ref_h, _ = ssd_scan(d)
    _check_y(y, ref_y.reshape(y.shape), f"y L={L} flags={FLAGS[flags]}")
    assert_close(h, ref_h.reshape(h.shape), h_tolerance(ref_h.reshape(h.shape), torch.bfloat16), "h_out")


@pytest.mark.parametrize("G", [1, 4])
def test_ssd_groups(G):
    d = _small(256, G, 3100 + G)
    y, h = _run(d)
    ref_y, ref_h, _ = ssd_scan(d)
    _check_y(y, ref_y.reshape(y.shape), f"y G={G}")
    assert_close(h, ref_h.reshape(h.shape), h_tolerance(ref_h.reshape(h.shape), torch.bfloat16), "h_out")


@pytest.mark.parametrize("L,flags", [(200, 0), (384, 1), (8, 2), (136, 3)])
def test_ssd_state_64(L, flags):
    """d_state 64: the same kernel with the B and C copies ending at state 64 (states 64..127 read as zeros)."""
    d = _small(L, 2, 3500 + L + flags, N=64, **FLAGS[flags])
    y, h = _run(d)
    assert tuple(h.shape) == (2, 4, 64, 64)
    ref_y, ref_h, _ = ssd_scan(d)
    _check_y(y, ref_y.reshape(y.shape), f"y N=64 L={L}")
    assert_close(h, ref_h.reshape(h.shape), h_tolerance(ref_h.reshape(h.shape), torch.bfloat16), "h_out N=64")


@pytest.mark.parametrize("zoh", [False, True])
def test_ssd_a_zero_head(zoh):
    """A = 0 on one head: no decay, and zero-order hold's input scale takes its limit dt."""
    d = _small(136, 2, 3200 + zoh, zoh=zoh)
    d["A"][1] = 0.0
    y, h = _run(d)
    ref_y, ref_h, _ = ssd_scan(d)
    _check_y(y, ref_y.reshape(y.shape), "y with A = 0")
    assert_close(h, ref_h.reshape(h.shape), h_tolerance(ref_h.reshape(h.shape), torch.bfloat16), "h_out")


def test_ssd_chunked_calls_equal_one_call():
    """Two calls of 256 steps, the second starting from the first's final state, give exactly the output
    and state of one call of 512 (the split falls on a chunk boundary, so the arithmetic is the same)."""
    d = _small(512, 2, 3300)
    y_full, h_full = _run(d)
    first = dict(d, x=d["x"][..., :256].contiguous(), dt=d["dt"][..., :256].contiguous(),
                 Bm=d["Bm"][:, :, :256].contiguous(), Cm=d["Cm"][:, :, :256].contiguous(),
                 z=d["z"][..., :256].contiguous())
    y1, h1 = _run(first)
    second = dict(d, x=d["x"][..., 256:].contiguous(), dt=d["dt"][..., 256:].contiguous(),
                  Bm=d["Bm"][:, :, 256:].contiguous(), Cm=d["Cm"][:, :, 256:].contiguous(),
                  z=d["z"][..., 256:].contiguous(), h0=h1.cpu())
    y2, h2 = _run(second)
    assert torch.equal(torch.cat([y1, y2], dim=-1), y_full)
    assert torch.equal(h2, h_full)


def test_ssd_state_may_be_updated_in_place():
    d = _small(128, 2, 3400)
    ref_y, ref_h, _ = ssd_scan(d)
    g = to_dev(d)
    st = g["h0"].clone()
    y = ssm.ssd_scan_fwd(g["x"], g["dt"], g["A"], g["Bm"], g["Cm"], nheads=d["nheads"], ngroups=d["ngroups"],
                         Dskip=g["Dskip"], dt_bias=g["dt_bias"], z=g["z"], h0=st, h_out=st)
    torch.cuda.synchronize()
    _check_y(y, ref_y.reshape(y.shape), "y")
    assert_close(st, ref_h.reshape(st.shape), h_tolerance(ref_h.reshape(st.shape), torch.bfloat16), "state")


def test_ssd_at_the_mamba2_layer_shape_sampled():
    """The Mamba-2 2.7B layer as the benchmark runs it: every output finite, 32 sampled channels (y over
    all 2048 steps and their final state) against the oracle."""
    cfg = workloads.SSD_CONFIGS["mamba2_2.7b"]
    d = workloads.make_ssd_inputs(cfg)
    y, h = _run(d)
    assert bool(torch.isfinite(y).all())
    rng = np.random.default_rng(77)
    H, P = cfg.nheads, cfg.headdim
    rows = [(int(rng.integers(cfg.batch)), int(rng.integers(H)), int(rng.integers(P))) for _ in range(30)]
    rows += [(0, 0, 0), (cfg.batch - 1, H - 1, P - 1)]
    ref_y, ref_h, _ = ssd_scan(d, rows=rows)
    got_y = torch.stack([y[b, hh * P + p] for b, hh, p in rows])
    got_h = torch.stack([h[b, hh, p] for b, hh, p in rows])
    # the bf16 bound uses the rms of the sampled rows, which stands for the whole output
    _check_y(got_y, ref_y, "y (sampled channels)")
    assert_close(got_h, ref_h, h_tolerance(ref_h, torch.bfloat16), "h_out (sampled channels)")
    assert ssm.ssm_device_error() == 0
