"""Parity of the backward pass (ssm_scan_bwd) against the fp64 autograd oracle, through the C ABI.

The forward runs on the GPU keeping state checkpoints (h_ckpt, every 8th step), the backward recomputes
the other states from them; every
gradient is compared element by element with the oracle's on the same (rounded) inputs and dy.  Small
problems cover the flags (conv with history, gate, zero-order hold or simplified, softplus on or off, an
A = 0 entry, dh_out, h0), ragged L and a ragged channel tail; the Mamba-1.4B layer shape is checked on
sampled rows (per-row gradients) and sampled channels (per-channel sums over the batch)."""
import numpy as np
import pytest
import torch

import oracle
import selective_state_space_156_b300 as ssm
import workloads
from gpu_helpers import assert_close, to_dev
from oracle import backward as obwd

pytestmark = pytest.mark.gpu

KEYS = ["u", "delta", "A", "Bm", "Cm", "Dskip", "delta_bias", "z", "conv_w", "conv_b", "conv_init", "h0"]


def _tol(ref, stored_dtype, in_dtype):
    """Per element: scale-relative (the reference's magnitude plus its rms).  Gradients stored in bf16 get
    the bf16 output bound; fp32 gradients from bf16 inputs 2e-3, from fp32 inputs 2e-4 (fp32 arithmetic
    over the recurrence, the forward's states included)."""
    rms = float(np.sqrt(np.mean(ref * ref))) if ref.size else 0.0
    if stored_dtype == torch.bfloat16:
        k = 2e-2
    else:
        k = 2e-3 if in_dtype == torch.bfloat16 else 2e-4
    return k * (np.abs(ref) + rms) + 1e-30


def _run(d, dy, dh_out=None, workspace="auto"):
    g = to_dev(d)
    Bsz, D, L = g["u"].shape
    N = g["A"].shape[1]
    kw = dict(Dskip=g.get("Dskip"), delta_bias=g.get("delta_bias"), z=g.get("z"), conv_w=g.get("conv_w"),
              conv_b=g.get("conv_b"), delta_softplus=d.get("delta_softplus", True), zoh=d.get("zoh", True))
    h_ckpt = torch.empty((Bsz, ssm.ckpt_count(L), D, N), dtype=torch.float32, device="cuda")
    ssm.ssm_scan_fwd(g["u"], g["delta"], g["A"], g["Bm"], g["Cm"], h0=g.get("h0"), h_ckpt=h_ckpt,
                     conv_init=g.get("conv_init"), **kw)
    dyd = dy.to(g["u"].dtype).cuda()
    grads = ssm.ssm_scan_bwd(g["u"], g["delta"], g["A"], g["Bm"], g["Cm"], dyd, h_ckpt, h0=g.get("h0"),
                             conv_init=g.get("conv_init"), dh_out=None if dh_out is None else dh_out.cuda(),
                             workspace=workspace, **kw)
    torch.cuda.synchronize()
    return grads, dyd.cpu()


def _compare(d, grads, ref, in_dtype):
    for k in KEYS:
        if k not in ref or d.get(k) is None and k != "h0":
            continue
        got = grads[k]
        r = ref[k]
        assert_close(got, r, _tol(r, got.dtype, in_dtype), f"d{k}")


def _inputs(Bsz, D, N, L, dt, seed, *, conv=True, z=True, zoh=True, softplus=True, h0=True):
    cfg = workloads.SCAN_CONFIGS["mamba1.4b_conv" if conv else "mamba130m"]
    d = workloads.make_scan_inputs(cfg, batch=Bsz, dim=D, seqlen=L, dstate=N, dtype=dt, with_h0=h0, seed=seed)
    d["zoh"] = zoh
    d["delta_softplus"] = softplus
    if not z:
        d["z"] = None
    if not softplus:  # dt = delta + bias directly: a positive step
        d["delta"] = (0.02 + 0.05 * d["delta"].float().abs()).to(d["delta"].dtype)
        d["delta_bias"] = torch.full((D,), 0.01)
    if conv:
        gen = torch.Generator().manual_seed(seed + 5)
        d["conv_init"] = torch.randn((Bsz, D, 3), generator=gen).to(d["u"].dtype)
    return d


@pytest.mark.parametrize("dt", ["f32", "bf16"])
@pytest.mark.parametrize("N,D,L", [(16, 150, 61), (4, 64, 128), (8, 130, 40)])
@pytest.mark.parametrize("flags", [dict(), dict(conv=False), dict(z=False, zoh=False), dict(softplus=False, h0=False)])
def test_backward_matches_oracle(dt, N, D, L, flags):
    seed = 9000 + N + D + L + 7 * len(flags)
    d = _inputs(2, D, N, L, dt, seed, **flags)
    d["A"][min(5, D - 1), N - 1] = 0.0
    gen = torch.Generator().manual_seed(seed + 1)
    dy = torch.randn((2, D, L), generator=gen).to(d["u"].dtype)
    dh = torch.randn((2, D, N), generator=gen) * 0.3
    grads, dyr = _run(d, dy, dh)
    ref = obwd.scan_bwd(d, dyr, dh)
    _compare(d, grads, ref, d["u"].dtype)


@pytest.mark.parametrize("W", [1, 2, 3])
def test_backward_conv_widths(W):
    """Filters narrower than 4 taps ((D, W) taps and their gradient, W - 1 steps of history)."""
    d = _inputs(2, 96, 8, 72, "bf16", 9500 + W)
    d["conv_w"] = d["conv_w"][:, 4 - W:].contiguous()
    d["conv_init"] = d["conv_init"][..., 4 - W:].contiguous() if W > 1 else None
    gen = torch.Generator().manual_seed(9600 + W)
    dy = torch.randn((2, 96, 72), generator=gen).to(torch.bfloat16)
    grads, dyr = _run(d, dy)
    ref = obwd.scan_bwd(d, dyr)
    _compare(d, grads, ref, torch.bfloat16)


def test_backward_at_the_layer_shape_sampled():
    """The Mamba-1.4B layer with its fused front end (8 x 4096 x 16 x 2048, bf16): per-row gradients on 6
    sampled rows (each row's oracle is the same problem cut to that row), per-channel sums (dA, D skip, dt
    bias, conv taps and bias) on 3 sampled channels over the whole batch."""
    cfg = workloads.SCAN_CONFIGS["mamba1.4b_conv"]
    d = workloads.make_scan_inputs(cfg)
    Bsz, D, L = d["u"].shape
    gen = torch.Generator().manual_seed(91)
    dy = torch.randn((Bsz, D, L), generator=gen).to(torch.bfloat16)
    grads, dyr = _run(d, dy)
    rng = np.random.default_rng(92)

    def cut(bs, ds):
        sub = {}
        for k, v in d.items():
            if not isinstance(v, torch.Tensor):
                sub[k] = v
            elif k in ("u", "delta", "z"):
                sub[k] = v[bs][:, ds]
            elif k in ("Bm", "Cm"):
                sub[k] = v[bs]
            elif k in ("A", "conv_w"):
                sub[k] = v[ds]
            elif k in ("Dskip", "delta_bias", "conv_b"):
                sub[k] = v[ds]
            else:
                sub[k] = v
        return sub, dyr[bs][:, ds]

    for _ in range(6):
        b, c = int(rng.integers(Bsz)), int(rng.integers(D))
        sub, dys = cut([b], [c])
        ref = obwd.scan_bwd(sub, dys)
        for k in ("u", "delta", "z", "h0"):
            got = grads[k][b, c][None, None]
            assert_close(got, ref[k], _tol(ref[k], got.dtype, torch.bfloat16), f"d{k} row ({b}, {c})")
    for _ in range(3):
        c = int(rng.integers(D))
        sub, dys = cut(list(range(Bsz)), [c])
        ref = obwd.scan_bwd(sub, dys)
        for k in ("A", "Dskip", "delta_bias", "conv_w", "conv_b"):
            got = grads[k][c][None]
            assert_close(got, ref[k], _tol(ref[k], got.dtype, torch.bfloat16), f"d{k} channel {c}")


@pytest.mark.parametrize("dt,conv,L", [("bf16", True, 2048), ("f32", False, 3000), ("bf16", True, 1100)])
def test_backward_with_the_l_split_matches_oracle(dt, conv, L):
    """Few rows and a long sequence: the pass splits L, summarises every later segment's adjoint and folds
    it in (and, with the conv, adds the input gradients each segment owes to the steps before it); every
    gradient against the oracle, and against the same pass without the split."""
    D, N = 64, 16
    d = _inputs(1, D, N, L, dt, 9800 + L, conv=conv)
    gen = torch.Generator().manual_seed(9801)
    dy = torch.randn((1, D, L), generator=gen).to(d["u"].dtype)
    dh = torch.randn((1, D, N), generator=gen) * 0.3
    grads, dyr = _run(d, dy, dh)
    ref = obwd.scan_bwd(d, dyr, dh)
    _compare(d, grads, ref, d["u"].dtype)
    plain, _ = _run(d, dy, dh, workspace=None)
    for k, v in plain.items():
        tol = 2e-2 if v.dtype == torch.bfloat16 else 1e-4
        torch.testing.assert_close(grads[k].float(), v.float(), rtol=tol, atol=tol * float(v.float().abs().max() + 1e-6))


@pytest.mark.parametrize("dt,L,D,split", [("bf16", 2048, 136, True), ("bf16", 512, 300, False),
                                          ("f32", 1021, 70, True), ("f32", 77, 40, False)])
def test_forward_checkpoints_are_the_states_at_every_8th_step(dt, L, D, split):
    """h_ckpt from the forward (packed kernel for aligned bf16, element-wise kernel otherwise; with and
    without the L split) holds the oracle's state after steps 7, 15, ... and after the last step."""
    d = _inputs(2, D, 16, L, dt, 9900 + L, conv=(dt == "bf16"))
    g = to_dev(d)
    h_ckpt = torch.full((2, ssm.ckpt_count(L), D, 16), float("nan"), dtype=torch.float32, device="cuda")
    ssm.ssm_scan_fwd(g["u"], g["delta"], g["A"], g["Bm"], g["Cm"], Dskip=g.get("Dskip"),
                     delta_bias=g.get("delta_bias"), z=g.get("z"), conv_w=g.get("conv_w"), conv_b=g.get("conv_b"),
                     conv_init=g.get("conv_init"), h0=g.get("h0"), h_ckpt=h_ckpt,
                     workspace="auto" if split else None)
    torch.cuda.synchronize()
    extra = {"h_all": True}
    oracle.scan(d, extra=extra)
    ha = extra["h_all"].reshape(2, D, L, 16)
    steps = [min(8 * c + 7, L - 1) for c in range(ssm.ckpt_count(L))]
    want = np.transpose(ha[:, :, steps, :], (0, 2, 1, 3))
    got = h_ckpt.double().cpu().numpy()
    tol = (1e-4 if dt == "f32" else 1e-3) * (1.0 + np.abs(want))
    assert_close(got, want, tol, "h_ckpt")
