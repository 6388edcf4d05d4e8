"""Parity of the serving-side variants of the path (pwwt.cn/news/5168881 section 3.4), through the C ABI:

- multi-token verification: a short scan that also returns the state after every step (h_all), so a
  speculative decoder can commit the state at the accepted length;
- per-request state slots: scan and decode read and write a state cache indexed by state_indices (a
  negative index marks a padding row: its y is zero and no slot changes).

The oracle sees the same rows gathered from the cache on the host; slots that no row uses must come back
bit-identical."""
import numpy as np
import pytest
import torch

import oracle
import selective_state_space_156_b300 as ssm
import workloads
from gpu_helpers import assert_close, h_tolerance, to_dev, y_tolerance

pytestmark = pytest.mark.gpu


def _inputs(Bsz, D, N, L, dtype, seed, conv=False):
    cfg = workloads.SCAN_CONFIGS["mamba1.4b_conv" if conv else "mamba130m"]
    return workloads.make_scan_inputs(cfg, batch=Bsz, dim=D, seqlen=L, dstate=N, dtype=dtype, with_h0=True, seed=seed)


def _kw(g):
    return dict(Dskip=g["Dskip"], delta_bias=g["delta_bias"], z=g["z"], conv_w=g.get("conv_w"), conv_b=g.get("conv_b"))


@pytest.mark.parametrize("dt,N,D,L", [("bf16", 16, 64, 4), ("bf16", 16, 150, 1), ("f32", 4, 64, 13),
                                      ("bf16", 8, 128, 8), ("f32", 16, 32, 3000), ("bf16", 16, 256, 64),
                                      ("bf16", 12, 128, 40), ("bf16", 16, 64, 2048)])
def test_multi_token_pass_returns_every_state(dt, N, D, L):
    """y, the final state and the state after every step.  bf16 with L % 8 == 0 takes the packed kernel
    ((16, 64, 2048) with the L split, N = 12 with padded states); the rest the element-wise kernel,
    (f32, 16, 32, 3000) with the L split."""
    Bsz = 3
    d = _inputs(Bsz, D, N, L, dt, seed=7000 + N + D + L)
    g = to_dev(d)
    h_all = torch.full((Bsz, L, D, N), float("nan"), device="cuda")
    y, h = ssm.ssm_scan_fwd(g["u"], g["delta"], g["A"], g["Bm"], g["Cm"], h0=g["h0"], return_state=True,
                            h_all=h_all, workspace="auto", **_kw(g))
    torch.cuda.synchronize()
    extra = {"h_all": True}
    y_ref, h_ref, _ = oracle.scan(d, extra=extra)
    y_ref = y_ref.reshape(Bsz, D, L)
    hall_ref = extra["h_all"].reshape(Bsz, D, L, N).transpose(0, 2, 1, 3)  # (B, L, D, N)
    assert_close(y, y_ref, y_tolerance(y_ref, y.dtype), "y")
    assert_close(h, h_ref.reshape(Bsz, D, N), h_tolerance(h_ref.reshape(Bsz, D, N), g["u"].dtype), "h_out")
    assert_close(h_all, hall_ref, h_tolerance(hall_ref, g["u"].dtype), "h_all")
    assert torch.equal(h_all[:, -1], h), "the last state of the sequence is h_out"


@pytest.mark.parametrize("dt", ["bf16", "f32"])
@pytest.mark.parametrize("conv", [False, True])
def test_scan_on_state_slots(dt, conv):
    """Four requests on a cache of 7 slots, one of them padding; h0 and h_out are the same cache, and so
    are conv_init and conv_final."""
    Bsz, D, N, L, S = 4, 64, 16, 24, 7
    idx = torch.tensor([5, -1, 0, 3], dtype=torch.int32)
    d = _inputs(Bsz, D, N, L, dt, seed=7100 + int(conv), conv=conv)
    gen = torch.Generator().manual_seed(7101)
    cache = torch.randn((S, D, N), generator=gen) * 0.5
    W1 = 3
    ccache = torch.randn((S, D, W1), generator=gen).to(d["u"].dtype) if conv else None
    g = to_dev(d)
    cache_dev, idx_dev = cache.cuda(), idx.cuda()
    cc_dev = ccache.cuda() if conv else None
    hall = torch.full((Bsz, L, D, N), float("nan"), device="cuda")
    y = torch.full(d["u"].shape, float("nan"), dtype=g["u"].dtype, device="cuda")
    ssm.ssm_scan_fwd(g["u"], g["delta"], g["A"], g["Bm"], g["Cm"], h0=cache_dev, h_out=cache_dev, y=y,
                     state_indices=idx_dev, conv_init=cc_dev, conv_final=cc_dev, h_all=hall, **_kw(g))
    torch.cuda.synchronize()
    live = [b for b in range(Bsz) if idx[b] >= 0]
    sub = {k: (v[live] if isinstance(v, torch.Tensor) and v.dim() == 3 and v.shape[0] == Bsz else v)
           for k, v in d.items()}
    sub["h0"] = cache[idx[live].long()]
    if conv:
        sub["conv_init"] = ccache[idx[live].long()]
    extra = {"h_all": True}
    y_ref, h_ref, _ = oracle.scan(sub, extra=extra)
    nl = len(live)
    y_ref = y_ref.reshape(nl, D, L)
    assert_close(y[live], y_ref, y_tolerance(y_ref, y.dtype), "y of the live rows")
    assert bool((y[1] == 0).all()), "a padding row's y is zero"
    h_new = cache_dev.cpu()
    for k, b in enumerate(live):
        ref = h_ref.reshape(nl, D, N)[k]
        assert_close(h_new[int(idx[b])], ref, h_tolerance(ref, g["u"].dtype), f"slot {int(idx[b])}")
    for s_ in set(range(S)) - {int(i) for i in idx if i >= 0}:
        assert torch.equal(h_new[s_], cache[s_]), f"unused slot {s_} changed"
    hall_ref = extra["h_all"].reshape(nl, D, L, N).transpose(0, 2, 1, 3)
    assert_close(hall[live], hall_ref, h_tolerance(hall_ref, g["u"].dtype), "h_all of the live rows")
    assert bool(torch.isnan(hall[1]).all()), "a padding row's h_all is untouched"
    if conv:
        cnew = cc_dev.cpu()
        for b in live:
            assert torch.equal(cnew[int(idx[b])], d["u"][b, :, -W1:]), "conv history of a live slot"
        for s_ in set(range(S)) - {int(i) for i in idx if i >= 0}:
            assert torch.equal(cnew[s_], ccache[s_]), f"unused conv slot {s_} changed"


@pytest.mark.parametrize("D", [128, 100])   # streamed kernel, row kernel
@pytest.mark.parametrize("conv", [False, True])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_decode_on_state_slots(D, conv, dtype):
    Bsz, N, S, W = 5, 16, 9, 4
    idx = torch.tensor([8, 2, -1, 0, 6], dtype=torch.int32)
    gen = torch.Generator().manual_seed(7200 + D + int(conv))
    cache = torch.randn((S, D, N), generator=gen) * 0.5
    ccache = torch.randn((S, D, W - 1), generator=gen).to(dtype)
    s = {
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
    }
    g = to_dev(s)
    cd, ccd = cache.cuda(), ccache.cuda()
    y = torch.full((Bsz, D), float("nan"), dtype=dtype, device="cuda")
    ssm.ssm_state_update(cd, g["x"], g["delta"], g["A"], g["Bm"], g["Cm"], Dskip=g["Dskip"], delta_bias=g["delta_bias"],
                         z=g["z"], y=y, conv_w=g["conv_w"] if conv else None, conv_b=g["conv_b"] if conv else None,
                         conv_state=ccd if conv else None, state_indices=idx.cuda())
    assert ssm.ssm_device_error() == 0
    live = [b for b in range(Bsz) if idx[b] >= 0]
    li = idx[live].long()
    kw = dict(conv_w=s["conv_w"], conv_b=s["conv_b"], conv_state=ccache[li]) if conv else {}
    out = oracle.state_update(cache[li], s["x"][live], s["delta"][live], s["A"], s["Bm"][live], s["Cm"][live],
                              s["Dskip"], s["delta_bias"], s["z"][live], **kw)
    st_ref, y_ref = out[0], out[1]
    assert_close(y[live], y_ref, y_tolerance(y_ref, dtype), "y of the live rows")
    assert bool((y[2] == 0).all()), "a padding row's y is zero"
    cnew, ccnew = cd.cpu(), ccd.cpu()
    for k, b in enumerate(live):
        assert_close(cnew[int(idx[b])], st_ref[k], h_tolerance(st_ref[k], dtype), f"slot {int(idx[b])}")
        if conv:
            assert torch.equal(ccnew[int(idx[b])].double(), torch.tensor(np.ascontiguousarray(out[2][k])))
    for s_ in set(range(S)) - {int(i) for i in idx if i >= 0}:
        assert torch.equal(cnew[s_], cache[s_]), f"unused slot {s_} changed"
        assert torch.equal(ccnew[s_], ccache[s_]), f"unused conv slot {s_} changed"


def test_speculative_verify_then_commit_equals_plain_decode():
    """A verification pass over T candidate tokens of every request (h_all kept), then the state of each
    request committed at its accepted length k_b, then one more decode step: equal to decoding the
    accepted tokens one by one and then that step."""
    Bsz, D, N, T, S = 4, 128, 16, 5, 6
    idx = torch.tensor([4, 1, 5, 2], dtype=torch.int32, device="cuda")
    accepted = [5, 0, 3, 1]
    d = _inputs(Bsz, D, N, T + 1, "bf16", seed=7300)
    g = to_dev(d)
    gen = torch.Generator().manual_seed(7301)
    cache0 = (torch.randn((S, D, N), generator=gen) * 0.5).cuda()
    piece = {k: g[k][..., :T].contiguous() for k in ("u", "delta", "z", "Bm", "Cm")}
    # verify: y of all T candidates and the state after each; the cache itself is not written
    cache = cache0.clone()
    h_all = torch.empty((Bsz, T, D, N), device="cuda")
    ssm.ssm_scan_fwd(piece["u"], piece["delta"], g["A"], piece["Bm"], piece["Cm"], h0=cache, state_indices=idx,
                     h_all=h_all, Dskip=g["Dskip"], delta_bias=g["delta_bias"], z=piece["z"])
    for b, k in enumerate(accepted):
        if k > 0:
            cache[int(idx[b])] = h_all[b, k - 1]
    # reference: decode the accepted tokens one by one on a copy of the cache
    ref = cache0.clone()
    for b, k in enumerate(accepted):
        st = ref[int(idx[b])][None].clone()
        for t in range(k):
            ssm.ssm_state_update(st, g["u"][b:b + 1, :, t].contiguous(), g["delta"][b:b + 1, :, t].contiguous(),
                                 g["A"], g["Bm"][b:b + 1, :, t].contiguous(), g["Cm"][b:b + 1, :, t].contiguous(),
                                 Dskip=g["Dskip"], delta_bias=g["delta_bias"], z=g["z"][b:b + 1, :, t].contiguous())
        ref[int(idx[b])] = st[0]
    torch.cuda.synchronize()
    torch.testing.assert_close(cache, ref, rtol=1e-4, atol=1e-5)
    # one more step on the slots, from both caches
    step = {k: g[k][..., T].contiguous() for k in ("u", "delta", "z", "Bm", "Cm")}
    ya = ssm.ssm_state_update(cache, step["u"], step["delta"], g["A"], step["Bm"], step["Cm"], Dskip=g["Dskip"],
                              delta_bias=g["delta_bias"], z=step["z"], state_indices=idx)
    yb = ssm.ssm_state_update(ref, step["u"], step["delta"], g["A"], step["Bm"], step["Cm"], Dskip=g["Dskip"],
                              delta_bias=g["delta_bias"], z=step["z"], state_indices=idx)
    torch.cuda.synchronize()
    torch.testing.assert_close(ya.float(), yb.float(), rtol=1e-2, atol=1e-2)
    torch.testing.assert_close(cache, ref, rtol=1e-4, atol=1e-5)
