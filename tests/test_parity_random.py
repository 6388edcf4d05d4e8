"""Randomised parity cases through the C ABI: fixed seeds draw shapes, dtypes and flags for the scan
forward, the backward pass, the decode step, the SSD layer and the state-slot paths of the scan and the
decode step, and each case is compared with the oracle at the stated bounds (the scan and decode on up to
48 sampled rows).

Ragged channel counts and lengths, every state size the dispatch distinguishes (1 to 16, 32, 64), fp32
and bf16 inputs and outputs, conv widths 1 to 4 with and without history, gate, D skip, dt bias, softplus
on or off, zero-order hold or the simplified scale, h0, checkpoints and per-step states, A drawn as S4D-real,
log-uniform small (|A| down to 1e-4) or with zeros.  Two regimes are left out by design: softplus off with
a negative step (the state grows without bound), and fp32 outputs of states that remember thousands of
steps at large dt, where the fp32 bound is relative to a y that cancels terms a thousand times larger and
a plain float32 recurrence misses it too."""
import random

import numpy as np
import pytest
import torch

import oracle
import selective_state_space_156_b300 as ssm
import workloads
from gpu_helpers import h_tolerance, y_tolerance
from oracle import backward as obwd
from oracle.ssd import ssd_scan
from test_parity_bwd import _compare as bwd_compare, _run as bwd_run
from test_parity_ssd import _check_y, _run as ssd_run, _small as ssd_small

pytestmark = pytest.mark.gpu


def _ratio(got, ref, tol):
    g = got.detach().float().cpu().double().numpy().reshape(ref.shape) if hasattr(got, "detach") else got
    assert np.isfinite(g).all(), "non-finite output"
    return float((np.abs(g - ref) / tol).max())


def _a(kind, D, N, g):
    if kind == "s4d":
        return -torch.arange(1, N + 1, dtype=torch.float32).repeat(D, 1)
    if kind == "small":   # |A| log-uniform in [1e-4, 1]
        return -torch.exp(torch.empty(D, N).uniform_(-9.2, 0.0, generator=g))
    A = -torch.exp(torch.empty(D, N).uniform_(-9.2, 2.5, generator=g))
    A[torch.rand(D, N, generator=g) < 0.1] = 0.0
    return A


def _scan_case(rng):
    N = rng.choice([1, 2, 3, 4, 5, 7, 8, 9, 12, 15, 16, 16, 32, 64])
    c = dict(seed=rng.randint(0, 10**9), B=rng.choice([1, 1, 2, 3]), N=N,
             D=rng.choice([rng.randint(1, 64), rng.randint(65, 500), 128 * rng.randint(1, 4)]),
             L=rng.choice([8 * rng.randint(1, 300), rng.randint(1, 300), rng.randint(300, 4000)]),
             in_bf=rng.random() < 0.7, conv=rng.choice([0, 0, 1, 2, 3, 4]), z=rng.random() < 0.7,
             Dsk=rng.random() < 0.7, bias=rng.random() < 0.8, sp=rng.random() < 0.85, zoh=rng.random() < 0.8,
             h0=rng.random() < 0.5, A=rng.choice(["s4d", "s4d", "small", "mixed"]), init=rng.random() < 0.4,
             states=rng.choice(["", "", "", "ckpt", "all"]))
    c["out_bf"] = c["in_bf"] if rng.random() < 0.8 else not c["in_bf"]
    if N > 16:   # only the packed bf16 kernels take 32 and 64 states
        c.update(in_bf=True, out_bf=True, L=max(8, c["L"] // 8 * 8), states="")
    if not c["out_bf"] and c["A"] != "s4d":   # fp32 outputs of slow states: small steps (dt bias on)
        c["bias"] = True
        c["L"] = min(c["L"], 2048)
    if not c["sp"]:
        c["L"] = min(c["L"], 1024)
    if c["B"] * c["D"] * c["L"] * N > 2e7:
        c["states"] = ""
    return c


def _run_scan_case(c, rng):
    Bsz, D, N, L, W = c["B"], c["D"], c["N"], c["L"], c["conv"]
    cfg = workloads.ScanConfig("random", Bsz, D, N, L, "bf16" if c["in_bf"] else "f32", conv=W > 0,
                               seed=c["seed"] % 100000)
    d = workloads.make_scan_inputs(cfg, with_h0=c["h0"])
    g = torch.Generator().manual_seed(c["seed"])
    d["A"] = _a(c["A"], D, N, g)
    for k, on in (("z", c["z"]), ("Dskip", c["Dsk"]), ("delta_bias", c["bias"])):
        if not on:
            d[k] = None
    if W:
        d["conv_w"] = d["conv_w"][:, 4 - W:].contiguous()
        d["conv_b"] = torch.randn(D, generator=g) * 0.2
        if c["init"] and W > 1:
            d["conv_init"] = torch.randn(Bsz, D, W - 1, generator=g).to(d["u"].dtype)
    if not c["sp"]:   # the step is taken as given: positive
        d["delta"] = (d["delta"].float().abs() * 0.05 + 1e-3).to(d["u"].dtype)
        d["delta_bias"] = None
    d["zoh"], d["delta_softplus"] = c["zoh"], c["sp"]
    gd = {k: (v.cuda().contiguous() if isinstance(v, torch.Tensor) else v) for k, v in d.items()}
    od = torch.bfloat16 if c["out_bf"] else torch.float32
    kw = dict(Dskip=gd.get("Dskip"), delta_bias=gd.get("delta_bias"), z=gd.get("z"), conv_w=gd.get("conv_w"),
              conv_b=gd.get("conv_b"), h0=gd.get("h0"), delta_softplus=c["sp"], zoh=c["zoh"], out_dtype=od,
              return_state=True, conv_init=gd.get("conv_init"))
    if c["states"] == "ckpt":
        kw["h_ckpt"] = torch.full((Bsz, ssm.ckpt_count(L), D, N), float("nan"), device="cuda")
    elif c["states"] == "all":
        kw["h_all"] = torch.full((Bsz, L, D, N), float("nan"), device="cuda")
    y, h = ssm.ssm_scan_fwd(gd["u"], gd["delta"], gd["A"], gd["Bm"], gd["Cm"], **kw)
    torch.cuda.synchronize()
    assert ssm.ssm_device_error() == 0
    R = Bsz * D
    idx = sorted(rng.sample(range(R), min(R, 48)))
    extra = {"h_all": True} if c["states"] else None
    ry, rh, _ = oracle.scan(d, rows=[(i // D, i % D) for i in idx], extra=extra)
    worst = max(_ratio(y.reshape(R, L)[idx], ry, y_tolerance(ry, od)),
                _ratio(h.reshape(R, N)[idx], rh, h_tolerance(rh, d["u"].dtype)))
    if c["states"]:
        ha = extra["h_all"]
        if c["states"] == "all":
            got = kw["h_all"].permute(0, 2, 1, 3).reshape(R, L, N)[idx]
            ref = ha
        else:
            steps = [min(8 * (j + 1), L) - 1 for j in range(ssm.ckpt_count(L))]
            got = kw["h_ckpt"].permute(0, 2, 1, 3).reshape(R, len(steps), N)[idx]
            ref = ha[:, steps, :]
        worst = max(worst, _ratio(got, ref, h_tolerance(ref, d["u"].dtype)))
    return worst


@pytest.mark.parametrize("block", range(4))
def test_random_scan_cases(block):
    rng = random.Random(7100 + block)
    for i in range(40):
        c = _scan_case(rng)
        r = _run_scan_case(c, rng)
        assert r <= 1.0, f"case {i} {c}: worst error {r:.3f} of the bound"


@pytest.mark.parametrize("block", range(2))
def test_random_backward_cases(block):
    rng = random.Random(7200 + block)
    for i in range(25):
        seed = rng.randint(0, 10**6)
        Bsz, D, N = rng.choice([1, 2]), rng.randint(1, 160), rng.randint(1, 16)
        L = rng.choice([rng.randint(1, 64), rng.randint(65, 300)])
        dt = rng.choice(["f32", "bf16"])
        W = rng.choice([0, 0, 2, 3, 4])
        z, zoh, sp, h0 = rng.random() < 0.6, rng.random() < 0.7, rng.random() < 0.8, rng.random() < 0.5
        cfg = workloads.SCAN_CONFIGS["mamba1.4b_conv" if W else "mamba130m"]
        d = workloads.make_scan_inputs(cfg, batch=Bsz, dim=D, seqlen=L, dstate=N, dtype=dt, with_h0=h0, seed=seed)
        g = torch.Generator().manual_seed(seed)
        d["zoh"], d["delta_softplus"] = zoh, sp
        if not z:
            d["z"] = None
        if not sp:
            d["delta"] = (0.02 + 0.05 * d["delta"].float().abs()).to(d["delta"].dtype)
            d["delta_bias"] = torch.full((D,), 0.01)
        if W:
            d["conv_w"] = d["conv_w"][:, 4 - W:].contiguous()
            d["conv_init"] = torch.randn((Bsz, D, W - 1), generator=g).to(d["u"].dtype)
        d["A"] = _a(rng.choice(["s4d", "small", "mixed"]), D, N, g)
        dy = torch.randn((Bsz, D, L), generator=g).to(d["u"].dtype)
        dh = torch.randn((Bsz, D, N), generator=g) * 0.3 if rng.random() < 0.5 else None
        grads, dyr = bwd_run(d, dy, dh)
        ref = obwd.scan_bwd(d, dyr, dh)
        bwd_compare(d, grads, ref, d["u"].dtype)


@pytest.mark.parametrize("block", range(2))
def test_random_decode_cases(block):
    rng = random.Random(7300 + block)
    for i in range(40):
        seed = rng.randint(0, 10**9)
        g = torch.Generator().manual_seed(seed)
        Bsz, D = rng.choice([1, 2, 7, 64, 256]), rng.choice([rng.randint(1, 300), 8 * rng.randint(1, 80)])
        N = rng.choice([1, 2, 4, 5, 8, 12, 16, 16, 32, 64])
        dt_ = rng.choice([torch.float32, torch.bfloat16])
        zoh, sp, has_z, has_d, has_b = (rng.random() < p for p in (0.8, 0.8, 0.7, 0.7, 0.7))
        W = rng.choice([0, 0, 1, 2, 3, 4])
        A = _a(rng.choice(["s4d", "small", "mixed"]), D, N, g)
        st = torch.randn((Bsz, D, N), generator=g) * 0.5
        Dskip = torch.randn(D, generator=g) if has_d else None
        bias = torch.log(torch.expm1(torch.empty(D).uniform_(1e-3, 1e-1, generator=g))) if (has_b and sp) else None
        cw = torch.randn((D, W), generator=g) * 0.5 if W else None
        cb = torch.randn(D, generator=g) * 0.1 if W else None
        cs = torch.randn((Bsz, D, W - 1), generator=g).to(dt_) if W > 1 else None
        st_g, cs_g = st.cuda(), (cs.cuda() if cs is not None else None)
        st_r, cs_r = st.double(), cs
        dev = {k: (v.cuda() if v is not None else None) for k, v in (("A", A), ("D", Dskip), ("b", bias), ("w", cw),
                                                                     ("cb", cb))}
        for k in range(rng.choice([1, 4, 12])):
            u = torch.randn((Bsz, D), generator=g).to(dt_)
            de = (torch.randn((Bsz, D), generator=g) * 0.5).to(dt_)
            if not sp:
                de = (de.float().abs() * 0.05 + 1e-3).to(dt_)
            Bm, Cm = torch.randn((Bsz, N), generator=g).to(dt_), torch.randn((Bsz, N), generator=g).to(dt_)
            z = torch.randn((Bsz, D), generator=g).to(dt_) if has_z else None
            y = ssm.ssm_state_update(st_g, u.cuda(), de.cuda(), dev["A"], Bm.cuda(), Cm.cuda(), Dskip=dev["D"],
                                     delta_bias=dev["b"], z=z.cuda() if z is not None else None, delta_softplus=sp,
                                     zoh=zoh, conv_w=dev["w"], conv_b=dev["cb"], conv_state=cs_g)
            res = oracle.state_update(st_r, u, de, A, Bm, Cm, Dskip, bias, z, zoh=zoh, delta_softplus=sp, conv_w=cw,
                                      conv_b=cb, conv_state=cs_r)
            st_r, y_r = res[0], res[1]
            if W > 1:
                cs_r = torch.from_numpy(np.ascontiguousarray(res[2])).to(dt_)
            r = _ratio(y, y_r, y_tolerance(y_r, dt_))
            assert r <= 1.0, f"case {i} step {k}: y at {r:.3f} of the bound"
        r = _ratio(st_g, np.asarray(st_r), h_tolerance(np.asarray(st_r), dt_))
        assert r <= 1.0, f"case {i}: state at {r:.3f} of the bound"
        assert ssm.ssm_device_error() == 0


@pytest.mark.parametrize("block", range(2))
def test_random_ssd_cases(block):
    rng = random.Random(7400 + block)
    for i in range(25):
        seed = rng.randint(0, 10**6)
        Bsz, G = rng.choice([1, 2, 3]), rng.choice([1, 2, 4])
        H, N, L = G * rng.choice([1, 2, 3]), rng.choice([64, 128]), 8 * rng.randint(1, 100)
        flags = dict(z=rng.random() < 0.6, h0=rng.random() < 0.5, zoh=rng.random() < 0.5, softplus=rng.random() < 0.8)
        d = ssd_small(L, G, seed, H=H, Bsz=Bsz, N=N, **flags)
        if rng.random() < 0.2:
            d["A"][rng.randrange(H)] = 0.0
        y, h = ssd_run(d)
        ref_y, ref_h, _ = ssd_scan(d)
        _check_y(y, ref_y.reshape(y.shape), f"case {i} y")
        r = _ratio(h, ref_h.reshape(h.shape), h_tolerance(ref_h.reshape(h.shape), torch.bfloat16))
        assert r <= 1.0, f"case {i}: h_out at {r:.3f} of the bound"


@pytest.mark.parametrize("block", range(2))
def test_random_slot_cases(block):
    """Scan and decode on per-request state slots (state_indices): random batch-to-slot maps with padding
    rows, conv widths 0 to 4 with the conv history kept in a slot cache too; unused slots must come back
    bit-identical and a padding row's y zero."""
    rng = random.Random(7500 + block)
    for i in range(40):
        seed = rng.randint(0, 10**9)
        g = torch.Generator().manual_seed(seed)
        Bsz = rng.randint(1, 9)
        S = Bsz + rng.randint(0, 6)
        D, N = rng.choice([rng.randint(1, 200), 8 * rng.randint(1, 40)]), rng.randint(1, 16)
        L = rng.choice([1, rng.randint(1, 40), rng.randint(41, 600)])
        dt, W, which = rng.choice(["f32", "bf16"]), rng.choice([0, 0, 1, 2, 3, 4]), rng.choice(["scan", "decode"])
        idx = torch.tensor([s if rng.random() > 0.2 else -1 for s in rng.sample(range(S), Bsz)], dtype=torch.int32)
        d = workloads.make_scan_inputs(workloads.ScanConfig("slots", Bsz, D, N, L, dt, conv=W > 0, seed=seed % 100000))
        if W:
            d["conv_w"] = d["conv_w"][:, 4 - W:].contiguous()
        idt = d["u"].dtype
        cache = torch.randn((S, D, N), generator=g) * 0.5
        cc = torch.randn((S, D, W - 1), generator=g).to(idt) if W > 1 else None
        cache_d, cc_d = cache.cuda(), (cc.cuda() if cc is not None else None)
        live = [b for b in range(Bsz) if idx[b] >= 0]
        li = idx[live].long()
        what = f"case {i} ({which}, B {Bsz}, S {S}, D {D}, N {N}, L {L}, {dt}, W {W}, slots {idx.tolist()})"
        if which == "scan":
            gd = {k: (v.cuda().contiguous() if isinstance(v, torch.Tensor) else v) for k, v in d.items()}
            y = ssm.ssm_scan_fwd(gd["u"], gd["delta"], gd["A"], gd["Bm"], gd["Cm"], Dskip=gd["Dskip"],
                                 delta_bias=gd["delta_bias"], z=gd["z"], conv_w=gd.get("conv_w"),
                                 conv_b=gd.get("conv_b"), h0=cache_d, h_out=cache_d, state_indices=idx.cuda(),
                                 conv_init=cc_d, conv_final=cc_d)
            torch.cuda.synchronize()
            if live:
                sub = {k: (v[live] if isinstance(v, torch.Tensor) and v.dim() == 3 and v.shape[0] == Bsz else v)
                       for k, v in d.items()}
                sub["h0"] = cache[li]
                if cc is not None:
                    sub["conv_init"] = cc[li]
                yr, hr, _ = oracle.scan(sub)
                yr, hr = yr.reshape(len(live), D, L), hr.reshape(len(live), D, N)
                assert _ratio(y[live], yr, y_tolerance(yr, idt)) <= 1.0, what + ": y"
                assert _ratio(cache_d.cpu()[li], hr, h_tolerance(hr, idt)) <= 1.0, what + ": slot states"
            assert all(bool((y[b] == 0).all()) for b in range(Bsz) if idx[b] < 0), what + ": padding y"
            if cc is not None:
                for b in live:
                    want = torch.cat([cc[int(idx[b])], d["u"][b]], dim=-1)[:, -(W - 1):]
                    assert torch.equal(cc_d.cpu()[int(idx[b])], want), what + ": conv history"
        else:
            x, de, z = (d[k][..., 0].contiguous() for k in ("u", "delta", "z"))
            Bm, Cm = d["Bm"][..., 0].contiguous(), d["Cm"][..., 0].contiguous()
            y = ssm.ssm_state_update(cache_d, x.cuda(), de.cuda(), d["A"].cuda(), Bm.cuda(), Cm.cuda(),
                                     Dskip=d["Dskip"].cuda(), delta_bias=d["delta_bias"].cuda(), z=z.cuda(),
                                     conv_w=d["conv_w"].cuda() if W else None,
                                     conv_b=d["conv_b"].cuda() if W else None, conv_state=cc_d,
                                     state_indices=idx.cuda())
            torch.cuda.synchronize()
            if live:
                kw = dict(conv_w=d["conv_w"], conv_b=d["conv_b"],
                          conv_state=cc[li] if cc is not None else None) if W else {}
                out = oracle.state_update(cache[li], x[live], de[live], d["A"], Bm[live], Cm[live], d["Dskip"],
                                          d["delta_bias"], z[live], **kw)
                assert _ratio(y[live], out[1], y_tolerance(out[1], idt)) <= 1.0, what + ": y"
                assert _ratio(cache_d.cpu()[li], out[0], h_tolerance(out[0], idt)) <= 1.0, what + ": slot states"
        unused = sorted(set(range(S)) - set(li.tolist()))
        assert torch.equal(cache_d.cpu()[unused], cache[unused]), what + ": an unused slot changed"
        if cc is not None:
            assert torch.equal(cc_d.cpu()[unused], cc[unused]), what + ": an unused conv slot changed"
        assert ssm.ssm_device_error() == 0
