"""Pins for the CPU oracle: checks against what the pages and the mathematics fix, with no GPU.

Each pin computes its expectation by a route that does not reuse the oracle's recurrence:
closed forms (convolution and semiseparable forms, geometric series), an ODE integration of the
continuous system under a zero-order hold, brute force, algebraic invariants, and library
routines (torch conv1d / softplus / silu in fp64).  A plausible slip in the oracle -- a dropped
term, an off-by-one in the product range, a transposed B/C index, the wrong ZOH factor, the wrong
conv tap orientation, the gate applied before the D skip -- fails at least one of them.
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle
import workloads

pytestmark = pytest.mark.cpu

RNG = np.random.default_rng(12345)


def _inputs(Bsz, D, N, L, *, zoh=True, with_z=False, with_D=True, conv=False, h0=False, seed=0,
            const_in_time=False, delta_softplus=True):
    g = np.random.default_rng(seed)
    d = {}
    d["u"] = torch.tensor(g.standard_normal((Bsz, D, L)))
    if const_in_time:
        d["delta"] = torch.tensor(np.repeat(0.5 * g.standard_normal((Bsz, D, 1)), L, axis=2))
        d["Bm"] = torch.tensor(np.repeat(g.standard_normal((Bsz, N, 1)), L, axis=2))
        d["Cm"] = torch.tensor(np.repeat(g.standard_normal((Bsz, N, 1)), L, axis=2))
    else:
        d["delta"] = torch.tensor(0.5 * g.standard_normal((Bsz, D, L)))
        d["Bm"] = torch.tensor(g.standard_normal((Bsz, N, L)))
        d["Cm"] = torch.tensor(g.standard_normal((Bsz, N, L)))
    d["A"] = torch.tensor(-np.tile(np.arange(1, N + 1, dtype=np.float64), (D, 1)) * (0.5 + g.random((D, 1))))
    d["Dskip"] = torch.tensor(g.standard_normal(D)) if with_D else None
    d["delta_bias"] = torch.tensor(np.log(np.expm1(1e-3 + (1e-1 - 1e-3) * g.random(D))))
    d["z"] = torch.tensor(g.standard_normal((Bsz, D, L))) if with_z else None
    d["conv_w"] = torch.tensor(0.5 * g.standard_normal((D, 4))) if conv else None
    d["conv_b"] = torch.tensor(0.1 * g.standard_normal(D)) if conv else None
    d["h0"] = torch.tensor(0.5 * g.standard_normal((Bsz, D, N))) if h0 else None
    d["zoh"] = zoh
    d["delta_softplus"] = delta_softplus
    return d


def _np(d, k):
    v = d[k]
    return None if v is None else v.numpy().astype(np.float64)


def _softplus_torch(x):
    # library routine (fp64); threshold far above any input used here so it is the exact function
    return torch.nn.functional.softplus(torch.as_tensor(x, dtype=torch.float64), threshold=1e9).numpy()


def _silu_torch(x):
    return torch.nn.functional.silu(torch.as_tensor(x, dtype=torch.float64)).numpy()


def _disc(d):
    """Abar (B,D,N,L) and Bbar (B,D,N,L), the step sizes (B,D,L), from the definitions.

    Bbar for the zero-order hold is taken from the matrix-exponential form (dt A)^-1 (exp(dt A) - I) dt B
    evaluated with scipy's expm on each diagonal entry's 1x1 block -- not from expm1 -- so this
    helper does not retype the oracle's formula."""
    from scipy.linalg import expm
    dt_raw = _np(d, "delta") + _np(d, "delta_bias")[None, :, None]
    dt = _softplus_torch(dt_raw) if d["delta_softplus"] else dt_raw
    A = _np(d, "A")
    Bm = _np(d, "Bm")
    Bsz, D, L = dt.shape
    N = A.shape[1]
    Abar = np.exp(dt[:, :, None, :] * A[None, :, :, None])
    if d["zoh"]:
        fac = np.empty_like(Abar)
        for idx in np.ndindex(Bsz, D, N, L):
            b, dd, n, t = idx
            M = np.array([[dt[b, dd, t] * A[dd, n]]])
            fac[idx] = (np.linalg.solve(M, expm(M) - np.eye(1)) * dt[b, dd, t])[0, 0]
        Bbar = fac * Bm[:, None, :, :]
    else:
        Bbar = dt[:, :, None, :] * Bm[:, None, :, :]
    return Abar, Bbar, dt


# ---------------------------------------------------------------------------------------------
# P0: golden worked example (hand-derived from the page's convolution-mode expansion)
# ---------------------------------------------------------------------------------------------
def test_golden_impulse_response():
    path = os.path.join(os.path.dirname(__file__), "golden", "impulse_response.txt")
    rows = [l.split() for l in open(path) if l.strip() and not l.startswith("#")]
    for r in rows:
        zoh = bool(int(r[0]))
        want = np.array([float(v) for v in r[1:]])
        d = {
            "u": torch.tensor([[[1.0, 0.0, 0.0, 0.0]]], dtype=torch.float64),
            "delta": torch.ones((1, 1, 4), dtype=torch.float64),
            "Bm": torch.ones((1, 1, 4), dtype=torch.float64),
            "Cm": torch.ones((1, 1, 4), dtype=torch.float64),
            "A": torch.tensor([[-math.log(2.0)]], dtype=torch.float64),
            "Dskip": None, "delta_bias": None, "z": None, "conv_w": None, "conv_b": None, "h0": None,
            "zoh": zoh, "delta_softplus": False,
        }
        y, h, _ = oracle.scan(d)
        np.testing.assert_allclose(y[0], want, rtol=1e-15, atol=1e-16)


# ---------------------------------------------------------------------------------------------
# P1: LTI case equals the convolution form y = K * u, K_k = sum_n C Abar^k Bbar (O(L^2) brute force)
# ---------------------------------------------------------------------------------------------
@pytest.mark.parametrize("zoh", [True, False])
def test_p1_lti_convolution_form(zoh):
    d = _inputs(2, 3, 4, 40, zoh=zoh, const_in_time=True, seed=1)
    y, _, _ = oracle.scan(d)
    Abar, Bbar, _ = _disc(d)
    C = _np(d, "Cm")
    u = _np(d, "u")
    Dk = _np(d, "Dskip")
    Bsz, D, L = u.shape
    want = np.zeros((Bsz, D, L))
    for b in range(Bsz):
        for dd in range(D):
            a = Abar[b, dd, :, 0]
            bb = Bbar[b, dd, :, 0]
            c = C[b, :, 0]
            K = np.array([np.sum(c * a ** k * bb) for k in range(L)])
            for t in range(L):
                want[b, dd, t] = sum(K[k] * u[b, dd, t - k] for k in range(t + 1)) + Dk[dd] * u[b, dd, t]
    np.testing.assert_allclose(y.reshape(Bsz, D, L), want, rtol=1e-11, atol=1e-12)


# ---------------------------------------------------------------------------------------------
# P2: time-varying semiseparable closed form (no recurrence), O(L^2 N)
# ---------------------------------------------------------------------------------------------
@pytest.mark.parametrize("zoh", [True, False])
def test_p2_semiseparable_form(zoh):
    d = _inputs(1, 3, 4, 24, zoh=zoh, seed=2)
    y, _, _ = oracle.scan(d)
    Abar, Bbar, _ = _disc(d)
    C = _np(d, "Cm")
    u = _np(d, "u")
    Dk = _np(d, "Dskip")
    _, D, L = u.shape
    want = np.zeros((D, L))
    for dd in range(D):
        for t in range(L):
            acc = 0.0
            for i in range(t + 1):
                prod = np.prod(Abar[0, dd, :, i + 1:t + 1], axis=1)   # empty product = 1 when i == t
                acc += np.sum(C[0, :, t] * prod * Bbar[0, dd, :, i]) * u[0, dd, i]
            want[dd, t] = acc + Dk[dd] * u[0, dd, t]
    np.testing.assert_allclose(y, want, rtol=1e-11, atol=1e-12)


# ---------------------------------------------------------------------------------------------
# P11: zero-order hold = exact solution of h' = A h + B x with x held constant over each step
# ---------------------------------------------------------------------------------------------
def test_p11_zoh_matches_continuous_ode():
    from scipy.integrate import solve_ivp
    d = _inputs(1, 2, 3, 12, zoh=True, h0=True, with_D=False, seed=11)
    y, h_out, _ = oracle.scan(d)
    _, _, dt = _disc(d)
    A = _np(d, "A")
    Bm = _np(d, "Bm")
    C = _np(d, "Cm")
    u = _np(d, "u")
    h0 = _np(d, "h0")
    for dd in range(2):
        h = h0[0, dd].copy()
        for t in range(12):
            rhs = lambda s, hh: A[dd] * hh + Bm[0, :, t] * u[0, dd, t]
            sol = solve_ivp(rhs, (0.0, dt[0, dd, t]), h, method="DOP853", rtol=1e-13, atol=1e-15)
            h = sol.y[:, -1]
            np.testing.assert_allclose(y[dd, t], np.sum(C[0, :, t] * h), rtol=1e-9, atol=1e-12)
        np.testing.assert_allclose(h_out[dd], h, rtol=1e-9, atol=1e-12)


# ---------------------------------------------------------------------------------------------
# P3: dt -> 0 keeps the state (the "small dt keeps history" statement of section 4.1)
# ---------------------------------------------------------------------------------------------
@pytest.mark.parametrize("zoh", [True, False])
def test_p3_small_dt_keeps_state(zoh):
    d = _inputs(2, 4, 8, 16, zoh=zoh, h0=True, seed=3)
    d["delta"] = torch.full_like(d["delta"], -60.0)
    _, h_out, _ = oracle.scan(d)
    np.testing.assert_allclose(h_out.reshape(2, 4, 8), _np(d, "h0"), rtol=0, atol=1e-12)


# ---------------------------------------------------------------------------------------------
# P4: with no gate and zero initial state the map u -> y is linear
# ---------------------------------------------------------------------------------------------
@pytest.mark.parametrize("zoh", [True, False])
def test_p4_linear_in_u(zoh):
    d1 = _inputs(2, 3, 4, 32, zoh=zoh, seed=4)
    d2 = dict(d1)
    d2["u"] = torch.tensor(np.random.default_rng(44).standard_normal(d1["u"].shape))
    a, b = 0.7, -1.3
    d3 = dict(d1)
    d3["u"] = a * d1["u"] + b * d2["u"]
    y1, _, _ = oracle.scan(d1)
    y2, _, _ = oracle.scan(d2)
    y3, _, _ = oracle.scan(d3)
    np.testing.assert_allclose(y3, a * y1 + b * y2, rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------------------------------------
# P5: splitting L into two runs with the final state carried equals one run (segment state passing)
# ---------------------------------------------------------------------------------------------
@pytest.mark.parametrize("zoh", [True, False])
def test_p5_split_invariance(zoh):
    d = _inputs(2, 3, 4, 50, zoh=zoh, with_z=True, h0=True, seed=5)
    y, h, _ = oracle.scan(d)
    L1 = 17

    def part(lo, hi, h0):
        p = dict(d)
        for k in ("u", "delta", "z", "Bm", "Cm"):
            p[k] = d[k][..., lo:hi].contiguous()
        p["h0"] = h0
        return p

    ya, ha, _ = oracle.scan(part(0, L1, d["h0"]))
    yb, hb, _ = oracle.scan(part(L1, 50, torch.tensor(ha.reshape(2, 3, 4))))
    np.testing.assert_allclose(np.concatenate([ya, yb], axis=1), y, rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(hb, h, rtol=1e-13, atol=1e-14)


# ---------------------------------------------------------------------------------------------
# P6: ZOH step response is a geometric series whose limit -B/A does not depend on dt
# ---------------------------------------------------------------------------------------------
def test_p6_zoh_step_response_dc_gain():
    L = 4000
    for dt in (0.01, 0.1):
        d = {
            "u": torch.ones((1, 1, L), dtype=torch.float64),
            "delta": torch.full((1, 1, L), dt, dtype=torch.float64),
            "Bm": torch.tensor([[[1.5]], [[-0.25]]], dtype=torch.float64).reshape(1, 2, 1).repeat(1, 1, L),
            "Cm": torch.zeros((1, 2, L), dtype=torch.float64),
            "A": torch.tensor([[-1.0, -3.0]], dtype=torch.float64),
            "Dskip": None, "delta_bias": None, "z": None, "conv_w": None, "conv_b": None, "h0": None,
            "zoh": True, "delta_softplus": False,
        }
        # states after t steps: Bbar * (1 - Abar^t) / (1 - Abar); check t = 7 and the limit
        d7 = dict(d)
        for k in ("u", "delta", "Bm", "Cm"):
            d7[k] = d[k][..., :7].contiguous()
        _, h7, _ = oracle.scan(d7)
        _, hL, _ = oracle.scan(d)
        A = np.array([-1.0, -3.0])
        B = np.array([1.5, -0.25])
        Abar = np.exp(dt * A)
        # Bbar from its own definition as the integral of exp(A s) B over one step (Simpson, fine grid)
        s = np.linspace(0.0, dt, 20001)
        w = np.ones_like(s); w[1:-1:2] = 4; w[2:-1:2] = 2
        Bbar = np.array([np.sum(w * np.exp(a * (dt - s))) * (s[1] - s[0]) / 3 for a in A]) * B
        np.testing.assert_allclose(h7[0], Bbar * (1 - Abar ** 7) / (1 - Abar), rtol=1e-10)
        np.testing.assert_allclose(hL[0], -B / A, rtol=1e-10)


# ---------------------------------------------------------------------------------------------
# P7: ZOH and the simplified Bbar = dt B agree to first order: ratio expm1(x)/x -> 1 as x = dt A -> 0
# ---------------------------------------------------------------------------------------------
def test_p7_zoh_vs_simplified_first_order():
    for dt in (1e-2, 1e-4, 1e-6):
        d = {
            "u": torch.ones((1, 1, 1), dtype=torch.float64),
            "delta": torch.full((1, 1, 1), dt, dtype=torch.float64),
            "Bm": torch.ones((1, 3, 1), dtype=torch.float64),
            "Cm": torch.zeros((1, 3, 1), dtype=torch.float64),
            "A": torch.tensor([[-1.0, -4.0, -16.0]], dtype=torch.float64),
            "Dskip": None, "delta_bias": None, "z": None, "conv_w": None, "conv_b": None, "h0": None,
            "delta_softplus": False,
        }
        _, hz, _ = oracle.scan(dict(d, zoh=True))
        _, hs, _ = oracle.scan(dict(d, zoh=False))
        x = dt * np.array([-1.0, -4.0, -16.0])
        series = sum(x ** k / math.factorial(k + 1) for k in range(12))   # expm1(x)/x as its Taylor series
        np.testing.assert_allclose(hs[0], dt, rtol=1e-15)
        np.testing.assert_allclose(hz[0] / hs[0], series, rtol=1e-9)


def test_zoh_zero_A_limit_is_simplified():
    d = _inputs(1, 2, 3, 20, zoh=True, seed=71)
    d["A"] = torch.zeros_like(d["A"])
    yz, hz, _ = oracle.scan(d)
    ys, hs, _ = oracle.scan(dict(d, zoh=False))
    np.testing.assert_allclose(yz, ys, rtol=1e-15)
    np.testing.assert_allclose(hz, hs, rtol=1e-15)


# ---------------------------------------------------------------------------------------------
# P8: L single-token decode steps equal one scan of length L (recurrent/convolution duality)
# ---------------------------------------------------------------------------------------------
@pytest.mark.parametrize("zoh", [True, False])
def test_p8_decode_equals_scan(zoh):
    d = _inputs(3, 4, 8, 20, zoh=zoh, with_z=True, h0=True, seed=8)
    y, h, _ = oracle.scan(d)
    st = d["h0"].clone()
    ys = []
    for t in range(20):
        st_np, yt = oracle.state_update(st, d["u"][..., t], d["delta"][..., t], d["A"], d["Bm"][..., t],
                                        d["Cm"][..., t], d["Dskip"], d["delta_bias"], d["z"][..., t], zoh=zoh)
        st = torch.tensor(st_np)
        ys.append(yt)
    np.testing.assert_allclose(np.stack(ys, axis=-1).reshape(12, 20), y, rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(st.numpy().reshape(12, 8), h, rtol=1e-13, atol=1e-14)


# ---------------------------------------------------------------------------------------------
# P9: the conv front end equals torch's conv1d(padding=W-1, groups=D)[..., :L] followed by SiLU
# ---------------------------------------------------------------------------------------------
def test_p9_conv_front_end_matches_library_conv1d():
    d = _inputs(2, 5, 4, 33, conv=True, seed=9)
    x = d["u"]
    ref = torch.nn.functional.conv1d(x, d["conv_w"][:, None, :], d["conv_b"], padding=3, groups=5)[..., :33]
    got = oracle.conv1d(x, d["conv_w"], d["conv_b"], silu=False)
    np.testing.assert_allclose(got.reshape(2, 5, 33), ref.numpy(), rtol=1e-13, atol=1e-14)
    got_s = oracle.conv1d(x, d["conv_w"], d["conv_b"], silu=True)
    np.testing.assert_allclose(got_s.reshape(2, 5, 33), _silu_torch(ref.numpy()), rtol=1e-13, atol=1e-14)
    # the fused scan equals the unfused scan of SiLU(conv(x))
    y_fused, h_fused, _ = oracle.scan(d)
    d2 = dict(d, conv_w=None, conv_b=None, u=torch.tensor(_silu_torch(ref.numpy())))
    y_plain, h_plain, _ = oracle.scan(d2)
    np.testing.assert_allclose(y_fused, y_plain, rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(h_fused, h_plain, rtol=1e-13, atol=1e-14)


# ---------------------------------------------------------------------------------------------
# P12: conv history carried across calls.  With conv_init (the W-1 inputs before t = 0) the front end
# equals torch's conv1d over the history and x concatenated; conv_final returns the last W-1 inputs;
# and a split run that passes conv_final and h_out on equals one run (dpshk.com/news/5205047 1.3,
# pwwt.cn/news/5168881 3.1: the carried state of a chunked prefill)
# ---------------------------------------------------------------------------------------------
@pytest.mark.parametrize("W", [2, 3, 4])
def test_p12_conv_history_matches_library_conv1d(W):
    d = _inputs(2, 5, 4, 19, conv=True, seed=12 + W)
    d["conv_w"] = d["conv_w"][:, :W].contiguous()
    g = np.random.default_rng(40 + W)
    hist = torch.tensor(g.standard_normal((2, 5, W - 1)))
    d["conv_init"] = hist
    full = torch.cat([hist, d["u"]], dim=-1)
    ref = torch.nn.functional.conv1d(full, d["conv_w"][:, None, :], d["conv_b"], groups=5)  # valid: length L
    assert ref.shape[-1] == 19
    extra = {}
    y_fused, h_fused, _ = oracle.scan(d, extra=extra)
    d2 = dict(d, conv_w=None, conv_b=None, conv_init=None, u=torch.tensor(_silu_torch(ref.numpy())))
    y_plain, h_plain, _ = oracle.scan(d2)
    np.testing.assert_allclose(y_fused, y_plain, rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(h_fused, h_plain, rtol=1e-13, atol=1e-14)
    np.testing.assert_array_equal(extra["conv_final"], full[..., -(W - 1):].reshape(10, W - 1).numpy())


@pytest.mark.parametrize("L1", [1, 2, 3, 7, 16])
def test_p12_split_with_conv_history_equals_one_run(L1):
    L = 23
    d = _inputs(2, 3, 4, L, conv=True, with_z=True, h0=True, seed=120 + L1)
    y, h, _ = oracle.scan(d)
    first = dict(d, u=d["u"][..., :L1], delta=d["delta"][..., :L1], z=d["z"][..., :L1], Bm=d["Bm"][..., :L1],
                 Cm=d["Cm"][..., :L1])
    e1 = {}
    y1, h1, _ = oracle.scan(first, extra=e1)
    second = dict(d, u=d["u"][..., L1:], delta=d["delta"][..., L1:], z=d["z"][..., L1:], Bm=d["Bm"][..., L1:],
                  Cm=d["Cm"][..., L1:], h0=torch.tensor(h1.reshape(2, 3, 4)),
                  conv_init=torch.tensor(e1["conv_final"].reshape(2, 3, 3)))
    e2 = {}
    y2, h2, _ = oracle.scan(second, extra=e2)
    np.testing.assert_allclose(np.concatenate([y1, y2], axis=1), y, rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(h2, h, rtol=1e-13, atol=1e-14)
    np.testing.assert_array_equal(e2["conv_final"], d["u"][..., -3:].reshape(6, 3).numpy())


# ---------------------------------------------------------------------------------------------
# P13: decode with a conv state: L single-token steps that carry (conv state, SSM state) equal one
# fused scan of length L (datadaily.news "State space models vs Transformer: a practical guide";
# lshu.cn/news/79586 6.5: the cache holds the conv and the SSM state)
# ---------------------------------------------------------------------------------------------
@pytest.mark.parametrize("W", [1, 2, 4])
def test_p13_decode_with_conv_state_equals_fused_scan(W):
    L = 12
    d = _inputs(2, 3, 4, L, conv=True, with_z=True, h0=True, seed=130 + W)
    d["conv_w"] = d["conv_w"][:, :W].contiguous()
    y, h, _ = oracle.scan(d)
    st = d["h0"].clone()
    cs = torch.zeros((2, 3, max(W - 1, 1)), dtype=torch.float64)[..., :W - 1]
    ys = []
    for t in range(L):
        st_np, yt, cs_np = oracle.state_update(st, d["u"][..., t], d["delta"][..., t], d["A"], d["Bm"][..., t],
                                               d["Cm"][..., t], d["Dskip"], d["delta_bias"], d["z"][..., t],
                                               conv_w=d["conv_w"], conv_b=d["conv_b"], conv_state=cs)
        st, cs = torch.tensor(st_np), torch.tensor(np.ascontiguousarray(cs_np))
        ys.append(yt)
    np.testing.assert_allclose(np.stack(ys, axis=-1).reshape(6, L), y, rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(st.numpy().reshape(6, 4), h, rtol=1e-13, atol=1e-14)
    if W > 1:
        np.testing.assert_array_equal(cs.numpy(), d["u"][..., -(W - 1):].numpy())


# ---------------------------------------------------------------------------------------------
# P14: the state sequence of a multi-token verification pass (pwwt.cn/news/5168881 3.4): the state
# after step t equals the final state of the same scan cut after t + 1 steps
# ---------------------------------------------------------------------------------------------
def test_p14_state_sequence_equals_truncated_runs():
    L = 9
    d = _inputs(2, 3, 4, L, with_z=True, h0=True, seed=14)
    extra = {"h_all": True}
    y, h, _ = oracle.scan(d, extra=extra)
    for t in range(L):
        cut = dict(d, u=d["u"][..., :t + 1], delta=d["delta"][..., :t + 1], z=d["z"][..., :t + 1],
                   Bm=d["Bm"][..., :t + 1], Cm=d["Cm"][..., :t + 1])
        _, ht, _ = oracle.scan(cut)
        np.testing.assert_array_equal(extra["h_all"][:, t, :], ht)
    np.testing.assert_array_equal(extra["h_all"][:, -1, :], h)
    # and the closed form of the state sequence, h_t = prod_{j<=t} Abar_j h0 + sum_{i<=t} prod_{i<j<=t} Abar_j
    # Bbar_i u_i, from the definitions (no recurrence)
    Abar, Bbar, _ = _disc(d)
    u = _np(d, "u")
    h0 = _np(d, "h0")
    ref = np.zeros((2, 3, L, 4))
    for t in range(L):
        acc = np.prod(Abar[..., :t + 1], axis=-1) * h0
        for i in range(t + 1):
            acc = acc + np.prod(Abar[..., i + 1:t + 1], axis=-1) * Bbar[..., i] * u[:, :, None, i]
        ref[:, :, t, :] = acc
    np.testing.assert_allclose(extra["h_all"].reshape(2, 3, L, 4), ref, rtol=1e-11, atol=1e-12)


# ---------------------------------------------------------------------------------------------
# P10: N = 1, no D, simplified Bbar: scalar closed form y_k = c_k sum_i (prod_{j=i+1..k} a_j) b_i x_i
# ---------------------------------------------------------------------------------------------
def test_p10_scalar_closed_form():
    d = _inputs(1, 1, 1, 30, zoh=False, with_D=False, seed=10)
    y, _, _ = oracle.scan(d)
    dt = _softplus_torch(_np(d, "delta")[0, 0] + _np(d, "delta_bias")[0])
    a = np.exp(dt * _np(d, "A")[0, 0])
    b = dt * _np(d, "Bm")[0, 0]
    c = _np(d, "Cm")[0, 0]
    x = _np(d, "u")[0, 0]
    want = [c[k] * sum(np.prod(a[i + 1:k + 1]) * b[i] * x[i] for i in range(k + 1)) for k in range(30)]
    np.testing.assert_allclose(y[0], want, rtol=1e-12, atol=1e-14)


# ---------------------------------------------------------------------------------------------
# softplus and the SiLU gate against torch's fp64 library routines; gate applied after the D skip
# ---------------------------------------------------------------------------------------------
def test_softplus_and_gate_order():
    g = np.random.default_rng(13)
    L = 64
    raw = g.uniform(-30, 30, L)
    bias = 0.37
    # N = 1, A = -1, B = 1, u = 1, zero state, simplified Bbar, L = 1 per row: h_out = softplus(raw + bias)
    d = {
        "u": torch.ones((1, L, 1), dtype=torch.float64),
        "delta": torch.tensor(raw.reshape(1, L, 1)),
        "Bm": torch.ones((1, 1, 1), dtype=torch.float64),
        "Cm": torch.zeros((1, 1, 1), dtype=torch.float64),
        "A": -torch.ones((L, 1), dtype=torch.float64),
        "Dskip": None, "delta_bias": torch.full((L,), bias, dtype=torch.float64),
        "z": None, "conv_w": None, "conv_b": None, "h0": None, "zoh": False, "delta_softplus": True,
    }
    _, h, _ = oracle.scan(d)
    np.testing.assert_allclose(h[:, 0], _softplus_torch(raw + bias), rtol=1e-14)
    # gate: y = (C h + D u) * silu(z)
    u = g.standard_normal(L)
    z = g.uniform(-20, 20, L)
    d2 = {
        "u": torch.tensor(u.reshape(1, 1, L)), "delta": torch.zeros((1, 1, L), dtype=torch.float64),
        "Bm": torch.ones((1, 1, L), dtype=torch.float64), "Cm": torch.full((1, 1, L), 2.0, dtype=torch.float64),
        "A": torch.tensor([[-1.0]], dtype=torch.float64), "Dskip": torch.tensor([0.75], dtype=torch.float64),
        "delta_bias": None, "z": torch.tensor(z.reshape(1, 1, L)), "conv_w": None, "conv_b": None, "h0": None,
        "zoh": False, "delta_softplus": False,
    }
    y, _, _ = oracle.scan(d2)   # dt = 0: h stays 0, y = D u silu(z)
    np.testing.assert_allclose(y[0], 0.75 * u * _silu_torch(z), rtol=1e-14, atol=1e-300)


def test_rows_subset_matches_full():
    cfg = workloads.SCAN_CONFIGS["tiny"]
    d = workloads.make_scan_inputs(cfg, batch=2, dim=8, seqlen=37, with_h0=True)
    y, h, _ = oracle.scan(d)
    rows = [(1, 5), (0, 0), (1, 7)]
    ys, hs, _ = oracle.scan(d, rows=rows)
    for i, (b, dd) in enumerate(rows):
        np.testing.assert_array_equal(ys[i], y[b * 8 + dd])
        np.testing.assert_array_equal(hs[i], h[b * 8 + dd])


def test_threads_do_not_change_results():
    cfg = workloads.SCAN_CONFIGS["tiny"]
    d = workloads.make_scan_inputs(cfg, batch=3, dim=16, seqlen=64)
    y1, h1, n1 = oracle.scan(d, nthreads=1)
    y8, h8, n8 = oracle.scan(d, nthreads=8)
    assert n1 == 1
    np.testing.assert_array_equal(y1, y8)
    np.testing.assert_array_equal(h1, h8)


# ---------------------------------------------------------------------------------------------
# Backward oracle (autograd of a plain fp64 torch recurrence) against central finite differences of
# the C forward oracle: d/dp of sum(y * dy) + sum(h_L * dh) for every input p, at sampled coordinates
# ---------------------------------------------------------------------------------------------
def _objective(d, dy, dh):
    y, h, _ = oracle.scan(d, nthreads=1)
    Bsz, D, L = d["u"].shape
    return float((y.reshape(Bsz, D, L) * dy).sum() + (h.reshape(dh.shape) * dh).sum())


@pytest.mark.parametrize("zoh,conv,softplus", [(True, True, True), (False, False, True), (True, False, False)])
def test_backward_oracle_matches_finite_differences(zoh, conv, softplus):
    from oracle import backward as bwd
    Bsz, D, N, L = 2, 3, 4, 7
    d = _inputs(Bsz, D, N, L, zoh=zoh, with_z=True, conv=conv, h0=True, seed=200 + int(zoh) + 2 * int(conv),
                delta_softplus=softplus)
    d["A"][1, 2] = 0.0  # the a -> 0 limit and its derivative
    if not softplus:  # dt = delta + bias directly: keep it positive, as a step size is
        d["delta"] = 0.02 + 0.1 * d["delta"].abs()
        d["delta_bias"] = torch.full((D,), 0.01, dtype=torch.float64)
    if conv:
        d["conv_init"] = torch.tensor(np.random.default_rng(5).standard_normal((Bsz, D, 3)))
    g = np.random.default_rng(21)
    dy = g.standard_normal((Bsz, D, L))
    dh = g.standard_normal((Bsz, D, N))
    grads = bwd.scan_bwd(d, dy, dh)
    y_ref, _, _ = oracle.scan(d, nthreads=1)
    np.testing.assert_allclose(grads["y"].reshape(-1, L), y_ref, rtol=1e-12, atol=1e-13)
    keys = ["u", "delta", "A", "Bm", "Cm", "Dskip", "delta_bias", "z", "h0"] + (["conv_w", "conv_b", "conv_init"]
                                                                                if conv else [])
    eps = 1e-6
    for k in keys:
        base = d[k]
        flat = base.reshape(-1)
        for i in g.choice(flat.numel(), size=min(6, flat.numel()), replace=False):
            orig = float(flat[i])
            flat[i] = orig + eps
            fp = _objective(d, dy, dh)
            flat[i] = orig - eps
            fm = _objective(d, dy, dh)
            flat[i] = orig
            fd = (fp - fm) / (2 * eps)
            got = grads[k].reshape(-1)[i]
            assert abs(got - fd) <= 1e-6 * (1.0 + abs(fd)), (k, int(i), got, fd)
