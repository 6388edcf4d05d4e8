"""Pins of the SSD (Mamba-2) oracle against forms that do not run its recurrence.

P15  The matrix ("dual") form of dpshk.com/news/3333417 section 6.1: y = M x with
     M[k,i] = sum_n C_k[n] B_i[n] w_i prod_{j=i+1..k} a_j  (i <= k), plus the initial state's
     contribution C_k prod_{j<=k} a_j h0 and the D skip, then the gate; and the final state
     h_L = prod_j a_j h0 + sum_i prod_{j>i} a_j w_i B_i x_i.  Brute force, O(L^2 N) per channel,
     with the group of head h written out as h // (H / G).
P16  With A = 0 (no decay) the same layer is causal linear attention with the structured mask of
     section 6.1: Y = (tril(C B^T) diag(w)) X per head, computed here with matrix products; ZOH's
     A -> 0 limit gives w = dt.

Sizes are tiny (L <= 16) so that the brute force is exact to rounding; tolerance 1e-12 relative."""
import math

import numpy as np
import pytest
import torch

import workloads
from oracle import f64
from oracle.ssd import ssd_scan


def _softplus(v):
    return np.where(v > 0, v + np.log1p(np.exp(-np.abs(v))), np.log1p(np.exp(v)))


def _tiny(seed, *, H=4, G=2, P=3, N=5, L=12, z=True, h0=True):
    cfg = workloads.SsdConfig("pin", 2, H, P, G, N, L, has_z=z, seed=seed)
    return workloads.make_ssd_inputs(cfg, with_h0=h0)


def _brute(d):
    x, dtr = f64(d["x"]), f64(d["dt"])
    Bm, Cm = f64(d["Bm"]), f64(d["Cm"])
    A, bias = f64(d["A"]), f64(d["dt_bias"])
    Dsk = f64(d["Dskip"])
    z = f64(d.get("z"))
    h0 = f64(d.get("h0"))
    Bsz, Dm, L = x.shape
    H, G = d["nheads"], d["ngroups"]
    P, N = Dm // H, Bm.shape[-1]
    y = np.zeros((Bsz, Dm, L))
    hL = np.zeros((Bsz, H, P, N))
    for b in range(Bsz):
        for h in range(H):
            g = h // (H // G)
            s = dtr[b, h] + bias[h]
            dt = _softplus(s) if d["delta_softplus"] else s
            la = dt * A[h]                                   # log of a_t
            w = np.expm1(la) / A[h] if (d["zoh"] and A[h] != 0) else dt
            cum = np.concatenate([[0.0], np.cumsum(la)])    # cum[k+1] = sum_{j<=k} log a_j
            for p in range(P):
                c = h * P + p
                for k in range(L):
                    acc = 0.0
                    for i in range(k + 1):
                        m = float(Cm[b, g, k] @ Bm[b, g, i]) * w[i] * math.exp(cum[k + 1] - cum[i + 1])
                        acc += m * x[b, c, i]
                    if h0 is not None:
                        acc += math.exp(cum[k + 1]) * float(Cm[b, g, k] @ h0[b, h, p])
                    if Dsk is not None:
                        acc += Dsk[h] * x[b, c, k]
                    if z is not None:
                        acc *= z[b, c, k] / (1.0 + math.exp(-z[b, c, k]))
                    y[b, c, k] = acc
                st = np.zeros(N) if h0 is None else math.exp(cum[L]) * h0[b, h, p]
                for i in range(L):
                    st = st + math.exp(cum[L] - cum[i + 1]) * w[i] * Bm[b, g, i] * x[b, c, i]
                hL[b, h, p] = st
    return y, hL


def _check(d):
    Bsz, Dm, L = d["x"].shape
    H = d["nheads"]
    P, N = Dm // H, d["Bm"].shape[-1]
    y, h, _ = ssd_scan(d)
    yb, hb = _brute(d)
    np.testing.assert_allclose(y, yb.reshape(Bsz * Dm, L), rtol=1e-12, atol=1e-12 * (1 + np.abs(yb).max()))
    np.testing.assert_allclose(h, hb.reshape(Bsz * Dm, N), rtol=1e-12, atol=1e-12 * (1 + np.abs(hb).max()))
    return y, h


@pytest.mark.parametrize("zoh", [False, True])
@pytest.mark.parametrize("softplus", [True, False])
@pytest.mark.parametrize("h0,z", [(True, True), (False, False)])
def test_p15_ssd_oracle_matches_the_matrix_form(zoh, softplus, h0, z):
    d = _tiny(31 + 2 * zoh + softplus, z=z, h0=h0)
    d["zoh"] = zoh
    d["delta_softplus"] = softplus
    if not softplus:  # dt = raw + bias directly: keep it a positive step
        d["dt"] = (0.05 + 0.1 * d["dt"].float().abs()).to(torch.bfloat16)
    _check(d)


def test_p15_groups_follow_consecutive_heads():
    """H = 6 heads in G = 3 groups: heads 0-1 read group 0, 2-3 group 1, 4-5 group 2 (a mapping by
    h % G would pair heads 0 and 3 instead and fail the brute force)."""
    _check(_tiny(41, H=6, G=3, P=2, N=4, L=9))


def test_p15_sampled_rows_equal_the_full_run():
    d = _tiny(43)
    y, h, _ = ssd_scan(d)
    P = d["x"].shape[1] // d["nheads"]
    rows = [(1, 3, 2), (0, 0, 0), (1, 1, 1)]
    ys, hs, _ = ssd_scan(d, rows=rows)
    for r, (b, hh, p) in enumerate(rows):
        idx = b * d["x"].shape[1] + hh * P + p
        np.testing.assert_array_equal(ys[r], y[idx])
        np.testing.assert_array_equal(hs[r], h[idx])


@pytest.mark.parametrize("zoh", [False, True])
def test_p16_no_decay_is_masked_linear_attention(zoh):
    d = _tiny(47, z=False, h0=False, L=16, N=6)
    d["A"] = torch.zeros_like(d["A"])
    d["zoh"] = zoh
    y, _, _ = ssd_scan(d)
    x, Bm, Cm = f64(d["x"]), f64(d["Bm"]), f64(d["Cm"])
    Bsz, Dm, L = x.shape
    H, G = d["nheads"], d["ngroups"]
    P = Dm // H
    dt = _softplus(f64(d["dt"]) + f64(d["dt_bias"])[None, :, None])
    ref = np.zeros((Bsz, Dm, L))
    for b in range(Bsz):
        for h in range(H):
            g = h // (H // G)
            Mk = np.tril(Cm[b, g] @ Bm[b, g].T) * dt[b, h][None, :]          # (L, L) structured mask
            X = x[b, h * P:(h + 1) * P].T                                     # (L, P)
            ref[b, h * P:(h + 1) * P] = (Mk @ X).T + f64(d["Dskip"])[h] * x[b, h * P:(h + 1) * P]
    np.testing.assert_allclose(y, ref.reshape(Bsz * Dm, L), rtol=1e-12, atol=1e-12 * np.abs(ref).max())
