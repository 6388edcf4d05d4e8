"""GPU parity of ssm_scan_fwd (through the C ABI) against the fp64 CPU oracle.

Small cases compare every element; the full-size workloads, launched exactly as bench.py launches
them, compare sampled (batch, channel) rows that the oracle computes one by one and check that every
output is finite.  Edge cases: L = 1, L not a multiple of 8, ragged channel blocks, every supported
dstate, h0 given / aliased with h_out, no gate / no D / no bias / softplus off, both discretisations,
zero entries of A, conv widths 1-4, unaligned rows, mixed input/output dtypes, the L split through
the workspace, and chained calls with carried state."""
import numpy as np
import pytest
import torch

import oracle
import selective_state_space_156_b300 as ssm
import workloads
from gpu_helpers import Guarded, assert_close, h_tolerance, sample_rows, to_dev, y_tolerance

pytestmark = pytest.mark.gpu

TINY = workloads.SCAN_CONFIGS["tiny"]


def run_gpu(d: dict, out_dtype=None, workspace="auto", guard=True, alias_state=False):
    g = to_dev(d)
    u = g["u"]
    Bsz, D, L = u.shape
    N = g["A"].shape[1]
    out_dtype = out_dtype or u.dtype
    yg = Guarded((Bsz, D, L), out_dtype) if guard else None
    y = yg.t if guard else torch.empty((Bsz, D, L), dtype=out_dtype, device="cuda")
    if alias_state:
        h = g["h0"]
        h_out = h
    else:
        h_out = Guarded((Bsz, D, N), torch.float32) if guard else None
        h = h_out.t if guard else torch.empty((Bsz, D, N), dtype=torch.float32, device="cuda")
    ssm.ssm_scan_fwd(u, g["delta"], g["A"], g["Bm"], g["Cm"], Dskip=g.get("Dskip"), delta_bias=g.get("delta_bias"),
                     z=g.get("z"), conv_w=g.get("conv_w"), conv_b=g.get("conv_b"), h0=g.get("h0"), h_out=h, y=y,
                     delta_softplus=d.get("delta_softplus", True), zoh=d.get("zoh", True), workspace=workspace)
    torch.cuda.synchronize()
    if guard:
        yg.check_bands()
        if not alias_state:
            h_out.check_bands()
    return y, h


def check_full(d, out_dtype=None, **kw):
    y, h = run_gpu(d, out_dtype=out_dtype, **kw)
    y_ref, h_ref, _ = oracle.scan(d)
    Bsz, D, L = d["u"].shape
    od = out_dtype or d["u"].dtype
    assert_close(y, y_ref.reshape(Bsz, D, L), y_tolerance(y_ref.reshape(Bsz, D, L), od), "y")
    assert_close(h, h_ref.reshape(Bsz, D, -1), h_tolerance(h_ref.reshape(Bsz, D, -1), d["u"].dtype), "h_out")
    return y, h


def test_tiny_config_every_element():
    check_full(workloads.make_scan_inputs(TINY))


@pytest.mark.parametrize("L", [1, 2, 7, 8, 61, 64, 65, 200])
def test_lengths(L):
    check_full(workloads.make_scan_inputs(TINY, batch=2, dim=40, seqlen=L, with_h0=True))


@pytest.mark.parametrize("N", [1, 2, 3, 4, 5, 8, 11, 16])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_dstate(N, dtype):
    check_full(workloads.make_scan_inputs(TINY, batch=2, dim=130, seqlen=77, dstate=N, dtype=dtype))


@pytest.mark.parametrize("zoh", [True, False])
@pytest.mark.parametrize("has_z,has_D,has_bias,softplus", [
    (True, True, True, True), (False, True, True, True), (True, False, True, True),
    (True, True, False, True), (False, False, False, True), (True, True, True, False)])
def test_flags(zoh, has_z, has_D, has_bias, softplus):
    d = workloads.make_scan_inputs(TINY, batch=3, dim=33, seqlen=96, with_h0=True)
    d["zoh"] = zoh
    d["delta_softplus"] = softplus
    if not has_z:
        d["z"] = None
    if not has_D:
        d["Dskip"] = None
    if not has_bias:
        d["delta_bias"] = None
    if not softplus:
        # keep dt positive and in the usual range when it is taken raw
        d["delta"] = d["delta"].abs() * 0.05 + 1e-3
        d["delta_bias"] = None
    check_full(d)


@pytest.mark.parametrize("width", [1, 2, 3, 4])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_fused_conv(width, dtype):
    cfg = workloads.SCAN_CONFIGS["mamba1.4b_conv"]
    d = workloads.make_scan_inputs(cfg, batch=2, dim=140, seqlen=133, dtype=dtype)
    g = torch.Generator().manual_seed(width)
    d["conv_w"] = (torch.randn((140, width), generator=g) * 0.5).contiguous()
    d["conv_b"] = torch.randn(140, generator=g) * 0.1
    check_full(d)


def test_fused_conv_without_bias():
    d = workloads.make_scan_inputs(workloads.SCAN_CONFIGS["mamba1.4b_conv"], batch=1, dim=64, seqlen=100, dtype="f32")
    d["conv_b"] = None
    check_full(d)


def test_zero_and_positive_A():
    d = workloads.make_scan_inputs(TINY, batch=2, dim=70, seqlen=50, with_h0=True)
    A = d["A"].clone()
    A[3, :] = 0.0           # every state of channel 3
    A[40, 1] = 0.0          # one state of channel 40 (its warp takes the a == 0 loop body)
    A[65, 2] = 0.05         # a slowly growing mode
    d["A"] = A
    check_full(d)
    d["zoh"] = False
    check_full(d)


@pytest.mark.parametrize("in_dtype,out_dtype", [("bf16", torch.float32), ("f32", torch.bfloat16)])
def test_mixed_dtypes(in_dtype, out_dtype):
    d = workloads.make_scan_inputs(TINY, batch=2, dim=64, seqlen=128, dtype=in_dtype)
    check_full(d, out_dtype=out_dtype)


def test_unaligned_rows_take_the_element_path():
    d = workloads.make_scan_inputs(TINY, batch=2, dim=48, seqlen=72, dtype="bf16")
    g = to_dev(d)
    # shift every (B, D, L) tensor by one element inside a larger allocation: rows lose 16-byte alignment
    for k in ("u", "delta", "z"):
        big = torch.empty(g[k].numel() + 1, dtype=g[k].dtype, device="cuda")
        big[1:].copy_(g[k].reshape(-1))
        g[k] = big[1:].view(g[k].shape)
    y = torch.empty(g["u"].numel() + 1, dtype=torch.bfloat16, device="cuda")[1:].view(g["u"].shape)
    ssm.ssm_scan_fwd(g["u"], g["delta"], g["A"], g["Bm"], g["Cm"], Dskip=g["Dskip"], delta_bias=g["delta_bias"],
                     z=g["z"], y=y)
    y_ref, _, _ = oracle.scan(d)
    assert_close(y, y_ref.reshape(y.shape), y_tolerance(y_ref.reshape(y.shape), torch.bfloat16), "y")


@pytest.mark.parametrize("split", [False, True])
def test_h0_aliases_h_out(split):
    # one channel block and a long L: with a workspace the scan splits L into segments
    d = workloads.make_scan_inputs(TINY, batch=1, dim=96, seqlen=4096, dstate=16, with_h0=True)
    y_ref, h_ref, _ = oracle.scan(d)
    y, h = run_gpu(d, workspace="auto" if split else None, alias_state=True)
    assert_close(y, y_ref.reshape(y.shape), y_tolerance(y_ref.reshape(y.shape), torch.float32), "y")
    assert_close(h, h_ref.reshape(h.shape), h_tolerance(h_ref.reshape(h.shape), torch.float32), "h_out")


def test_split_path_is_taken_and_matches():
    d = workloads.make_scan_inputs(TINY, batch=1, dim=200, seqlen=5000, dstate=16, dtype="bf16", with_h0=True)
    g = to_dev(d)
    nbytes = ssm.ssm_scan_workspace_size(g["u"], g["delta"], g["A"], g["Bm"], g["Cm"], h0=g["h0"])
    assert nbytes > 0, "a 2-block problem should ask for the L split"
    y_split, h_split = check_full(d, workspace="auto")
    y_one, h_one = check_full(d, workspace=None)
    # the two launch shapes differ only by fp32 rounding order of the carried state
    torch.testing.assert_close(h_split, h_one, rtol=1e-4, atol=1e-4)


@pytest.mark.parametrize("dim,L", [(64, 512), (64, 1000), (200, 2048), (300, 4104), (40, 8192)])
def test_split_segment_plans(dim, L):
    """The packed kernel's L split at several grid sizes and lengths, so that the planner takes different
    segment counts and first-segment lengths (segment 0's final pass runs beside the later segments'
    summaries): every element against the oracle, with h0 and the gate."""
    d = workloads.make_scan_inputs(workloads.SCAN_CONFIGS["mamba130m"], batch=1, dim=dim, seqlen=L, with_h0=True,
                                   seed=4200 + dim + L)
    g = to_dev(d)
    assert ssm.ssm_scan_workspace_size(g["u"], g["delta"], g["A"], g["Bm"], g["Cm"], h0=g["h0"], z=g["z"]) > 0
    check_full(d, workspace="auto")


def test_packed_split_with_h0_aliasing_h_out():
    """bf16 on the packed kernel with the L split and h0 == h_out: segment 0 reads h0 in the first launch,
    the last segment writes h_out in the second."""
    d = workloads.make_scan_inputs(workloads.SCAN_CONFIGS["mamba130m"], batch=1, dim=96, seqlen=4096, with_h0=True)
    y_ref, h_ref, _ = oracle.scan(d)
    y, h = run_gpu(d, workspace="auto", alias_state=True)
    assert_close(y, y_ref.reshape(y.shape), y_tolerance(y_ref.reshape(y.shape), torch.bfloat16), "y")
    assert_close(h, h_ref.reshape(h.shape), h_tolerance(h_ref.reshape(h.shape), torch.bfloat16), "h_out")


def test_chained_calls_equal_one_call():
    d = workloads.make_scan_inputs(workloads.SCAN_CONFIGS["long2.8b"], batch=1, dim=64, seqlen=4096, with_h0=True)
    g = to_dev(d)
    y_one, h_one = ssm.ssm_scan_fwd(g["u"], g["delta"], g["A"], g["Bm"], g["Cm"], Dskip=g["Dskip"],
                                    delta_bias=g["delta_bias"], z=g["z"], h0=g["h0"], return_state=True,
                                    workspace="auto")
    h = g["h0"].clone()
    ys = []
    for c in range(0, 4096, 1024):
        sl = slice(c, c + 1024)
        yc = ssm.ssm_scan_fwd(g["u"][..., sl].contiguous(), g["delta"][..., sl].contiguous(), g["A"],
                              g["Bm"][..., sl].contiguous(), g["Cm"][..., sl].contiguous(), Dskip=g["Dskip"],
                              delta_bias=g["delta_bias"], z=g["z"][..., sl].contiguous(), h0=h, h_out=h)
        ys.append(yc)
    y_chain = torch.cat(ys, dim=-1)
    y_ref, h_ref, _ = oracle.scan(d)
    for y in (y_one, y_chain):
        assert_close(y, y_ref.reshape(y.shape), y_tolerance(y_ref.reshape(y.shape), torch.bfloat16), "y")
    for hh in (h_one, h):
        assert_close(hh, h_ref.reshape(hh.shape), h_tolerance(h_ref.reshape(hh.shape), torch.bfloat16), "h")


# ------------------------------------------------------------------------------------------------
# Full-size workloads, launched as bench.py launches them, compared on sampled rows
# ------------------------------------------------------------------------------------------------
def _full_size(cfg, nrows, seed, chunk_check=False):
    d = workloads.make_scan_inputs(cfg)
    g = to_dev(d)
    y, h = ssm.ssm_scan_fwd(g["u"], g["delta"], g["A"], g["Bm"], g["Cm"], Dskip=g.get("Dskip"),
                            delta_bias=g.get("delta_bias"), z=g.get("z"), conv_w=g.get("conv_w"),
                            conv_b=g.get("conv_b"), return_state=True, workspace="auto")
    torch.cuda.synchronize()
    assert bool(torch.isfinite(y).all()), "non-finite outputs"
    Bsz, D, L = d["u"].shape
    rows = sample_rows(Bsz, D, nrows, seed)
    y_ref, h_ref, _ = oracle.scan(d, rows=rows)
    bi = torch.tensor([r[0] for r in rows])
    di = torch.tensor([r[1] for r in rows])
    ys = y[bi.cuda(), di.cuda()]
    hs = h[bi.cuda(), di.cuda()]
    assert_close(ys, y_ref, y_tolerance(y_ref, y.dtype), "y (sampled rows)")
    assert_close(hs, h_ref, h_tolerance(h_ref, d["u"].dtype), "h_out (sampled rows)")
    return d, g, rows, y_ref, h_ref


def test_full_mamba130m_sampled():
    _full_size(workloads.SCAN_CONFIGS["mamba130m"], 96, 1)


def test_full_mamba14b_conv_sampled():
    _full_size(workloads.SCAN_CONFIGS["mamba1.4b_conv"], 96, 2)


def test_full_long_context_sampled_and_chunk_split():
    cfg = workloads.SCAN_CONFIGS["long2.8b"]
    d, g, rows, y_ref, h_ref = _full_size(cfg, 66, 3)
    # the same sequence as 32 calls of 2048 steps with the state carried between calls
    Bsz, D, L = d["u"].shape
    h = torch.zeros((Bsz, D, cfg.dstate), dtype=torch.float32, device="cuda")
    di = torch.tensor([r[1] for r in rows], device="cuda")
    ys = []
    for c in range(0, L, cfg.chunk):
        sl = slice(c, c + cfg.chunk)
        yc = ssm.ssm_scan_fwd(g["u"][..., sl].contiguous(), g["delta"][..., sl].contiguous(), g["A"],
                              g["Bm"][..., sl].contiguous(), g["Cm"][..., sl].contiguous(), Dskip=g["Dskip"],
                              delta_bias=g["delta_bias"], z=g["z"][..., sl].contiguous(), h0=h, h_out=h,
                              workspace="auto")
        ys.append(yc[0, di])
    y_chain = torch.cat(ys, dim=-1)
    assert_close(y_chain, y_ref, y_tolerance(y_ref, torch.bfloat16), "y (32 chained calls)")
    assert_close(h[0, di], h_ref, h_tolerance(h_ref, torch.bfloat16), "h (32 chained calls)")


# ------------------------------------------------------------------------------------------------
# The four-lanes-per-channel kernel (bf16 in and out, rows 16-byte aligned, L % 8 == 0)
# ------------------------------------------------------------------------------------------------
@pytest.mark.parametrize("N", [1, 4, 7, 16, 32, 64])
@pytest.mark.parametrize("L", [8, 40, 96])
def test_g4_dstate_and_lengths(N, L):
    d = workloads.make_scan_inputs(workloads.SCAN_CONFIGS["mamba130m"], batch=2, dim=70, seqlen=L, dstate=N,
                                   with_h0=True)
    check_full(d)


@pytest.mark.parametrize("width", [1, 2, 3, 4])
@pytest.mark.parametrize("zoh", [True, False])
def test_g4_fused_conv(width, zoh):
    d = workloads.make_scan_inputs(workloads.SCAN_CONFIGS["mamba1.4b_conv"], batch=2, dim=96, seqlen=200)
    g = torch.Generator().manual_seed(17 + width)
    d["conv_w"] = (torch.randn((96, width), generator=g) * 0.5).contiguous()
    d["conv_b"] = torch.randn(96, generator=g) * 0.1
    d["zoh"] = zoh
    check_full(d)


@pytest.mark.parametrize("has_z,has_D,softplus", [(False, True, True), (True, False, True), (True, True, False)])
def test_g4_flags(has_z, has_D, softplus):
    d = workloads.make_scan_inputs(workloads.SCAN_CONFIGS["mamba130m"], batch=3, dim=40, seqlen=128, with_h0=True)
    if not has_z:
        d["z"] = None
    if not has_D:
        d["Dskip"] = None
    if not softplus:
        d["delta_softplus"] = False
        d["delta"] = (d["delta"].float().abs() * 0.05 + 1e-3).to(torch.bfloat16)
        d["delta_bias"] = None
    check_full(d)


def test_g4_zero_A():
    d = workloads.make_scan_inputs(workloads.SCAN_CONFIGS["mamba130m"], batch=2, dim=64, seqlen=64, with_h0=True)
    A = d["A"].clone()
    A[5, :] = 0.0
    A[33, 7] = 0.0
    d["A"] = A
    check_full(d)


@pytest.mark.parametrize("N", [16, 64])
def test_g4_split_with_aliased_state(N):
    d = workloads.make_scan_inputs(workloads.SCAN_CONFIGS["long2.8b"], batch=1, dim=64, seqlen=6144, dstate=N,
                                   with_h0=True)
    g = to_dev(d)
    assert ssm.ssm_scan_workspace_size(g["u"], g["delta"], g["A"], g["Bm"], g["Cm"], h0=g["h0"], z=g["z"]) > 0
    y_ref, h_ref, _ = oracle.scan(d)
    y, h = run_gpu(d, workspace="auto", alias_state=True)
    assert_close(y, y_ref.reshape(y.shape), y_tolerance(y_ref.reshape(y.shape), torch.bfloat16), "y")
    assert_close(h, h_ref.reshape(h.shape), h_tolerance(h_ref.reshape(h.shape), torch.bfloat16), "h_out")


def test_chained_calls_captured_in_a_cuda_graph():
    """A prefill in 8 chunked calls (carried state, L split through a preallocated workspace) captured once
    as a CUDA graph and replayed: bit-identical to the same calls made directly, and within the bound of
    the oracle."""
    d = workloads.make_scan_inputs(workloads.SCAN_CONFIGS["long2.8b"], batch=1, dim=256, seqlen=4096, with_h0=True)
    g = to_dev(d)
    pieces = [{k: g[k][..., a:a + 512].contiguous() for k in ("u", "delta", "z", "Bm", "Cm")}
              for a in range(0, 4096, 512)]
    kw = dict(Dskip=g["Dskip"], delta_bias=g["delta_bias"])
    p0 = pieces[0]
    ws = torch.empty(max(ssm.ssm_scan_workspace_size(p0["u"], p0["delta"], g["A"], p0["Bm"], p0["Cm"], h0=g["h0"],
                                                     z=p0["z"], **kw), 1), dtype=torch.uint8, device="cuda")
    h = torch.empty_like(g["h0"])
    ys = [torch.empty_like(pc["u"]) for pc in pieces]

    def chain():
        h.copy_(g["h0"])
        for pc, yc in zip(pieces, ys):
            ssm.ssm_scan_fwd(pc["u"], pc["delta"], g["A"], pc["Bm"], pc["Cm"], z=pc["z"], h0=h, h_out=h, y=yc,
                             workspace=ws, **kw)

    chain()
    torch.cuda.synchronize()
    y_direct = torch.cat([y.clone() for y in ys], dim=-1)
    h_direct = h.clone()
    for y in ys:
        y.zero_()
    h.zero_()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        chain()
    torch.cuda.current_stream().wait_stream(s)
    graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(torch.cat(ys, dim=-1), y_direct)
    assert torch.equal(h, h_direct)
    y_ref, h_ref, _ = oracle.scan(d)
    assert_close(y_direct, y_ref.reshape(y_direct.shape), y_tolerance(y_ref.reshape(y_direct.shape), torch.bfloat16), "y")
    assert_close(h_direct, h_ref.reshape(h.shape), h_tolerance(h_ref.reshape(h.shape), torch.bfloat16), "h")
