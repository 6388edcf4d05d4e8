"""Host-side checks of the C ABI (no GPU): the library builds and loads, exports every function the
public header declares, the Python ctypes mirror of ssm_scan_params matches the C layout, and
invalid calls are rejected on the host with the documented status before anything is launched."""
import ctypes
import os
import re
import subprocess
import tempfile

import pytest

import selective_state_space_156_b300 as ssm
from selective_state_space_156_b300 import build as ssm_build

pytestmark = pytest.mark.cpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "ssm_scan.h")


@pytest.fixture(scope="module")
def L():
    ssm_build.build()
    return ssm.lib()


def declared_functions():
    text = open(HEADER).read()
    return re.findall(r"SSM_API\s+[\w\s\*]+?\b(\w+)\s*\(", text)


def test_header_declares_the_boundary():
    names = set(declared_functions())
    assert {"ssm_scan_fwd", "causal_conv1d_fwd", "ssm_state_update", "ssm_last_error",
            "ssm_scan_workspace_size", "ssm_version"} <= names


def test_library_exports_every_declared_symbol(L):
    out = subprocess.run(["nm", "-D", "--defined-only", ssm.LIB_PATH], capture_output=True, text=True, check=True).stdout
    exported = {l.split()[-1] for l in out.splitlines() if l.strip()}
    for name in declared_functions():
        assert name in exported, name
        assert hasattr(L, name)
    # nothing but the C ABI is exported (hidden visibility for everything else)
    ours = {n for n in exported if n.startswith(("ssm_", "causal_"))}
    assert ours == set(declared_functions())


def test_version_string(L):
    assert b"sm_103a" in L.ssm_version()


def test_params_struct_layout_matches_c():
    src = r"""
#include <stdio.h>
#include <stddef.h>
#include "ssm_scan.h"
#define F(f) printf(#f " %zu\n", offsetof(ssm_scan_params, f));
int main(void) {
  printf("sizeof %zu\n", sizeof(ssm_scan_params));
  F(batch) F(dim) F(dstate) F(seqlen) F(in_dtype) F(out_dtype) F(u) F(delta) F(A) F(Bm) F(Cm) F(Dskip)
  F(delta_bias) F(z) F(conv_w) F(conv_b) F(conv_width) F(h0) F(h_out) F(y) F(delta_softplus) F(zoh)
  F(workspace) F(workspace_bytes)
  return 0;
}
"""
    with tempfile.TemporaryDirectory() as td:
        c = os.path.join(td, "layout.c")
        exe = os.path.join(td, "layout")
        open(c, "w").write(src)
        subprocess.run(["gcc", "-I", os.path.join(ROOT, "include"), "-o", exe, c], check=True)
        out = subprocess.run([exe], capture_output=True, text=True, check=True).stdout
    got = dict(l.split() for l in out.splitlines())
    assert int(got.pop("sizeof")) == ctypes.sizeof(ssm.ScanParams)
    for name, off in got.items():
        assert getattr(ssm.ScanParams, name).offset == int(off), name


def _params(**kw):
    p = ssm.ScanParams()
    p.batch, p.dim, p.dstate, p.seqlen = 2, 64, 16, 128
    p.in_dtype = p.out_dtype = ssm.SSM_BF16
    fake = 1 << 40  # never dereferenced: every case below fails validation before any launch
    p.u, p.delta, p.A, p.Bm, p.Cm = fake, fake + (1 << 30), fake + (2 << 30), fake + (3 << 30), fake + (4 << 30)
    p.y = fake + (5 << 30)
    p.delta_softplus, p.zoh = 1, 1
    for k, v in kw.items():
        setattr(p, k, v)
    return p


@pytest.mark.parametrize("field,value,status", [
    ("batch", 0, ssm.SSM_ERR_INVALID_ARG),
    ("seqlen", -3, ssm.SSM_ERR_INVALID_ARG),
    ("dstate", 17, ssm.SSM_ERR_UNSUPPORTED),
    ("dstate", 128, ssm.SSM_ERR_UNSUPPORTED),
    ("in_dtype", 7, ssm.SSM_ERR_INVALID_ARG),
    ("u", None, ssm.SSM_ERR_INVALID_ARG),
    ("Cm", None, ssm.SSM_ERR_INVALID_ARG),
    ("y", None, ssm.SSM_ERR_INVALID_ARG),
    ("zoh", 2, ssm.SSM_ERR_INVALID_ARG),
    ("batch", 70000, ssm.SSM_ERR_UNSUPPORTED),
])
def test_scan_rejects_bad_arguments_on_host(L, field, value, status):
    p = _params(**{field: value})
    assert L.ssm_scan_fwd(ctypes.byref(p), None) == status
    assert L.ssm_last_error().decode().startswith("ssm_scan_fwd")
    assert L.ssm_scan_workspace_size(ctypes.byref(p)) == 0


def test_scan_rejects_null_params(L):
    assert L.ssm_scan_fwd(None, None) == ssm.SSM_ERR_INVALID_ARG


def test_scan_rejects_overlapping_output(L):
    p = _params()
    p.y = p.u + 64  # y starts inside u
    assert L.ssm_scan_fwd(ctypes.byref(p), None) == ssm.SSM_ERR_INVALID_ARG
    assert "overlaps" in L.ssm_last_error().decode()


def test_scan_rejects_bad_conv_width(L):
    p = _params(conv_w=1 << 44, conv_width=5)
    assert L.ssm_scan_fwd(ctypes.byref(p), None) == ssm.SSM_ERR_INVALID_ARG


def test_conv_and_decode_reject_bad_arguments_on_host(L):
    f = 1 << 40
    assert L.causal_conv1d_fwd(f, f + (1 << 30), None, f + (2 << 30), 1, 8, 16, 5, 1, 1, None) == ssm.SSM_ERR_INVALID_ARG
    assert L.causal_conv1d_fwd(None, f, None, f + (2 << 30), 1, 8, 16, 4, 1, 1, None) == ssm.SSM_ERR_INVALID_ARG
    assert L.causal_conv1d_fwd(f, f + (1 << 30), None, f + 8, 1, 8, 16, 4, 1, 1, None) == ssm.SSM_ERR_INVALID_ARG
    args = [f + (k << 30) for k in range(10)]
    assert L.ssm_state_update(*args, 4, 8, 48, 1, 1, 1, None) == ssm.SSM_ERR_UNSUPPORTED
    assert L.ssm_state_update(*args, 0, 8, 16, 1, 1, 1, None) == ssm.SSM_ERR_INVALID_ARG
    args[9] = args[1]  # y aliases u
    assert L.ssm_state_update(*args, 4, 8, 16, 1, 1, 1, None) == ssm.SSM_ERR_INVALID_ARG


def test_calls_without_library_fail_loudly(monkeypatch):
    monkeypatch.setattr(ssm, "_lib", None)
    monkeypatch.setattr(ssm, "LIB_PATH", "/nonexistent/libssm_b300.so")
    with pytest.raises(ImportError):
        ssm.lib()
