"""Shared helpers for the GPU parity tests: moving workload dicts to the device, guarded output
buffers (canary bands around the output and a NaN pre-fill, standing in for a memory checker), and
the parity tolerances.

Tolerances (per element, against the oracle's unrounded fp64 result y_ref):
  fp32 output : |y - y_ref| <= 1e-4 * (1 + |y_ref|)
  bf16 output : |y - y_ref| <= 2e-2 * (|y_ref| + rms(y_ref))
  final state : |h - h_ref| <= 1e-4 * (1 + |h_ref|) with fp32 inputs, 1e-3 * (1 + |h_ref|) with bf16 inputs
"""
import numpy as np
import torch

CANARY = 0x7FC0DEAD  # a NaN bit pattern with a payload that no kernel writes


def to_dev(d: dict, device="cuda") -> dict:
    return {k: (v.to(device).contiguous() if isinstance(v, torch.Tensor) else v) for k, v in d.items()}


class Guarded:
    """An output tensor placed between two canary bands inside a larger buffer, pre-filled with NaN."""

    def __init__(self, shape, dtype, device="cuda", band=256):
        n = int(np.prod(shape))
        esz = torch.tensor([], dtype=dtype).element_size()
        words = (band * 2 * 4 + n * esz + 3) // 4 + 1
        self.raw = torch.full((words,), CANARY, dtype=torch.int32, device=device)
        self.band_bytes = band * 4
        self.nbytes = n * esz
        byte_view = self.raw.view(torch.uint8)
        self.t = byte_view[self.band_bytes:self.band_bytes + self.nbytes].view(dtype).view(shape)
        self.t.fill_(float("nan"))

    def check_bands(self):
        bv = self.raw.view(torch.uint8)
        lo = bv[:self.band_bytes].view(torch.int32)
        hi_start = self.band_bytes + self.nbytes
        hi_start += (-hi_start) % 4
        hi = bv[hi_start:].view(torch.int32)
        assert bool((lo == CANARY).all()), "write before the output buffer"
        assert bool((hi == CANARY).all()), "write past the end of the output buffer"


def y_tolerance(ref: np.ndarray, out_dtype) -> np.ndarray:
    if out_dtype == torch.float32:
        return 1e-4 * (1.0 + np.abs(ref))
    rms = float(np.sqrt(np.mean(ref * ref))) if ref.size else 0.0
    return 2e-2 * (np.abs(ref) + rms)


def h_tolerance(ref: np.ndarray, in_dtype) -> np.ndarray:
    return (1e-4 if in_dtype == torch.float32 else 1e-3) * (1.0 + np.abs(ref))


def assert_close(got, ref: np.ndarray, tol: np.ndarray, what: str):
    g = got.detach().to("cpu").to(torch.float64).numpy() if isinstance(got, torch.Tensor) else np.asarray(got)
    g = g.reshape(ref.shape)
    assert np.isfinite(g).all(), f"{what}: non-finite values ({np.count_nonzero(~np.isfinite(g))})"
    err = np.abs(g - ref)
    ratio = err / tol
    i = np.unravel_index(int(np.argmax(ratio)), ratio.shape)
    assert ratio[i] <= 1.0, (f"{what}: worst element {i}: got {g[i]!r} want {ref[i]!r} |err| {err[i]:.3e} "
                             f"tol {tol[i]:.3e} (max |err| {err.max():.3e})")
    return float(ratio.max())


def sample_rows(Bsz: int, D: int, k: int, seed: int = 0):
    g = np.random.default_rng(seed)
    rows = {(0, 0), (Bsz - 1, D - 1), (0, D - 1), (Bsz - 1, 0)}
    while len(rows) < min(k, Bsz * D):
        rows.add((int(g.integers(Bsz)), int(g.integers(D))))
    return sorted(rows)
