"""Helpers for GPU-vs-oracle parity tests.

Tolerances: bf16 inputs with fp32 accumulation must match the float64 oracle
to max |dO| <= 2e-2 and max |dLSE| <= 1e-3; fp32 inputs to 1e-5 for both.
"""
import numpy as np
import torch

TOL = {torch.bfloat16: (2e-2, 1e-3), torch.float32: (1e-5, 1e-5)}


def to_np64(t):
    return t.detach().to("cpu", torch.float32).numpy().astype(np.float64)


def compare(o_gpu, lse_gpu, o_ref, lse_ref, dtype, what=""):
    """Element-by-element comparison; -inf LSE must match exactly."""
    tol_o, tol_l = TOL[dtype]
    o = to_np64(o_gpu)
    lse = to_np64(lse_gpu)
    assert o.shape == o_ref.shape, (what, o.shape, o_ref.shape)
    assert np.all(np.isfinite(o)), "%s: non-finite output" % what
    d_o = np.abs(o - o_ref).max() if o.size else 0.0
    fin = np.isfinite(lse_ref)
    assert np.array_equal(np.isfinite(lse), fin), "%s: -inf pattern of LSE differs" % what
    assert np.all(lse[~fin] == lse_ref[~fin])
    d_l = np.abs(lse[fin] - lse_ref[fin]).max() if fin.any() else 0.0
    assert d_o <= tol_o, "%s: max|dO| = %.3g > %.1g" % (what, d_o, tol_o)
    assert d_l <= tol_l, "%s: max|dLSE| = %.3g > %.1g" % (what, d_l, tol_l)
    return d_o, d_l


def guarded(shape, dtype, device, guard=4096, fill=7.0):
    """A tensor view with `guard` sentinel elements on both sides, to catch
    out-of-bounds writes.  Returns (view, backing, guard)."""
    n = int(np.prod(shape))
    backing = torch.full((n + 2 * guard,), fill, dtype=dtype, device=device)
    view = backing[guard:guard + n].view(*shape)
    return view, backing, guard


def guards_intact(backing, guard, fill=7.0):
    lo = backing[:guard]
    hi = backing[-guard:]
    return bool(torch.all(lo == fill)) and bool(torch.all(hi == fill))
