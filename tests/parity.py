"""Helpers for GPU-vs-oracle parity tests.

Tolerances: bf16 inputs with fp32 accumulation must match the float64 oracle
to max |dO| <= 2e-2 and max |dLSE| <= 1e-3; fp32 inputs to 1e-5 for both.
"""
import json
import os

import numpy as np
import torch

TOL = {torch.bfloat16: (2e-2, 1e-3), torch.float32: (1e-5, 1e-5)}


def _log(what, d_o, d_l, rows):
    """With ATTN_PARITY_LOG set, every comparison appends one JSON line
    (what, max |dO|, max |dLSE|, rows compared) to that file."""
    path = os.environ.get("ATTN_PARITY_LOG")
    if path:
        with open(path, "a") as f:
            f.write(json.dumps({"what": what, "max_abs_dO": float(d_o), "max_abs_dLSE": float(d_l),
                                "rows": int(rows)}) + "\n")


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
    _log(what, d_o, d_l, int(np.prod(o.shape[:-1])))
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


def e4m3_values():
    """All 256 e4m3 codes decoded from the format's definition (sign, 4-bit
    exponent with bias 7, 3-bit mantissa, subnormals at exponent 0, NaN at
    exponent 15 with mantissa 7)."""
    out = np.empty(256)
    for c in range(256):
        s = -1.0 if c & 0x80 else 1.0
        e, m = (c >> 3) & 0xF, c & 7
        if e == 15 and m == 7:
            out[c] = np.nan
        elif e == 0:
            out[c] = s * (m / 8.0) * 2.0 ** -6
        else:
            out[c] = s * (1.0 + m / 8.0) * 2.0 ** (e - 7)
    return out


def check_rotated_codes(codes_g, scales_g, x, signs, oracle_mod, block=128, max_frac=0.01):
    """GPU codes and scales of the rotated block quantiser against the
    oracle's: the oracle rotates exactly (float64) and rounds once to
    float32; a float32 evaluation of the rotation (the kernel's butterflies)
    may differ by the rounding of its order of evaluation, bounded by
    oracle.rotation_error_bound E.  So a scale may differ by the relative
    amount E_max / amax (+ a few ulps), and a code may differ from the
    oracle's only by one e4m3 step, only where the exact scaled value lies
    within that error of the midpoint between the two codes.  Returns the
    number of differing codes (at most max_frac of all)."""
    u = 2.0 ** -24
    codes_g = np.asarray(codes_g, np.uint8)
    scales_g = np.asarray(scales_g, np.float64)
    y = oracle_mod.hadamard_rotate(x, signs)                   # [B, N, H, d] float64
    E = oracle_mod.rotation_error_bound(x)[..., 0]            # [B, N, H]
    rc, rs = oracle_mod.quantize_fp8_blocks_rotated(x, signs, block)
    B, N, H, d = y.shape
    c = float(np.float32(1.0 / np.sqrt(np.float64(d))))
    vals = e4m3_values()
    order = np.sort(vals[~np.isnan(vals)])
    rank = {v: i for i, v in enumerate(np.unique(order))}
    n_diff = 0
    for b in range(B):
        for h in range(H):
            for bi in range((N + block - 1) // block):
                r0, r1 = bi * block, min(N, (bi + 1) * block)
                yb = y[b, r0:r1, h]                            # [rows, d]
                amax = np.abs(yb).max()
                sg, so = scales_g[b, h, bi], float(rs[b, h, bi])
                if amax == 0.0:
                    assert sg == so and np.all(codes_g[b, r0:r1, h] == 0), (b, h, bi)
                    continue
                emax = E[b, r0:r1, h].max()
                rel = emax / amax + 4 * u
                assert abs(sg - so) <= so * rel, ("scale", b, h, bi, sg, so)
                cg, co = codes_g[b, r0:r1, h], rc[b, r0:r1, h]
                bad = np.argwhere(cg != co)
                n_diff += len(bad)
                for i, j in bad:
                    vg, vo = vals[cg[i, j]], vals[co[i, j]]
                    if vg == vo:  # +0 and -0: a value below every code, of either sign
                        continue
                    assert abs(rank[abs(vg)] - rank[abs(vo)]) == 1 and np.sign(vg) * np.sign(vo) >= 0, \
                        ("codes not adjacent", b, r0 + i, h, j, vg, vo)
                    z = yb[i, j] * 448.0 / amax                # exact scaled value
                    tol = E[b, r0 + i, h] * 448.0 / amax + abs(z) * rel + 1e-12
                    assert abs(abs(z) - 0.5 * (abs(vg) + abs(vo))) <= tol, \
                        ("code differs away from a rounding boundary", b, r0 + i, h, j, z, vg, vo)
    assert n_diff <= max_frac * codes_g.size, n_diff
    return n_diff


def check_fp8_pv(o, lse, ro, rl, rabs, vabs_sum, what):
    """The e4m3 P V bar against the oracle on the dequantised inputs: LSE
    within attn_fwd's 1e-3 (l sums the unrounded P), and per element
    |dO_ic| <= 2^-4 sum_j w_ij |v_jc| + 2^-18 sum_j |v_jc| + 2e-2: rounding
    256 P to e4m3 (nearest even) moves each weight by at most half a step,
    2^-4 of it, or by 2^-18 below the normal range (2^-14); the sums over
    keys are bounded by all keys of the head; 2e-2 is attn_fwd's bf16 bar."""
    og = o.float().cpu().numpy().astype(np.float64)
    lg = lse.float().cpu().numpy().astype(np.float64)
    fin = np.isfinite(rl)
    assert np.array_equal(np.isfinite(lg), fin), what
    assert np.all(lg[~fin] == rl[~fin]), what
    d_l = np.abs(lg[fin] - rl[fin]).max() if fin.any() else 0.0
    assert d_l <= 1e-3, what
    bound = 2.0 ** -4 * (1 + 1e-3) * rabs + 2.0 ** -18 * vabs_sum + 2e-2
    err = np.abs(og - ro)
    assert np.all(np.isfinite(og)), what
    _log(what, err.max(), d_l, int(np.prod(og.shape[:-1])))
    assert np.all(err <= bound), "%s: worst excess %.3g" % (what, (err - bound).max())
    return err.max()
