"""The oracle's pins catch plausible mistakes (no GPU).

The pins in test_oracle.py are run here against stand-ins for the oracle: a
plain float64 restatement of algorithm 0 (Lecture 11 - Kernel Optimization
Techniques, section 2: materialise the scores, stable softmax, P V) into
which one mistake at a time is planted -- a dropped scale, the wrong causal
alignment or an off-by-one mask, the wrong GQA head, a missing
normalisation, the log-sum-exp without its max or in base 2, V read one key
off, the score matrix transposed, masked scores filled with 0 instead of
-inf -- for the log-sum-exp merge (section 3.2 in lse form), merges with
the max in place of the log-sum-exp, unweighted or unnormalised sums, or a
part left out -- and for decode over a block table (section 9), a slot past
the length read, an empty sequence attended, the pages taken in reverse
order or positions laid out slot-major; for the backward (section 5.1), dS
without the D term, dV from dS, dQ without the scale, dK from P, or a KV
head that gets the gradient of only one of its query heads.  Every planted mistake must fail at least one pin, and
the same restatement without a mistake must pass them all, so the pins are
neither vacuous nor too strict for a correct oracle."""
import math
import types

import numpy as np
import pytest
import torch

import test_oracle as pins

# pins that exercise the forward oracle (attn_fwd) and the merge (merge_lse)
FWD_PINS = [
    pins.test_zero_query_gives_mean_of_values,
    pins.test_dominant_score_selects_one_value_row,
    pins.test_probabilities_sum_to_one_and_convex_hull,
    pins.test_shift_invariance,
    pins.test_brute_force_tiny,
    pins.test_causal_alignment_readings,
    pins.test_empty_rows,
    pins.test_gqa_head_mapping,
]
MERGE_PINS = [
    pins.test_merge_lse_closed_forms,
    pins.test_decode_splits_merge_to_direct,
]
PAGED_PINS = [
    pins.test_paged_decode_zero_query_is_mean_of_named_rows,
    pins.test_paged_decode_dominant_key_selects_its_row,
    pins.test_paged_decode_ignores_slots_past_the_length,
]
BWD_PINS = [
    pins.test_backward_matches_finite_differences,
    pins.test_backward_gqa_sums_over_the_group,
]


def _param_sets(fn):
    """The argument tuples of a pin's parametrisation (one empty tuple if none)."""
    for mark in getattr(fn, "pytestmark", []):
        if mark.name == "parametrize":
            names, values = mark.args[0], mark.args[1]
            n = len([x for x in names.split(",") if x.strip()]) if isinstance(names, str) else len(names)
            return [tuple(v) if n > 1 else (v,) for v in values]
    return [()]


def _failed_pins(module, battery):
    """Names of the pins (any parametrisation) that reject `module`."""
    failed = []
    for fn in battery:
        for args in _param_sets(fn):
            try:
                fn(module, *args)
            except AssertionError:
                failed.append(fn.__name__)
                break
    return failed


def _f64(x):
    if isinstance(x, torch.Tensor):
        return x.float().numpy().astype(np.float64)
    return np.asarray(x, np.float32).astype(np.float64)


def _alg0(q, k, v, causal, scale, slip=None):
    """Algorithm 0 in float64, one (sequence, head) at a time, with an
    optional planted mistake.  q [B, Nq, Hq, d], k/v [B, Nk, Hkv, d];
    returns (o [B, Nq, Hq, d], lse [B, Hq, Nq])."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, Nq, Hq, d = q.shape
    Nk, Hkv = k.shape[1], k.shape[2]
    G = Hq // Hkv
    o = np.zeros((B, Nq, Hq, d))
    lse = np.zeros((B, Hq, Nq))
    i = np.arange(Nq)[:, None]
    j = np.arange(Nk)[None, :]
    if not causal:
        allowed = np.ones((Nq, Nk), bool)
    elif slip == "top_left":
        allowed = j <= i
    elif slip == "off_by_one":
        allowed = j < i + (Nk - Nq)
    else:
        allowed = j <= i + (Nk - Nq)
    for b in range(B):
        for h in range(Hq):
            g = h % Hkv if slip == "gqa" else h // G
            kk, vv = k[b, :, g], v[b, :, g]
            if slip == "v_shift":
                vv = np.roll(vv, -1, axis=0)
            s = q[b, :, h] @ kk.T
            if slip == "transpose" and Nq == Nk:
                s = s.T
            if slip != "scale":
                s = s * scale
            s = np.where(allowed, s, 0.0 if slip == "fill_zero" else -np.inf)
            m = s.max(axis=1, keepdims=True)
            has = np.isfinite(m[:, 0])
            msafe = np.where(np.isfinite(m), m, 0.0)
            e = np.exp(s - msafe)
            ell = e.sum(axis=1)
            out = e @ vv
            if slip != "no_norm":
                out = out / np.where(has, ell, 1.0)[:, None]
            with np.errstate(divide="ignore"):  # rows with no allowed key: ell = 0
                if slip == "lse_no_max":
                    ls = np.log(ell)
                elif slip == "lse_log2":
                    ls = msafe[:, 0] + np.log2(ell)
                else:
                    ls = msafe[:, 0] + np.log(ell)
            o[b, :, h] = np.where(has[:, None], out, 0.0)
            lse[b, h] = np.where(has, ls, -np.inf)
    return o, lse


def _merge(o_parts, lse_parts, slip=None):
    """LSE-form merge with an optional planted mistake: o_parts [P, rows, d],
    lse_parts [P, rows]."""
    o_parts = np.asarray(o_parts, np.float64)
    lse_parts = np.asarray(lse_parts, np.float64)
    if slip == "drop_last":
        o_parts, lse_parts = o_parts[:-1], lse_parts[:-1]
    P, rows, d = o_parts.shape
    o = np.zeros((rows, d))
    lse = np.full((rows,), -np.inf)
    for r in range(rows):
        ls = lse_parts[:, r]
        live = np.isfinite(ls)
        if not live.any():
            continue
        M = ls[live].max()
        w = np.where(live, np.exp(np.where(live, ls, M) - M), 0.0)
        if slip == "unweighted":
            o[r] = o_parts[live, r].mean(axis=0)
        elif slip == "unnormalised":
            o[r] = (w[:, None] * o_parts[:, r]).sum(axis=0)
        else:
            o[r] = (w[:, None] * o_parts[:, r]).sum(axis=0) / w.sum()
        lse[r] = M if slip == "max_for_lse" else M + math.log(w.sum())
    return o, lse


def _paged(oracle_mod, q, kp, vp, table, lens, scale, slip=None):
    """Decode over a block table (Lecture 11, section 9) as the plain
    gather-then-attend, with an optional planted mistake: position j of
    sequence b is slot j % page_size of page table[b, j // page_size]."""
    q = np.asarray(q, np.float32)
    kp, vp = np.asarray(kp, np.float32), np.asarray(vp, np.float32)
    B, _, Hq, d = q.shape
    ps, Hkv = kp.shape[1], kp.shape[2]
    o = np.zeros((B, 1, Hq, d))
    lse = np.full((B, Hq), -np.inf)
    for b in range(B):
        L = int(lens[b])
        if slip == "one_past_the_length":  # (while the table has a slot for it)
            L = min(L + 1, table.shape[1] * ps)
        if L <= 0 and slip != "empty_attends":
            continue
        npg = (L + ps - 1) // ps
        pages = list(table[b, :npg])
        if slip == "pages_reversed":
            pages = pages[::-1]
        if slip == "slot_major":  # position j -> page j % npg, slot j // npg
            pos = [(pages[j % npg], j // npg) for j in range(L)]
        else:
            pos = [(pages[j // ps], j % ps) for j in range(L)]
        kb = np.array([kp[pg, r] for pg, r in pos], np.float32).reshape(1, L, Hkv, d)
        vb = np.array([vp[pg, r] for pg, r in pos], np.float32).reshape(1, L, Hkv, d)
        if L == 0:  # the slip: attend over nothing (0/0)
            o[b] = np.nan
            lse[b] = np.nan
            continue
        ob, lb = oracle_mod.attn_fwd(q[b:b + 1], kb, vb, False, scale)
        o[b] = ob[0]
        lse[b] = lb[0, :, 0]
    return o, lse


def _bwd(q, k, v, do, causal, scale, slip=None):
    """The gradients of Lecture 11, section 5.1 in float64 with an optional
    planted mistake: P = softmax(scale S), dV = P^T dO, dP = dO V^T,
    D = rowsum(dO o O), dS = P o (dP - D), dQ = scale dS K, dK = scale dS^T Q,
    each KV head summing over its query heads."""
    q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(do)
    B, Nq, Hq, d = q.shape
    Nk, Hkv = k.shape[1], k.shape[2]
    G = Hq // Hkv
    dq, dk, dv = np.zeros(q.shape), np.zeros(k.shape), np.zeros(v.shape)
    allowed = (np.arange(Nk)[None, :] <= np.arange(Nq)[:, None] + (Nk - Nq)) if causal else \
        np.ones((Nq, Nk), bool)
    for b in range(B):
        for h in range(Hq):
            g = h // G
            if slip == "one_head_per_group" and h % G != 0:
                continue
            s = np.where(allowed, scale * (q[b, :, h] @ k[b, :, g].T), -np.inf)
            m = s.max(axis=1, keepdims=True)
            m = np.where(np.isfinite(m), m, 0.0)
            e = np.exp(s - m)
            ell = e.sum(axis=1, keepdims=True)
            P = np.where(ell > 0, e / np.where(ell > 0, ell, 1.0), 0.0)
            O = P @ v[b, :, g]
            dO = do[b, :, h]
            dP = dO @ v[b, :, g].T
            Dv = (dO * O).sum(axis=1, keepdims=True)
            dS = P * dP if slip == "no_D" else P * (dP - Dv)
            dv[b, :, g] += (dS if slip == "dv_from_ds" else P).T @ dO
            dq[b, :, h] = (1.0 if slip == "dq_unscaled" else scale) * dS @ k[b, :, g]
            dk[b, :, g] += scale * (P if slip == "dk_from_p" else dS).T @ q[b, :, h]
    return dq, dk, dv


def _stand_in(oracle_mod, **overrides):
    """The oracle module with some functions replaced."""
    ns = {n: getattr(oracle_mod, n) for n in dir(oracle_mod) if not n.startswith("_")}
    ns.update(overrides)
    return types.SimpleNamespace(**ns)


FWD_SLIPS = ["scale", "top_left", "off_by_one", "gqa", "no_norm", "lse_no_max", "lse_log2", "v_shift",
             "transpose", "fill_zero"]
MERGE_SLIPS = ["max_for_lse", "unweighted", "unnormalised", "drop_last"]
PAGED_SLIPS = ["one_past_the_length", "empty_attends", "pages_reversed", "slot_major"]
BWD_SLIPS = ["no_D", "dv_from_ds", "dq_unscaled", "dk_from_p", "one_head_per_group"]


def test_restatement_without_a_slip_passes_every_pin(oracle_mod):
    fwd = _stand_in(oracle_mod, attn_fwd=lambda q, k, v, c, s: _alg0(q, k, v, c, s))
    assert _failed_pins(fwd, FWD_PINS) == []
    mrg = _stand_in(oracle_mod, merge_lse=lambda o, l: _merge(o, l))
    assert _failed_pins(mrg, MERGE_PINS) == []
    pgd = _stand_in(oracle_mod, decode_paged=lambda *a: _paged(oracle_mod, *a))
    assert _failed_pins(pgd, PAGED_PINS) == []
    bwd = _stand_in(oracle_mod, attn_bwd=lambda *a: _bwd(*a))
    assert _failed_pins(bwd, BWD_PINS) == []


@pytest.mark.parametrize("slip", FWD_SLIPS)
def test_planted_forward_slip_fails_a_pin(oracle_mod, slip):
    fwd = _stand_in(oracle_mod, attn_fwd=lambda q, k, v, c, s: _alg0(q, k, v, c, s, slip))
    assert _failed_pins(fwd, FWD_PINS), "no pin rejects the forward with slip %r" % slip


@pytest.mark.parametrize("slip", MERGE_SLIPS)
def test_planted_merge_slip_fails_a_pin(oracle_mod, slip):
    mrg = _stand_in(oracle_mod, merge_lse=lambda o, l: _merge(o, l, slip))
    assert _failed_pins(mrg, MERGE_PINS), "no pin rejects the merge with slip %r" % slip


@pytest.mark.parametrize("slip", PAGED_SLIPS)
def test_planted_paged_slip_fails_a_pin(oracle_mod, slip):
    pgd = _stand_in(oracle_mod, decode_paged=lambda *a: _paged(oracle_mod, *a, slip=slip))
    assert _failed_pins(pgd, PAGED_PINS), "no pin rejects the paged decode with slip %r" % slip


@pytest.mark.parametrize("slip", BWD_SLIPS)
def test_planted_backward_slip_fails_a_pin(oracle_mod, slip):
    bwd = _stand_in(oracle_mod, attn_bwd=lambda *a: _bwd(*a, slip=slip))
    assert _failed_pins(bwd, BWD_PINS), "no pin rejects the backward with slip %r" % slip
