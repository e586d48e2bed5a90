"""Pins for the CPU oracle (no GPU).

Each test checks the oracle against something other than itself: numbers
printed in the lecture notes (tests/golden), closed forms, invariants, and
brute force on tiny inputs written out with Python loops.  A plausible slip in
the oracle (a dropped term, a wrong sign or index, a transposed operand, a
wrong causal offset or GQA mapping) fails at least one of them.
"""
import json
import math
import os
import random

import numpy as np
import pytest
import torch

from exact_attention_62_gb300.inputs import make_qkv

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# ---------------------------------------------------------------- worked numbers

def test_online_softmax_worked_example(oracle_mod):
    """Lecture 11, exercise 1: blocks [1,3] then [2,5]."""
    g = _golden("online_softmax_ex1.json")
    m, l, a = oracle_mod.online_trace(g["scores"], g["block"])
    dec = g["decimals"]
    for b, want in enumerate(g["after_block"]):
        assert round(m[b], dec) == want["m"]
        assert round(l[b], dec) == want["l"]
        if "alpha" in want:
            assert round(a[b], dec) == want["alpha"]
    assert round(l[-1], dec) == g["one_shot_l_at_m5"]


def test_state_merge_worked_example(oracle_mod):
    """The two blocks of exercise 1 merged as partial states give the one-shot l."""
    g = _golden("online_softmax_ex1.json")
    x = g["scores"]

    def state(seg):
        m = max(seg)
        return m, sum(math.exp(s - m) for s in seg), np.zeros(1)

    m, l, _ = oracle_mod.state_merge(state(x[:2]), state(x[2:]))
    assert m == 5.0
    assert round(l, g["decimals"]) == g["one_shot_l_at_m5"]


def test_causal_block_fraction(oracle_mod):
    """Lecture 11 section 5.3: computed-block fraction at N=4096, blocks 64/128/256."""
    g = _golden("causal_block_fraction.json")
    N = g["N"]
    q, k, v = make_qkv(1, 1, 1, N, N, 2, seed=3, dtype=torch.float32)
    for blk, want in g["fractions"].items():
        blk = int(blk)
        _, _, nb = oracle_mod.attn_fwd_tiled(q, k, v, True, 1.0, blk, blk)
        T = N // blk
        assert nb == T * (T + 1) // 2
        assert round(nb / (T * T), g["decimals"]) == want


# ---------------------------------------------------------------- closed forms

@pytest.mark.parametrize("causal,Nq,Nk,Hq,Hkv", [
    (False, 5, 9, 4, 2), (True, 9, 9, 2, 2), (True, 3, 11, 6, 3), (True, 7, 4, 2, 1)])
def test_zero_query_gives_mean_of_values(oracle_mod, causal, Nq, Nk, Hq, Hkv):
    """Q = 0 makes every allowed score equal: O = mean of the allowed V rows,
    LSE = ln(#allowed keys)."""
    B, d = 2, 8
    _, k, v = make_qkv(B, Hq, Hkv, Nq, Nk, d, seed=11, dtype=torch.float32)
    q = torch.zeros(B, Nq, Hq, d)
    o, lse = oracle_mod.attn_fwd(q, k, v, causal, 0.37)
    G = Hq // Hkv
    vv = v.double().numpy()
    for b in range(B):
        for h in range(Hq):
            for i in range(Nq):
                last = min(Nk - 1, i + Nk - Nq) if causal else Nk - 1
                if last < 0:
                    assert np.all(o[b, i, h] == 0) and lse[b, h, i] == -np.inf
                    continue
                want = vv[b, :last + 1, h // G].mean(axis=0)
                np.testing.assert_allclose(o[b, i, h], want, atol=1e-13, rtol=0)
                assert abs(lse[b, h, i] - math.log(last + 1)) < 1e-13


def test_dominant_score_selects_one_value_row(oracle_mod):
    """A score 900 above all others puts all weight on that key: O = v_j*,
    LSE = s_j* (exp(-900) underflows to zero in double)."""
    B, Hq, Hkv, Nq, Nk, d = 1, 2, 1, 6, 6, 8
    k = torch.zeros(B, Nk, Hkv, d)
    q = torch.zeros(B, Nq, Hq, d)
    perm = [3, 0, 5, 1, 4, 2]
    for j in range(Nk):
        k[0, j, 0, j] = 30.0
    for i in range(Nq):
        for h in range(Hq):
            q[0, i, h, perm[(i + h) % Nk]] = 30.0
    _, _, v = make_qkv(B, Hq, Hkv, Nq, Nk, d, seed=5, dtype=torch.float32)
    o, lse = oracle_mod.attn_fwd(q, k, v, False, 1.0)
    for i in range(Nq):
        for h in range(Hq):
            j = perm[(i + h) % Nk]
            np.testing.assert_array_equal(o[0, i, h], v[0, j, 0].double().numpy())
            assert lse[0, h, i] == 900.0


def test_probabilities_sum_to_one_and_convex_hull(oracle_mod):
    """V = 1 gives O = 1 (rows of P sum to 1); for random V every output
    coordinate lies between the min and max of the allowed V rows."""
    B, Hq, Hkv, Nq, Nk, d = 2, 4, 2, 13, 17, 16
    q, k, v = make_qkv(B, Hq, Hkv, Nq, Nk, d, seed=21, dtype=torch.float32)
    for causal in (False, True):
        o1, _ = oracle_mod.attn_fwd(q, k, torch.ones_like(v), causal, 0.25)
        np.testing.assert_allclose(o1, 1.0, atol=1e-14, rtol=0)
        o, _ = oracle_mod.attn_fwd(q, k, v, causal, 0.25)
        vv = v.double().numpy()
        for b in range(B):
            for h in range(Hq):
                for i in range(Nq):
                    last = min(Nk - 1, i + Nk - Nq) if causal else Nk - 1
                    rows = vv[b, :last + 1, h // (Hq // Hkv)]
                    assert np.all(o[b, i, h] >= rows.min(axis=0) - 1e-14)
                    assert np.all(o[b, i, h] <= rows.max(axis=0) + 1e-14)


def test_shift_invariance(oracle_mod):
    """Adding w to every key adds scale*(q_i . w) to every score of row i:
    O is unchanged and LSE shifts by exactly that constant."""
    B, Hq, Hkv, Nq, Nk, d = 1, 2, 2, 7, 9, 8
    rng = np.random.default_rng(0)
    # dyadic values so that k + w is exact in float32
    q = torch.tensor(rng.integers(-8, 9, (B, Nq, Hq, d)) / 8.0, dtype=torch.float32)
    k = torch.tensor(rng.integers(-8, 9, (B, Nk, Hkv, d)) / 8.0, dtype=torch.float32)
    v = torch.tensor(rng.standard_normal((B, Nk, Hkv, d)), dtype=torch.float32)
    w = torch.tensor(rng.integers(-4, 5, (Hkv, d)) / 4.0, dtype=torch.float32)
    scale = 0.5
    for causal in (False, True):
        o0, l0 = oracle_mod.attn_fwd(q, k, v, causal, scale)
        o1, l1 = oracle_mod.attn_fwd(q, k + w, v, causal, scale)
        np.testing.assert_allclose(o1, o0, atol=1e-12, rtol=0)
        G = Hq // Hkv
        for h in range(Hq):
            shift = scale * (q[0, :, h].double() @ w[h // G].double()).numpy()
            np.testing.assert_allclose(l1[0, h], l0[0, h] + shift, atol=1e-11, rtol=0)


# ---------------------------------------------------------------- brute force

def _brute(q, k, v, causal, scale):
    """Textbook attention with explicit Python loops (no max subtraction:
    inputs are tiny and bounded, so exp cannot overflow)."""
    B, Nq, Hq, d = q.shape
    _, Nk, Hkv, _ = k.shape
    G = Hq // Hkv
    o = np.zeros((B, Nq, Hq, d))
    lse = np.zeros((B, Hq, Nq))
    for b in range(B):
        for h in range(Hq):
            g = h // G
            for i in range(Nq):
                allowed = [j for j in range(Nk) if (not causal or j <= i + Nk - Nq)]
                if not allowed:
                    lse[b, h, i] = -math.inf
                    continue
                e = {}
                for j in allowed:
                    s = 0.0
                    for t in range(d):
                        s += float(q[b, i, h, t]) * float(k[b, j, g, t])
                    e[j] = math.exp(scale * s)
                z = sum(e.values())
                for t in range(d):
                    o[b, i, h, t] = sum(e[j] / z * float(v[b, j, g, t]) for j in allowed)
                lse[b, h, i] = math.log(z)
    return o, lse


@pytest.mark.parametrize("B,Hq,Hkv,Nq,Nk,d,causal", [
    (1, 1, 1, 1, 1, 1, False), (1, 1, 1, 4, 4, 4, True), (2, 2, 1, 3, 4, 2, True),
    (1, 4, 2, 4, 2, 3, True), (2, 3, 3, 2, 4, 4, False), (1, 2, 2, 4, 3, 1, False)])
def test_brute_force_tiny(oracle_mod, B, Hq, Hkv, Nq, Nk, d, causal):
    q, k, v = make_qkv(B, Hq, Hkv, Nq, Nk, d, seed=B * 100 + Nq * 10 + d,
                       dtype=torch.float32)
    scale = 0.7
    o, lse = oracle_mod.attn_fwd(q, k, v, causal, scale)
    ob, lb = _brute(q.numpy(), k.numpy(), v.numpy(), causal, scale)
    np.testing.assert_allclose(o, ob, atol=1e-13, rtol=0)
    np.testing.assert_allclose(lse, lb, atol=1e-13, rtol=0)


# ---------------------------------------------------------------- agreements

@pytest.mark.parametrize("B,Hq,Hkv,Nq,Nk,d,causal,Br,Bc", [
    (2, 4, 2, 37, 37, 16, True, 8, 8),
    (1, 3, 3, 50, 70, 8, False, 16, 12),
    (1, 2, 1, 1, 1000, 8, True, 64, 128),     # decode case of the lecture demo
    (1, 2, 2, 20, 9, 4, True, 4, 4),          # Nq > Nk: leading rows are empty
    (2, 6, 2, 33, 65, 32, True, 16, 32)])
def test_tiled_online_matches_plain(oracle_mod, B, Hq, Hkv, Nq, Nk, d, causal, Br, Bc):
    """Lecture 11 section 4.1: the tiled online forward equals algorithm 0."""
    q, k, v = make_qkv(B, Hq, Hkv, Nq, Nk, d, seed=Nq + Nk, dtype=torch.float32)
    o, lse = oracle_mod.attn_fwd(q, k, v, causal, 1.0 / math.sqrt(d))
    ot, lt, _ = oracle_mod.attn_fwd_tiled(q, k, v, causal, 1.0 / math.sqrt(d), Br, Bc)
    np.testing.assert_allclose(ot, o, atol=1e-12, rtol=0)
    fin = np.isfinite(lse)
    assert np.array_equal(fin, np.isfinite(lt))
    np.testing.assert_allclose(lt[fin], lse[fin], atol=1e-12, rtol=1e-12)


def test_rows_match_full(oracle_mod):
    q, k, v = make_qkv(2, 4, 1, 30, 40, 16, seed=9)
    o, lse = oracle_mod.attn_fwd(q, k, v, True, 0.25)
    rows = [(0, 0, 0), (1, 3, 29), (0, 2, 17), (1, 1, 5)]
    os_, ls = oracle_mod.attn_rows(q, k, v, True, 0.25, rows)
    for n, (b, h, i) in enumerate(rows):
        np.testing.assert_array_equal(os_[n], o[b, i, h])
        assert ls[n] == lse[b, h, i]


def test_segment_merge_associative(oracle_mod):
    """Lecture 11 section 3.2: a row of 3000 keys cut into 12 random segments;
    sequential, tree and shuffled merges all equal the one-shot state."""
    Nk, d = 3000, 16
    q, k, v = make_qkv(1, 1, 1, 1, Nk, d, seed=12, dtype=torch.float32)
    rnd = random.Random(4)
    cuts = sorted(rnd.sample(range(1, Nk), 11))
    bounds = list(zip([0] + cuts, cuts + [Nk]))
    segs = [oracle_mod.segment_state(q, k, v, False, 0.3, 0, 0, 0, a, b) for a, b in bounds]
    full = oracle_mod.segment_state(q, k, v, False, 0.3, 0, 0, 0, 0, Nk)

    def seq(states):
        acc = states[0]
        for s in states[1:]:
            acc = oracle_mod.state_merge(acc, s)
        return acc

    def tree(states):
        while len(states) > 1:
            nxt = [oracle_mod.state_merge(states[i], states[i + 1])
                   for i in range(0, len(states) - 1, 2)]
            if len(states) % 2:
                nxt.append(states[-1])
            states = nxt
        return states[0]

    shuffled = segs[:]
    rnd.shuffle(shuffled)
    o_full, lse_full = oracle_mod.attn_rows(q, k, v, False, 0.3, [(0, 0, 0)])
    for m, l, acc in (seq(segs), tree(segs), seq(shuffled)):
        assert abs(m - full[0]) == 0.0
        assert abs(l - full[1]) <= 1e-12 * full[1]
        np.testing.assert_allclose(acc, full[2], atol=1e-12 * full[1], rtol=0)
        np.testing.assert_allclose(acc / l, o_full[0], atol=1e-12, rtol=0)
        assert abs(m + math.log(l) - lse_full[0]) <= 1e-12


@pytest.mark.parametrize("nsplit", [1, 7, 64, 1000])
def test_decode_splits_merge_to_direct(oracle_mod, nsplit):
    """Lecture 11 section 6.2: 1, 7, 64 and 1000 segments merged by log-sum-exp
    equal the direct result."""
    B, Hq, Hkv, Nk, d = 2, 8, 2, 1000, 32
    q, k, v = make_qkv(B, Hq, Hkv, 1, Nk, d, seed=nsplit)
    scale = 1.0 / math.sqrt(d)
    o, lse = oracle_mod.attn_fwd(q, k, v, False, scale)
    op, lp = oracle_mod.decode_split(q, k, v, scale, nsplit)
    om, lm = oracle_mod.merge_lse(op, lp)
    np.testing.assert_allclose(om, o.reshape(B * Hq, d), atol=1e-12, rtol=0)
    np.testing.assert_allclose(lm, lse.reshape(B * Hq), atol=1e-12, rtol=0)


def test_merge_lse_closed_forms(oracle_mod):
    """Two parts with equal lse a give lse = a + ln 2 and the mean output;
    empty parts (lse = -inf) are ignored; all-empty rows give 0 and -inf."""
    o_parts = np.array([[[1.0, 2.0], [5.0, 5.0], [0.0, 0.0]],
                        [[3.0, -2.0], [0.0, 0.0], [0.0, 0.0]]])
    lse_parts = np.array([[0.5, 1.25, -np.inf], [0.5, -np.inf, -np.inf]])
    o, lse = oracle_mod.merge_lse(o_parts, lse_parts)
    np.testing.assert_allclose(o[0], [2.0, 0.0], atol=1e-15)
    assert abs(lse[0] - (0.5 + math.log(2.0))) < 1e-15
    np.testing.assert_array_equal(o[1], [5.0, 5.0])
    assert lse[1] == 1.25
    np.testing.assert_array_equal(o[2], [0.0, 0.0])
    assert lse[2] == -np.inf


# ---------------------------------------------------------------- readings

def test_causal_alignment_readings(oracle_mod):
    """Bottom-right alignment: one query over 1000 keys sees every key (the
    decode case of the lecture's demo); with Nq == Nk, row 0 sees only key 0."""
    q, k, v = make_qkv(1, 2, 2, 1, 1000, 16, seed=2)
    oc, lc = oracle_mod.attn_fwd(q, k, v, True, 0.25)
    on, ln = oracle_mod.attn_fwd(q, k, v, False, 0.25)
    np.testing.assert_array_equal(oc, on)
    np.testing.assert_array_equal(lc, ln)
    q, k, v = make_qkv(1, 2, 2, 8, 8, 16, seed=2, dtype=torch.float32)
    o, lse = oracle_mod.attn_fwd(q, k, v, True, 0.25)
    for h in range(2):
        np.testing.assert_array_equal(o[0, 0, h], v[0, 0, h].double().numpy())
        s00 = 0.25 * float(q[0, 0, h].double() @ k[0, 0, h].double())
        assert abs(lse[0, h, 0] - s00) < 1e-14


def test_empty_rows(oracle_mod):
    """Causal with Nq > Nk: rows i < Nq - Nk have no allowed key: O = 0, LSE = -inf."""
    q, k, v = make_qkv(1, 2, 1, 10, 4, 8, seed=3)
    o, lse = oracle_mod.attn_fwd(q, k, v, True, 0.5)
    assert np.all(o[0, :6] == 0.0)
    assert np.all(lse[:, :, :6] == -np.inf)
    assert np.all(np.isfinite(lse[:, :, 6:]))


def test_gqa_head_mapping(oracle_mod):
    """Query head h reads key/value head h // (Hq/Hkv): equal to plain
    multi-head attention with each kv head repeated G times."""
    B, Hq, Hkv, N, d = 1, 8, 2, 12, 8
    q, k, v = make_qkv(B, Hq, Hkv, N, N, d, seed=6)
    o, lse = oracle_mod.attn_fwd(q, k, v, True, 0.3)
    kr = k.repeat_interleave(Hq // Hkv, dim=2)
    vr = v.repeat_interleave(Hq // Hkv, dim=2)
    o2, l2 = oracle_mod.attn_fwd(q, kr, vr, True, 0.3)
    np.testing.assert_array_equal(o, o2)
    np.testing.assert_array_equal(lse, l2)
    # and a different mapping (h % Hkv) would differ
    kw = k[:, :, [h % Hkv for h in range(Hq)]]
    vw = v[:, :, [h % Hkv for h in range(Hq)]]
    o3, _ = oracle_mod.attn_fwd(q, kw, vw, True, 0.3)
    assert np.abs(o3 - o).max() > 1e-3


# ---------------------------------------------------------------- paged decode
def _paged_case(seed, B=3, Hq=4, Hkv=2, d=8, ps=4, num_pages=12, max_pages=4):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((B, 1, Hq, d)).astype(np.float32)
    kp = rng.standard_normal((num_pages, ps, Hkv, d)).astype(np.float32)
    vp = rng.standard_normal((num_pages, ps, Hkv, d)).astype(np.float32)
    table = rng.permutation(num_pages)[:B * max_pages].reshape(B, max_pages)
    return q, kp, vp, table


def test_paged_decode_zero_query_is_mean_of_named_rows(oracle_mod):
    """q = 0: every allowed key has the same score, so O is the mean of exactly
    the V rows the table names among the first L positions, and LSE = ln L
    (catches a wrong page, an off-by-one at the partial last page, and the
    empty sequence)."""
    q, kp, vp, table = _paged_case(1)
    q[:] = 0.0
    lens = np.array([7, 16, 0])
    o, lse = oracle_mod.decode_paged(q, kp, vp, table, lens, 0.5)
    ps, G = kp.shape[1], 2
    for b, L in enumerate(lens):
        if L == 0:
            assert np.all(o[b] == 0.0) and np.all(np.isneginf(lse[b]))
            continue
        rows = [(table[b, j // ps], j % ps) for j in range(L)]
        for hq in range(q.shape[2]):
            want = np.mean([vp[pg, r, hq // G] for pg, r in rows], axis=0)
            assert np.allclose(o[b, 0, hq], want, atol=1e-12)
            assert lse[b, hq] == pytest.approx(math.log(L), abs=1e-12)


def test_paged_decode_dominant_key_selects_its_row(oracle_mod):
    q, kp, vp, table = _paged_case(2)
    lens = np.array([9, 13, 5])
    b, j = 1, 10                      # position 10 of sequence 1
    pg, r = table[b, j // 4], j % 4
    kp[pg, r, :, :] = 0.0
    kp[pg, r, 0, 0] = 10.0            # KV head 0; other keys have |k0| of a few units
    q[b, 0, 0, :] = 0.0
    q[b, 0, 0, 0] = 200.0             # query head 0 of group 0 aims at that key
    o, _ = oracle_mod.decode_paged(q, kp, vp, table, lens, 1.0)
    assert np.allclose(o[b, 0, 0], vp[pg, r, 0], atol=1e-9)


def test_paged_decode_ignores_slots_past_the_length(oracle_mod):
    q, kp, vp, table = _paged_case(3)
    lens = np.array([6, 11, 1])
    o1, l1 = oracle_mod.decode_paged(q, kp, vp, table, lens, 0.7)
    kp2, vp2 = kp.copy(), vp.copy()
    for b, L in enumerate(lens):      # poison every slot a sequence does not own
        for j in range(L, table.shape[1] * kp.shape[1]):
            kp2[table[b, j // 4], j % 4] = np.nan
            vp2[table[b, j // 4], j % 4] = np.nan
    o2, l2 = oracle_mod.decode_paged(q, kp2, vp2, table, lens, 0.7)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


# ---------------------------------------------------------------- backward
def _bwd_case(seed, B=1, Hq=2, Hkv=1, Nq=5, Nk=6, d=3):
    rng = np.random.default_rng(seed)
    q, k, v, do = (rng.standard_normal(s).astype(np.float32)
                   for s in ((B, Nq, Hq, d), (B, Nk, Hkv, d), (B, Nk, Hkv, d), (B, Nq, Hq, d)))
    return q, k, v, do


@pytest.mark.parametrize("causal,Nq,Nk", [(False, 5, 6), (True, 5, 6), (True, 7, 4)])
def test_backward_matches_finite_differences(oracle_mod, causal, Nq, Nk):
    """Central differences of L = sum(O * dO), with O from the forward oracle,
    against the backward's dQ, dK, dV (Lecture 11 section 5.1 reports ~1e-9
    with double inputs; here inputs are float32, stepped by 2^-10, which is
    exact for them, and the forward runs in double).  The Nq > Nk causal case
    has rows with no allowed key."""
    q, k, v, do = _bwd_case(11 + Nq, Nq=Nq, Nk=Nk)
    scale = 0.7
    h = 2.0 ** -10

    def loss(qq, kk, vv):
        o, _ = oracle_mod.attn_fwd(qq, kk, vv, causal, scale)
        return float((o * do.astype(np.float64)).sum())

    dq, dk, dv = oracle_mod.attn_bwd(q, k, v, do, causal, scale)
    for name, x, grad in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        fd = np.zeros(x.shape)
        for idx in np.ndindex(*x.shape):
            xp, xm = x.copy(), x.copy()
            xp[idx] += np.float32(h)
            xm[idx] -= np.float32(h)
            args_p = {"q": (xp, k, v), "k": (q, xp, v), "v": (q, k, xp)}[name]
            args_m = {"q": (xm, k, v), "k": (q, xm, v), "v": (q, k, xm)}[name]
            fd[idx] = (loss(*args_p) - loss(*args_m)) / (2 * h)
        assert np.abs(fd - grad).max() <= 2e-6 * max(1.0, np.abs(grad).max()), name


def test_backward_gqa_sums_over_the_group(oracle_mod):
    """A KV head shared by two query heads gets the sum of the gradients it
    would get as two separate (duplicated) KV heads."""
    q, k, v, do = _bwd_case(21, Hq=2, Hkv=1, Nq=6, Nk=6, d=4)
    dq1, dk1, dv1 = oracle_mod.attn_bwd(q, k, v, do, True, 0.5)
    k2, v2 = np.repeat(k, 2, axis=2), np.repeat(v, 2, axis=2)
    dq2, dk2, dv2 = oracle_mod.attn_bwd(q, k2, v2, do, True, 0.5)
    assert np.allclose(dq1, dq2, atol=1e-13)
    assert np.allclose(dk1[:, :, 0], dk2.sum(axis=2), atol=1e-13)
    assert np.allclose(dv1[:, :, 0], dv2.sum(axis=2), atol=1e-13)


# ---------------------------------------------------------------- FP8 block quantisation
def _e4m3_value(code):
    """The e4m3 (finite-only variant) format from its definition: sign bit,
    4 exponent bits with bias 7, 3 mantissa bits, subnormals at exponent 0,
    and exponent 15 with mantissa 7 reserved for NaN."""
    s = -1.0 if code & 0x80 else 1.0
    e = (code >> 3) & 0xF
    m = code & 0x7
    if e == 15 and m == 7:
        return float("nan")
    if e == 0:
        return s * (m / 8.0) * 2.0 ** (1 - 7)
    return s * (1.0 + m / 8.0) * 2.0 ** (e - 7)


def test_fp8_codes_decode_as_the_format_defines(oracle_mod):
    codes = np.arange(256, dtype=np.uint8).reshape(1, 1, 1, 256)
    got = oracle_mod.dequantize_fp8_blocks(codes, np.ones((1, 1, 1), np.float32))
    want = np.array([_e4m3_value(c) for c in range(256)])
    both_nan = np.isnan(got.ravel()) & np.isnan(want)
    assert np.all(both_nan | (got.ravel() == want))
    assert np.nanmax(want) == oracle_mod.FP8_MAX


def test_fp8_block_quantisation_properties(oracle_mod):
    rng = np.random.default_rng(4)
    x = rng.standard_normal((2, 300, 3, 64)).astype(np.float32)
    x[1, 128:256, 2] = 0.0                      # an all-zero block
    codes, scales = oracle_mod.quantize_fp8_blocks(x)
    assert codes.dtype == np.uint8 and scales.shape == (2, 3, 3)
    assert scales[1, 2, 1] == 1.0 and np.all(codes[1, 128:256, 2] == 0)
    deq = oracle_mod.dequantize_fp8_blocks(codes, scales)
    for b in range(2):
        for h in range(3):
            for bi in range(3):
                blk = x[b, bi * 128:(bi + 1) * 128, h].astype(np.float64)
                dq = deq[b, bi * 128:(bi + 1) * 128, h]
                amax = np.abs(blk).max()
                if amax == 0:
                    continue
                # the block's largest element maps to +-448 and back to ~amax
                assert np.isclose(np.abs(dq).max(), amax, rtol=1e-6)
                # e4m3 rounding: half a step of 2^-3 relative for normals, and
                # half the subnormal step 2^-9 (times the scale) near zero
                step = np.maximum(np.abs(blk) * 2.0 ** -4, 0.5 * 2.0 ** -9 * amax / 448.0)
                assert np.all(np.abs(dq - blk) <= step * (1 + 1e-6))


def test_score_perturbation_is_the_max_score_change(oracle_mod):
    rng = np.random.default_rng(5)
    q = rng.standard_normal((1, 4, 2, 8))
    k = rng.standard_normal((1, 5, 1, 8))
    q2 = q.copy()
    q2[0, 1, 1, 0] += 0.5                       # row 1 of head 1 only
    d = oracle_mod.score_perturbation(q2, k, q, k, False, 0.25)
    assert np.all(d[0, 0] == 0) and np.all(d[0, 1, [0, 2, 3]] == 0)
    assert d[0, 1, 1] == pytest.approx(0.25 * 0.5 * np.abs(k[0, :, 0, 0]).max())


# ---------------------------------------------------------------- incoherent processing
def test_hadamard_rotation_worked_example(oracle_mod):
    """d = 4 by hand: signs (1, -1, 1, 1) make y = (1, -2, 3, 4); with the
    Sylvester matrix H_4 = [[1,1,1,1], [1,-1,1,-1], [1,1,-1,-1], [1,-1,-1,1]],
    y H = (1-2+3+4, 1+2+3-4, 1-2-3-4, 1+2-3+4) = (6, 2, -8, 4)."""
    got = oracle_mod.hadamard_rotate(np.array([[1.0, 2.0, 3.0, 4.0]]), np.array([1.0, -1.0, 1.0, 1.0]))
    assert got.tolist() == [[6.0, 2.0, -8.0, 4.0]]


@pytest.mark.parametrize("d", [2, 8, 64, 128])
def test_hadamard_rotation_is_the_sylvester_matrix(oracle_mod, d):
    """Rotating the identity with all signs +1 gives H itself: it matches the
    Sylvester construction of scipy.linalg.hadamard, has entries +-1, and
    H H^T = d I."""
    scipy_linalg = pytest.importorskip("scipy.linalg")
    H = oracle_mod.hadamard_rotate(np.eye(d), np.ones(d))
    assert np.array_equal(H, scipy_linalg.hadamard(d).astype(np.float64))
    assert np.array_equal(np.abs(H), np.ones((d, d)))
    assert np.array_equal(H @ H.T, d * np.eye(d))
    # the signs multiply the rows of H (diag(s) H)
    s = np.where(np.arange(d) % 3 == 0, -1.0, 1.0)
    assert np.array_equal(oracle_mod.hadamard_rotate(np.eye(d), s), s[:, None] * H)


def test_hadamard_rotation_keeps_dot_products_and_spreads_outliers(oracle_mod):
    rng = np.random.default_rng(6)
    d = 128
    s = rng.choice([-1.0, 1.0], size=d)
    x = rng.standard_normal((5, d)).astype(np.float32)
    y = rng.standard_normal((7, d)).astype(np.float32)
    xr = oracle_mod.hadamard_rotate(x, s)
    yr = oracle_mod.hadamard_rotate(y, s)
    # (x R)(y R)^T = x y^T with R = diag(s) H / sqrt(d) orthogonal (float64 throughout)
    exact = x.astype(np.float64) @ y.astype(np.float64).T
    assert np.allclose(xr @ yr.T / d, exact, rtol=0, atol=1e-11)
    # the rows keep their norm up to sqrt(d)
    assert np.allclose((xr ** 2).sum(axis=1), d * (x.astype(np.float64) ** 2).sum(axis=1), rtol=1e-13)
    # a single outlier feature is spread evenly over all d columns
    one = np.zeros((1, d), np.float32)
    one[0, 5] = 1000.0
    assert np.array_equal(np.abs(oracle_mod.hadamard_rotate(one, s)), np.full((1, d), 1000.0))


def _fwht_float32(x, s):
    """A float32 fast Walsh-Hadamard evaluation (butterflies h = 1, 2, ...,
    d/2), written here only to test the error bound of the oracle against
    an order of evaluation other than its own."""
    y = (np.asarray(x, np.float32) * np.asarray(s, np.float32)).astype(np.float32)
    d = y.shape[-1]
    h = 1
    while h < d:
        z = y.reshape(y.shape[:-1] + (d // (2 * h), 2, h))
        a, b = z[..., 0, :], z[..., 1, :]
        y = np.stack([a + b, a - b], axis=-2).reshape(y.shape).astype(np.float32)
        h *= 2
    return y


@pytest.mark.parametrize("d", [64, 128])
def test_rotation_error_bound_holds_for_float32_butterflies(oracle_mod, d):
    """rotation_error_bound covers a float32 butterfly evaluation on inputs
    with widely spread magnitudes (where float32 partial sums must round), and
    is not vacuous (within a few hundred ulps of the row's sum of |x|)."""
    rng = np.random.default_rng(8)
    x = (rng.standard_normal((400, d)) * np.exp2(rng.integers(-12, 12, (400, d)))).astype(np.float32)
    s = rng.choice([-1.0, 1.0], size=d)
    y = oracle_mod.hadamard_rotate(x, s)
    y32 = _fwht_float32(x, s).astype(np.float64)
    E = oracle_mod.rotation_error_bound(x)
    err = np.abs(y32 - y)
    assert np.all(err <= E)
    assert err.max() > 0                          # float32 really did round somewhere
    assert np.all(E <= 2 * 7 * 2.0 ** -24 * np.abs(x.astype(np.float64)).sum(axis=-1, keepdims=True) * 1.0001)


def test_fp8_rounding_ties_go_to_even(oracle_mod):
    """e4m3 rounding is round-to-nearest with ties to the even code, pinned
    at exact midpoints between codes.  A block whose maximum is 448 has
    scale = inv = 1, so the quantiser sees the values unchanged.  Expected
    codes, derived from the format (code = sign << 7 | (e + 7) << 3 | m):
      1.0625  between 1.0 (0x38, m=000) and 1.125 (0x39)   -> 0x38
      1.1875  between 1.125 (0x39) and 1.25 (0x3A, m=010)  -> 0x3A
      -1.0625                                               -> 0xB8
      17      between 16 (0x58) and 18 (0x59)               -> 0x58
      19      between 18 (0x59) and 20 (0x5A)               -> 0x5A
      432     between 416 (0x7D, m=101) and 448 (0x7E)      -> 0x7E (the top code)
      -432                                                  -> 0xFE
      2^-10   between 0 and the smallest subnormal 2^-9     -> 0x00
      3 2^-10 between 2^-9 (0x01) and 2^-8 (0x02)           -> 0x02
    and just above a midpoint the value rounds up:
      1.0703125 (1.0625 + 2^-7)  -> 0x39;  2^-10 (1 + 2^-7) -> 0x01."""
    vals = [448.0, 1.0625, 1.1875, -1.0625, 17.0, 19.0, 432.0, -432.0, 2.0 ** -10, 3 * 2.0 ** -10,
            1.0703125, 2.0 ** -10 * (1 + 2.0 ** -7)]
    want = [0x7E, 0x38, 0x3A, 0xB8, 0x58, 0x5A, 0x7E, 0xFE, 0x00, 0x02, 0x39, 0x01]
    x = np.zeros((1, 128, 1, 16), np.float32)
    x[0, :len(vals), 0, 0] = vals
    codes, scales = oracle_mod.quantize_fp8_blocks(x)
    assert scales[0, 0, 0] == 1.0
    assert [int(c) for c in codes[0, :len(vals), 0, 0]] == want


def test_fp8_block_maximum_saturates_at_448(oracle_mod):
    """When amax * float32(448 / amax) rounds above 448 (amax = 1.359375 in
    float32: 448.00003), the block maximum still maps to the top code 448
    (0x7E) and never to NaN, and the scale is amax / 448."""
    amax = np.float32(1.359375)
    assert np.float32(amax * (np.float32(448.0) / amax)) > 448.0
    x = np.zeros((1, 128, 1, 8), np.float32)
    x[0, 3, 0, 2], x[0, 9, 0, 5] = amax, -amax
    codes, scales = oracle_mod.quantize_fp8_blocks(x)
    assert codes[0, 3, 0, 2] == 0x7E and codes[0, 9, 0, 5] == 0xFE
    assert scales[0, 0, 0] == np.float32(amax / np.float32(448.0))


def test_rotated_quantisation_dequantises_to_the_rotated_rows(oracle_mod):
    """codes * scales of the rotated quantiser approximate x R (R orthogonal)
    to e4m3 rounding, and the scale is the plain quantiser's scale of x H
    times float32(1 / sqrt(d))."""
    rng = np.random.default_rng(7)
    d = 128
    s = rng.choice([-1.0, 1.0], size=d).astype(np.float32)
    x = rng.standard_normal((1, 200, 2, d)).astype(np.float32)
    x[0, :, 0, 9] *= 40.0                       # an outlier feature
    codes, scales = oracle_mod.quantize_fp8_blocks_rotated(x, s)
    pc, ps = oracle_mod.quantize_fp8_blocks(oracle_mod.hadamard_rotate(x, s))
    assert np.array_equal(codes, pc)
    assert np.array_equal(scales, (ps * np.float32(1.0 / np.sqrt(128.0))).astype(np.float32))
    xr = oracle_mod.hadamard_rotate(x, s).astype(np.float64) / np.sqrt(d)
    deq = oracle_mod.dequantize_fp8_blocks(codes, scales)
    for h in range(2):
        for bi in range(2):
            blk = xr[0, bi * 128:(bi + 1) * 128, h]
            amax = np.abs(blk).max()
            step = np.maximum(np.abs(blk) * 2.0 ** -4, 0.5 * 2.0 ** -9 * amax / 448.0)
            assert np.all(np.abs(deq[0, bi * 128:(bi + 1) * 128, h] - blk) <= step * (1 + 1e-5))
    # the outlier head: rotation lowers the largest relative error of a score
    # q k^T against the plain quantiser (the reason for the transform)
    k = rng.standard_normal((1, 200, 2, d)).astype(np.float32)
    k[0, :, 0, 9] *= 40.0
    kc, ks = oracle_mod.quantize_fp8_blocks_rotated(k, s)
    qd = oracle_mod.dequantize_fp8_blocks(codes, scales)
    kd = oracle_mod.dequantize_fp8_blocks(kc, ks)
    qp, kp = (oracle_mod.dequantize_fp8_blocks(*oracle_mod.quantize_fp8_blocks(a)) for a in (x, k))
    exact = np.einsum("nd,md->nm", x[0, :, 0].astype(np.float64), k[0, :, 0].astype(np.float64))
    err_rot = np.abs(np.einsum("nd,md->nm", qd[0, :, 0], kd[0, :, 0]) - exact).mean()
    err_plain = np.abs(np.einsum("nd,md->nm", qp[0, :, 0], kp[0, :, 0]) - exact).mean()
    assert err_rot < err_plain


def test_rotated_code_checker_accepts_float32_rounding_and_rejects_real_errors(oracle_mod):
    """check_rotated_codes (used by the GPU test of the rotated quantiser)
    accepts the codes of a float32 butterfly evaluation and rejects a code
    moved by one step where the value is far from a rounding boundary, and a
    scale that is off by more than the rounding allows."""
    from parity import check_rotated_codes
    rng = np.random.default_rng(9)
    d = 128
    x = (rng.standard_normal((1, 300, 2, d)) * 3).astype(np.float32)
    x[0, :, 0, 5] *= 40
    x = torch.from_numpy(x).to(torch.bfloat16).float().numpy()   # bf16 inputs, as the kernel takes
    s = rng.choice([-1.0, 1.0], size=d).astype(np.float32)
    codes, scales = oracle_mod.quantize_fp8_blocks(_fwht_float32(x, s))
    scales = (scales * np.float32(1.0 / np.sqrt(128.0))).astype(np.float32)
    check_rotated_codes(codes, scales, x, s, oracle_mod)
    bad = codes.copy()
    y = oracle_mod.hadamard_rotate(x, s)
    amax = np.abs(y[0, :128, 1]).max()
    z = np.abs(y[0, :128, 1]) * 448.0 / amax
    # an element of a middle binade far from any midpoint: move its code by one
    frac = (z / 2.0 ** np.floor(np.log2(np.maximum(z, 1e-30)))) * 8 % 1
    i, j = np.argwhere((z > 4) & (z < 200) & (np.abs(frac - 0.5) > 0.4))[0]
    bad[0, i, 1, j] = bad[0, i, 1, j] + 1 if bad[0, i, 1, j] & 7 < 6 else bad[0, i, 1, j] - 1
    with pytest.raises(AssertionError, match="away from a rounding boundary"):
        check_rotated_codes(bad, scales, x, s, oracle_mod)
    off = scales.copy()
    off[0, 1, 0] *= np.float32(1 + 2.0 ** -10)
    with pytest.raises(AssertionError, match="scale"):
        check_rotated_codes(codes, off, x, s, oracle_mod)


# ---------------------------------------------------------------- precision readings
def test_row_sum_must_not_accumulate_in_fp16():
    """Lecture 11, section 3.4 and common pitfall 4: the running sum l is
    kept in fp32 (the kernels) or double (the oracle) because a low-precision
    accumulator stagnates once the partial sum is large: later small terms
    are rounded away.  A 4096-key row accumulated in fp16 is off by ~1e-1
    relative; in fp32 by ~1e-6."""
    rng = np.random.default_rng(11)
    s = rng.standard_normal(4096)
    p = np.exp(s - s.max())
    exact = math.fsum(p)
    l16 = np.float16(0)
    for x in p.astype(np.float16):
        l16 = np.float16(l16 + x)
    l32 = np.float32(0)
    for x in p.astype(np.float32):
        l32 = np.float32(l32 + x)
    assert abs(float(l16) - exact) / exact > 0.05          # stagnated: order 1e-1
    assert abs(float(l32) - exact) / exact < 1e-5


def test_fp16_exponential_overflows_near_11_09():
    """Lecture 11, section 3.4: subtracting the row maximum is not only for
    fp32's sake: fp16's e^x overflows at x ~ 11.09 = ln(65504), the largest
    fp16 value, so unshifted scores of that size would already be inf."""
    assert math.log(65504.0) == pytest.approx(11.09, abs=0.005)
    with np.errstate(over="ignore"):
        assert np.isfinite(np.float16(np.exp(11.08)))
        assert np.isinf(np.float16(np.exp(11.10)))


def test_fp8_pv_checker_accepts_e4m3_p_and_rejects_real_errors(oracle_mod):
    """check_fp8_pv (used by the GPU tests of the e4m3 P V forward) accepts
    an evaluation that rounds 256 P to e4m3 (nearest even) before P V, with
    l over the unrounded P, as the bound it states allows; and rejects
    results with a plausible mistake: a V row off by one key, a key left
    out, or the 2^8 factor of P not taken back out."""
    from parity import check_fp8_pv
    rng = np.random.default_rng(11)
    B, Hq, Hkv, Nq, Nk, d = 1, 2, 1, 40, 70, 16
    scale = 0.5
    q = torch.from_numpy(rng.standard_normal((B, Nq, Hq, d)).astype(np.float32)).to(torch.bfloat16)
    k = torch.from_numpy(rng.standard_normal((B, Nk, Hkv, d)).astype(np.float32)).to(torch.bfloat16)
    v = torch.from_numpy((rng.standard_normal((B, Nk, Hkv, d)) * 3).astype(np.float32)).to(torch.bfloat16)
    ro, rl = oracle_mod.attn_fwd(q, k, v, True, scale)
    rabs, _ = oracle_mod.attn_fwd(q, k, v.abs(), True, scale)
    vabs_sum = np.abs(v.double().numpy()).sum(axis=1)[:, None, :, :].repeat(Hq, axis=2)

    def emulate(v_shift=0, drop=None, undo=256.0):
        qd, kd, vd = q.double().numpy(), k.double().numpy(), v.double().numpy()
        o = np.zeros((B, Nq, Hq, d))
        for h in range(Hq):
            for i in range(Nq):
                last = i + (Nk - Nq)
                s = scale * kd[0, :last + 1, 0] @ qd[0, i, h]
                pr = np.exp(s - s.max())
                p8 = torch.from_numpy(256.0 * pr).to(torch.float8_e4m3fn).double().numpy()
                if drop is not None and drop <= last:
                    p8[drop] = 0.0
                rows = np.clip(np.arange(last + 1) + v_shift, 0, Nk - 1)
                o[0, i, h] = p8 @ vd[0, rows, 0] / (undo * pr.sum())
        return torch.from_numpy(o).to(torch.bfloat16), torch.from_numpy(rl.astype(np.float32))

    o, lse = emulate()
    err = check_fp8_pv(o, lse, ro, rl, rabs, vabs_sum, "emulated e4m3 P")
    assert err > 1e-3                          # the rounding of P is visible
    for bad in (dict(v_shift=1), dict(drop=35), dict(undo=1.0)):
        o_bad, _ = emulate(**bad)
        with pytest.raises(AssertionError):
            check_fp8_pv(o_bad, lse, ro, rl, rabs, vabs_sum, "planted %s" % bad)
