"""CPU float64 oracle for exact attention -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (the CUDA library and
its Python binding) never imports it and shares no code with it.

The arithmetic lives in ``attn_oracle.c`` (plain C, OpenMP over rows, double
precision); this module only builds that file with gcc and marshals numpy
arrays.  Every function is pinned by ``tests/test_oracle.py`` against values
that do not come from the oracle itself.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile ``attn_oracle.c`` into ``liboracle.so`` (gcc, -O2, OpenMP)."""
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = _LIB + ".tmp.%d" % os.getpid()
    # -ffp-contract=off: no fused multiply-add, so every product and sum is
    # rounded exactly as written.
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
           "-ffp-contract=off", "-o", tmp, _SRC, "-lm"]
    subprocess.check_call(cmd)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is not None:
        return _lib
    build()
    lib = ctypes.CDLL(_LIB)
    P = ctypes.c_void_p
    L = ctypes.c_long
    D = ctypes.c_double
    I = ctypes.c_int
    lib.oracle_num_threads.restype = I
    lib.oracle_attn_fwd.argtypes = [P, P, P, L, L, L, L, L, L, I, D, P, P]
    lib.oracle_attn_fwd.restype = I
    lib.oracle_attn_rows.argtypes = [P, P, P, L, L, L, L, L, L, I, D, L, P, P, P]
    lib.oracle_attn_rows.restype = I
    lib.oracle_attn_fwd_tiled.argtypes = [P, P, P, L, L, L, L, L, L, I, D, L, L, P, P, P]
    lib.oracle_attn_fwd_tiled.restype = I
    lib.oracle_online_trace.argtypes = [P, L, L, P, P, P]
    lib.oracle_online_trace.restype = None
    lib.oracle_segment_state.argtypes = [P, P, P, L, L, L, L, L, L, I, D, L, L, L, L, L, P, P, P]
    lib.oracle_segment_state.restype = None
    lib.oracle_state_merge.argtypes = [D, D, P, D, D, P, L, P, P, P]
    lib.oracle_state_merge.restype = None
    lib.oracle_merge_lse.argtypes = [L, L, L, P, P, P, P]
    lib.oracle_merge_lse.restype = None
    lib.oracle_decode_split.argtypes = [P, P, P, L, L, L, L, L, D, L, P, P]
    lib.oracle_decode_split.restype = I
    _lib = lib
    return lib


def _f32(a) -> np.ndarray:
    """Float32 C-contiguous view of a numpy array or CPU torch tensor.

    bf16 and fp32 values are exact in float32, so nothing is rounded here.
    """
    if hasattr(a, "detach"):  # torch tensor
        a = a.detach().to("cpu")
        import torch
        a = a.to(torch.float32).numpy()
    a = np.ascontiguousarray(a, dtype=np.float32)
    return a


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def num_threads() -> int:
    """Threads the oracle's OpenMP loops use."""
    return int(_load().oracle_num_threads())


def _shapes(q, k, Nq_axis=1):
    B, Nq, Hq, d = q.shape
    Bk, Nk, Hkv, dk = k.shape
    assert B == Bk and d == dk, "q/k shapes disagree"
    return B, Hq, Hkv, Nq, Nk, d


def attn_fwd(q, k, v, causal: bool, scale: float):
    """Algorithm 0, every row.  Returns (o [B,Nq,Hq,d], lse [B,Hq,Nq]) float64."""
    lib = _load()
    q, k, v = _f32(q), _f32(k), _f32(v)
    B, Hq, Hkv, Nq, Nk, d = _shapes(q, k)
    o = np.zeros((B, Nq, Hq, d), np.float64)
    lse = np.zeros((B, Hq, Nq), np.float64)
    rc = lib.oracle_attn_fwd(_ptr(q), _ptr(k), _ptr(v), B, Hq, Hkv, Nq, Nk, d,
                             int(causal), float(scale), _ptr(o), _ptr(lse))
    if rc != 0:
        raise ValueError("oracle_attn_fwd rejected the shapes (rc=%d)" % rc)
    return o, lse


def attn_rows(q, k, v, causal: bool, scale: float, rows):
    """Algorithm 0 for selected rows.

    ``rows`` is an int array [n, 3] of (b, hq, i).  Returns (o [n, d],
    lse [n]) float64.
    """
    lib = _load()
    q, k, v = _f32(q), _f32(k), _f32(v)
    B, Hq, Hkv, Nq, Nk, d = _shapes(q, k)
    sel = np.ascontiguousarray(np.asarray(rows, dtype=np.int64).reshape(-1, 3))
    n = sel.shape[0]
    o = np.zeros((n, d), np.float64)
    lse = np.zeros((n,), np.float64)
    rc = lib.oracle_attn_rows(_ptr(q), _ptr(k), _ptr(v), B, Hq, Hkv, Nq, Nk, d,
                              int(causal), float(scale), n,
                              sel.ctypes.data_as(ctypes.c_void_p), _ptr(o), _ptr(lse))
    if rc != 0:
        raise ValueError("oracle_attn_rows rejected its arguments (rc=%d)" % rc)
    return o, lse


def attn_fwd_tiled(q, k, v, causal: bool, scale: float, Br: int, Bc: int):
    """Tiled online-softmax forward.  Returns (o, lse, blocks_computed)."""
    lib = _load()
    q, k, v = _f32(q), _f32(k), _f32(v)
    B, Hq, Hkv, Nq, Nk, d = _shapes(q, k)
    o = np.zeros((B, Nq, Hq, d), np.float64)
    lse = np.zeros((B, Hq, Nq), np.float64)
    nb = ctypes.c_long(0)
    rc = lib.oracle_attn_fwd_tiled(_ptr(q), _ptr(k), _ptr(v), B, Hq, Hkv, Nq, Nk, d,
                                   int(causal), float(scale), int(Br), int(Bc),
                                   _ptr(o), _ptr(lse), ctypes.byref(nb))
    if rc != 0:
        raise ValueError("oracle_attn_fwd_tiled rejected its arguments (rc=%d)" % rc)
    return o, lse, int(nb.value)


def online_trace(x, block: int):
    """Online softmax over a score row in blocks: (m, l, alpha) after each block."""
    lib = _load()
    x = np.ascontiguousarray(np.asarray(x, dtype=np.float64))
    nb = (x.size + block - 1) // block
    m = np.zeros(nb)
    l = np.zeros(nb)
    a = np.zeros(nb)
    lib.oracle_online_trace(_ptr(x), x.size, int(block), _ptr(m), _ptr(l), _ptr(a))
    return m, l, a


def segment_state(q, k, v, causal: bool, scale: float, b: int, hq: int, i: int,
                  j0: int, j1: int):
    """Unnormalised partial state (m, l, acc) of keys [j0, j1) for row (b, hq, i)."""
    lib = _load()
    q, k, v = _f32(q), _f32(k), _f32(v)
    B, Hq, Hkv, Nq, Nk, d = _shapes(q, k)
    m = ctypes.c_double(0)
    l = ctypes.c_double(0)
    acc = np.zeros(d, np.float64)
    lib.oracle_segment_state(_ptr(q), _ptr(k), _ptr(v), B, Hq, Hkv, Nq, Nk, d,
                             int(causal), float(scale), b, hq, i, j0, j1,
                             ctypes.byref(m), ctypes.byref(l), _ptr(acc))
    return m.value, l.value, acc


def state_merge(a, b):
    """Merge two partial states (m, l, acc) of one row."""
    lib = _load()
    m_a, l_a, acc_a = a
    m_b, l_b, acc_b = b
    acc_a = np.ascontiguousarray(acc_a, np.float64)
    acc_b = np.ascontiguousarray(acc_b, np.float64)
    d = acc_a.size
    m = ctypes.c_double(0)
    l = ctypes.c_double(0)
    acc = np.zeros(d, np.float64)
    lib.oracle_state_merge(float(m_a), float(l_a), _ptr(acc_a), float(m_b), float(l_b),
                           _ptr(acc_b), d, ctypes.byref(m), ctypes.byref(l), _ptr(acc))
    return m.value, l.value, acc


def merge_lse(o_parts, lse_parts):
    """LSE-form merge.  o_parts [P, rows, d], lse_parts [P, rows] -> (o, lse)."""
    lib = _load()
    o_parts = np.ascontiguousarray(o_parts, np.float64)
    lse_parts = np.ascontiguousarray(lse_parts, np.float64)
    P, rows, d = o_parts.shape
    assert lse_parts.shape == (P, rows)
    o = np.zeros((rows, d), np.float64)
    lse = np.zeros((rows,), np.float64)
    lib.oracle_merge_lse(P, rows, d, _ptr(o_parts), _ptr(lse_parts), _ptr(o), _ptr(lse))
    return o, lse


def decode_split(q, k, v, scale: float, nsplit: int):
    """Per-segment partials of flash-decoding (Nq = 1).

    Returns (o_parts [nsplit, B*Hq, d], lse_parts [nsplit, B*Hq]) float64.
    """
    lib = _load()
    q, k, v = _f32(q), _f32(k), _f32(v)
    B, Hq, Hkv, Nq, Nk, d = _shapes(q, k)
    assert Nq == 1, "decode takes one query per sequence"
    rows = B * Hq
    o_parts = np.zeros((nsplit, rows, d), np.float64)
    lse_parts = np.zeros((nsplit, rows), np.float64)
    rc = lib.oracle_decode_split(_ptr(q), _ptr(k), _ptr(v), B, Hq, Hkv, Nk, d,
                                 float(scale), int(nsplit), _ptr(o_parts), _ptr(lse_parts))
    if rc != 0:
        raise ValueError("oracle_decode_split rejected its arguments (rc=%d)" % rc)
    return o_parts, lse_parts


def decode_paged(q, k_pages, v_pages, block_table, seq_lens, scale: float):
    """Decode (one query per sequence) over a paged KV cache.

    Paged KV is named in Lecture 11, section 9 (decode kernels on the
    flash-decoding framework of section 6.2 read a paged cache); the pages fix
    no layout, so this follows the plainest one: K/V pages [num_pages,
    page_size, Hkv, d], block_table [B, max_pages] (int), seq_lens [B].  The
    keys of sequence b are positions 0 .. seq_lens[b]-1 of the concatenation
    of its pages block_table[b, 0], block_table[b, 1], ...  The result is
    algorithm 0 (``attn_fwd``, non-causal) over exactly those keys; a sequence
    with no keys has o = 0 and lse = -inf.  Pool slots beyond a sequence's
    length are never read.  Returns (o [B, 1, Hq, d], lse [B, Hq]) float64.
    """
    q = _f32(q)
    kp, vp = _f32(k_pages), _f32(v_pages)
    table = np.asarray(block_table, np.int64)
    lens = np.asarray(seq_lens, np.int64)
    B, _, Hq, d = q.shape
    ps = kp.shape[1]
    o = np.zeros((B, 1, Hq, d), np.float64)
    lse = np.full((B, Hq), -np.inf, np.float64)
    for b in range(B):
        L = int(lens[b])
        if L <= 0:
            continue
        pages = table[b, :(L + ps - 1) // ps]
        kb = kp[pages].reshape(-1, kp.shape[2], d)[:L][None]
        vb = vp[pages].reshape(-1, vp.shape[2], d)[:L][None]
        ob, lb = attn_fwd(q[b:b + 1], kb, vb, False, scale)
        o[b] = ob[0]
        lse[b] = lb[0, :, 0]
    return o, lse


def attn_bwd(q, k, v, do, causal: bool, scale: float):
    """Gradients of algorithm 0 (Lecture 11, section 5.1), float64.

    With S = scale Q K^T (masked entries -inf), P = softmax(S) row-wise and
    O = P V, given dO:  dV = P^T dO;  dP = dO V^T;  D_i = sum_j P_ij dP_ij,
    which equals rowsum(dO_i * O_i) (the identity section 5.1 uses so that
    D needs only a row of O and dO);  dS = P * (dP - D);  dQ = scale dS K;
    dK = scale dS^T Q.  Query head hq uses KV head hq // (Hq / Hkv), so a KV
    head's dK and dV sum over its query heads.  A row with no allowed key has
    P = 0 and contributes nothing.  Inputs [B, N, H, d] (any float type);
    returns (dq, dk, dv) float64 in the shapes of q, k, v.
    """
    q = np.asarray(_f32(q), np.float64)
    k = np.asarray(_f32(k), np.float64)
    v = np.asarray(_f32(v), np.float64)
    do = np.asarray(_f32(do), np.float64)
    B, Nq, Hq, d = q.shape
    _, Nk, Hkv, _ = k.shape
    G = Hq // Hkv
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    i_idx = np.arange(Nq)[:, None]
    j_idx = np.arange(Nk)[None, :]
    allowed = np.ones((Nq, Nk), bool) if not causal else (j_idx <= i_idx + (Nk - Nq))
    for b in range(B):
        for hq in range(Hq):
            g = hq // G
            Q, K, V, dO = q[b, :, hq, :], k[b, :, g, :], v[b, :, g, :], do[b, :, hq, :]
            S = np.where(allowed, scale * (Q @ K.T), -np.inf)
            m = S.max(axis=1)
            has = np.isfinite(m)
            E = np.where(has[:, None], np.exp(S - np.where(has, m, 0.0)[:, None]), 0.0)
            den = E.sum(axis=1)
            P = np.where(has[:, None], E / np.where(has, den, 1.0)[:, None], 0.0)
            O = P @ V
            dv[b, :, g, :] += P.T @ dO
            dP = dO @ V.T
            D = (dO * O).sum(axis=1)
            dS = P * (dP - D[:, None])
            dq[b, :, hq, :] = scale * (dS @ K)
            dk[b, :, g, :] += scale * (dS.T @ Q)
    return dq, dk, dv


# ------------------------------------------------------------------ FP8 (block quantisation)
FP8_MAX = 448.0  # largest finite e4m3 value


def quantize_fp8_blocks(x, block: int = 128):
    """Block quantisation to e4m3 (Lecture 11, section 4.5, FP8 item: block
    quantisation).  x [B, N, H, d] -> (codes uint8 [B, N, H, d], scales
    float32 [B, H, ceil(N / block)]).  Per (b, h, block of `block` rows):
    amax = max |x| (as float32), scale = amax / 448 and inv = 448 / amax in
    float32 (1 and 1 for an all-zero block), code = e4m3(round to nearest
    even, clamped to +-448)(x * inv) with x * inv in float32."""
    import torch
    xt = torch.as_tensor(np.asarray(_f32(x)))
    B, N, H, d = xt.shape
    nb = (N + block - 1) // block
    codes = torch.zeros((B, N, H, d), dtype=torch.uint8)
    scales = torch.ones((B, H, nb), dtype=torch.float32)
    for bi in range(nb):
        r0, r1 = bi * block, min(N, (bi + 1) * block)
        blk = xt[:, r0:r1]                                    # [B, rows, H, d]
        amax = blk.abs().amax(dim=(1, 3))                     # [B, H] float32
        nz = amax > 0
        one = torch.ones_like(amax)
        inv = torch.where(nz, torch.full_like(amax, FP8_MAX) / torch.where(nz, amax, one), one)
        sc = torch.where(nz, amax / FP8_MAX, one)
        y = (blk * inv[:, None, :, None]).clamp(-FP8_MAX, FP8_MAX)
        codes[:, r0:r1] = y.to(torch.float8_e4m3fn).view(torch.uint8)
        scales[:, :, bi] = sc
    return codes.numpy(), scales.numpy()


def sylvester_hadamard(d: int) -> np.ndarray:
    """The d x d Sylvester Hadamard matrix (d a power of two) in float64:
    H_1 = [1], H_2n = [[H_n, H_n], [H_n, -H_n]].  H is symmetric with
    entries +-1 and H H^T = d I."""
    if d < 1 or d & (d - 1):
        raise ValueError("d must be a power of two")
    H = np.ones((1, 1), np.float64)
    while H.shape[0] < d:
        H = np.block([[H, H], [H, -H]])
    return H


def hadamard_rotate(x, signs):
    """x [..., d] times diag(signs) H, in float64: the unnormalised random
    orthogonal transform of incoherent processing (Lecture 11, section 4.5,
    FP8 item; R = diag(signs) H / sqrt(d) is orthogonal).  The plain
    definition: one float64 matrix product with the Sylvester matrix, no
    particular order of evaluation."""
    y = np.asarray(_f32(x), np.float64) * np.asarray(signs, np.float64)
    return y @ sylvester_hadamard(y.shape[-1])


def quantize_fp8_blocks_rotated(x, signs, block: int = 128):
    """Incoherent processing before block quantisation (Lecture 11, section
    4.5, FP8 item).  Reading: the rotated rows y = x diag(signs) H (exact, in
    float64) are rounded once to float32, the quantiser's working type, and
    block-quantised by quantize_fp8_blocks; each scale is then multiplied in
    float32 by c = float32(1 / sqrt(d)), so that codes * scales ~= x R with
    the orthogonal R = diag(signs) H / sqrt(d).  Returns (codes, scales) like
    quantize_fp8_blocks.  An implementation that forms y in float32 differs
    from this by the rounding of its own order of evaluation: see
    rotation_error_bound."""
    y = hadamard_rotate(x, signs)
    codes, scales = quantize_fp8_blocks(y.astype(np.float32), block)
    c = np.float32(1.0 / np.sqrt(np.float64(y.shape[-1])))
    return codes, (np.asarray(scales, np.float32) * c).astype(np.float32)


def rotation_error_bound(x):
    """Bound on |y32 - y| for the rows of any float32 evaluation of the
    rotation by the fast Walsh-Hadamard butterflies (log2 d stages of sums and
    differences of pairs): every stage rounds each intermediate once, with a
    relative error of at most u = 2^-24, and no intermediate exceeds
    sum_j |x_j| in magnitude, so the error of an output is at most
    log2(d) u sum_j |x_j| (first order; doubled here for the higher-order
    terms).  Returns [..., 1] float64."""
    xa = np.abs(np.asarray(_f32(x), np.float64))
    d = xa.shape[-1]
    return 2.0 * np.log2(d) * 2.0 ** -24 * xa.sum(axis=-1, keepdims=True)


def dequantize_fp8_blocks(codes, scales, block: int = 128):
    """codes uint8 [B, N, H, d] (e4m3) and scales [B, H, nblocks] -> float64."""
    import torch
    c = torch.as_tensor(np.asarray(codes, np.uint8)).view(torch.float8_e4m3fn).to(torch.float64)
    s = torch.as_tensor(np.asarray(scales, np.float32)).to(torch.float64)
    B, N, H, d = c.shape
    rows = torch.arange(N) // block
    return (c * s[:, :, rows].permute(0, 2, 1)[..., None]).numpy()


def score_perturbation(q_a, k_a, q_b, k_b, causal: bool, scale: float):
    """Per query row, max over allowed keys of |S_a - S_b| with S = scale q k^T
    (the two inputs e.g. dequantised and exact).  Returns [B, Hq, Nq] float64
    (0 for rows with no allowed key)."""
    qa, ka = np.asarray(q_a, np.float64), np.asarray(k_a, np.float64)
    qb, kb = np.asarray(q_b, np.float64), np.asarray(k_b, np.float64)
    B, Nq, Hq, d = qa.shape
    Nk, Hkv = ka.shape[1], ka.shape[2]
    G = Hq // Hkv
    out = np.zeros((B, Hq, Nq))
    allowed = np.ones((Nq, Nk), bool)
    if causal:
        allowed = np.arange(Nk)[None, :] <= np.arange(Nq)[:, None] + (Nk - Nq)
    for b in range(B):
        for h in range(Hq):
            g = h // G
            dS = scale * (qa[b, :, h] @ ka[b, :, g].T - qb[b, :, h] @ kb[b, :, g].T)
            out[b, h] = np.where(allowed, np.abs(dS), 0.0).max(axis=1)
    return out
