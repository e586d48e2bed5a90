"""The C ABI without a GPU: the library loads, exports every symbol the
header declares, and rejects bad arguments before launching anything."""
import ctypes
import os
import re

import pytest

import exact_attention_62_gb300 as pkg

INCLUDE = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include")
HEADER = os.path.join(INCLUDE, "attn.h")
TEST_HEADER = os.path.join(INCLUDE, "attn_test.h")

OK, INVALID, UNSUPPORTED, CUDA, TIMEOUT = range(5)
BF16, F32 = 0, 1
# aligned, never dereferenced: every call below is rejected (or is a no-op)
# before the library touches a pointer or the CUDA runtime
FAKE = ctypes.c_void_p(0x7f0000000000)
FAKE_LSE = ctypes.c_void_p(0x7f0000100000)


def declared_functions(header=HEADER):
    text = open(header).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(attn_[a-z0-9_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def L(attn):
    return attn.lib()


def test_header_declares_the_documented_set():
    assert declared_functions() == sorted(pkg.EXPORTED_SYMBOLS)


def test_test_header_declares_the_test_entry_points():
    assert declared_functions(TEST_HEADER) == sorted(pkg.TEST_SYMBOLS)


def test_every_declared_symbol_is_exported(L):
    for name in declared_functions() + declared_functions(TEST_HEADER):
        assert hasattr(L, name), name


def test_status_strings_and_version(L):
    for code in range(6):
        assert pkg.attn_status_string(code) and pkg.attn_status_string(code) != "unknown status"
    assert "bounds" in pkg.attn_status_string(pkg.ATTN_ERR_BOUNDS)
    assert pkg.attn_status_string(99) == "unknown status"
    assert "sm_103a" in pkg.attn_version()


def fwd(L, B=1, Hq=2, Hkv=1, Nq=8, Nk=8, d=64, causal=0, scale=0.125, dtype=BF16,
        q=FAKE, k=FAKE, v=FAKE, o=FAKE, lse=FAKE_LSE):
    return L.attn_fwd(q, k, v, o, lse, B, Hq, Hkv, Nq, Nk, d, causal, scale, dtype, None)


def test_fwd_rejects_bad_arguments(L):
    assert fwd(L, d=96) == UNSUPPORTED
    assert fwd(L, d=256) == UNSUPPORTED
    assert fwd(L, Hq=3, Hkv=2) == INVALID
    assert fwd(L, Hkv=0) == INVALID
    for bad in ({"B": -1}, {"Hq": -2}, {"Nq": -1}, {"Nk": -5}, {"d": 0}):
        assert fwd(L, **bad) == INVALID, bad
    for s in (0.0, -1.0, float("nan"), float("inf")):
        assert fwd(L, scale=s) == INVALID, s
    assert fwd(L, causal=2) == INVALID
    assert fwd(L, dtype=7) == INVALID
    assert fwd(L, q=None) == INVALID
    assert fwd(L, k=None) == INVALID
    assert fwd(L, lse=None) == INVALID
    assert fwd(L, o=ctypes.c_void_p(0x7f0000000008)) == INVALID  # not 16-byte aligned
    assert fwd(L, lse=ctypes.c_void_p(0x7f0000000002)) == INVALID


def test_fwd_empty_is_a_noop(L):
    assert fwd(L, B=0, q=None, k=None, v=None, o=None, lse=None) == OK
    assert fwd(L, Nq=0, q=None, k=None, v=None, o=None, lse=None) == OK
    assert fwd(L, Hq=0) == OK


def dec(L, B=1, Hq=8, Hkv=2, Nk=100, d=128, scale=0.1, S=0, ws=None, wbytes=0, dtype=BF16):
    return L.attn_decode_splitkv(FAKE, FAKE, FAKE, FAKE, FAKE_LSE, B, Hq, Hkv, Nk, d, scale, S,
                                 ws, wbytes, dtype, None)


def test_decode_rejects_bad_arguments(L):
    assert dec(L, dtype=F32) == UNSUPPORTED
    assert dec(L, d=80) == UNSUPPORTED
    assert dec(L, Hq=6, Hkv=4) == INVALID
    assert dec(L, S=-1) == INVALID
    assert dec(L, S=101) == INVALID            # more segments than keys
    assert dec(L, S=4, ws=None) == INVALID       # several segments need a workspace
    need = pkg.attn_decode_workspace_bytes(1, 8, 2, 100, 128, 4)
    assert dec(L, S=4, ws=FAKE, wbytes=need - 1) == INVALID
    assert dec(L, scale=float("nan")) == INVALID
    assert dec(L, B=0) == OK


def test_decode_workspace_layout():
    # o_parts [S, R, d] fp32 rounded up to 256 bytes, then lse_parts [S, R]
    for B, Hq, d, S in ((1, 32, 128, 19), (16, 32, 128, 3), (3, 5, 64, 7)):
        R = B * Hq
        o_bytes = S * R * d * 4
        want = (o_bytes + 255) // 256 * 256 + S * R * 4
        assert pkg.attn_decode_workspace_bytes(B, Hq, 1, 1000, d, S) == want
    assert pkg.attn_decode_workspace_bytes(1, 8, 2, 100, 128, 1) == 0  # one segment: none
    assert pkg.attn_decode_workspace_bytes(1, 8, 3, 100, 128, 2) == 0  # invalid sizes


def test_merge_rejects_bad_arguments(L):
    m = lambda P=2, rows=4, d=64, dt=F32: L.attn_merge_lse(FAKE, FAKE_LSE, P, rows, d, FAKE,
                                                          FAKE_LSE, dt, None)
    assert m(P=0) == INVALID
    assert m(d=6) == INVALID
    assert m(d=516) == INVALID
    assert m(rows=-1) == INVALID
    assert m(dt=5) == INVALID
    assert m(rows=0) == OK


def test_tile_counter_needs_a_pointer(L):
    assert L.attn_read_tile_counter(None, 0) == INVALID


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    """No silent fallback: a missing libattn.so is an error."""
    monkeypatch.setattr(pkg, "_lib", None)
    monkeypatch.setattr(pkg, "_LIB_PATH", str(tmp_path / "libattn.so"))
    with pytest.raises(RuntimeError, match="not built"):
        pkg.lib()


def paged(L, B=2, Hq=8, Hkv=2, d=128, num_pages=10, ps=64, max_pages=4, max_len=200, S=1,
          ws=None, wbytes=0, dtype=BF16):
    return L.attn_decode_paged(FAKE, FAKE, FAKE, FAKE_LSE, FAKE_LSE, FAKE, FAKE_LSE, B, Hq, Hkv, d,
                               num_pages, ps, max_pages, max_len, 0.1, S, ws, wbytes, dtype, None)


def test_paged_decode_rejects_bad_arguments(L):
    assert paged(L, ps=48, max_pages=10) == UNSUPPORTED   # page sizes: 16, 32 or multiples of 64
    assert paged(L, ps=8, max_pages=40) == UNSUPPORTED
    assert paged(L, ps=0) == INVALID
    assert paged(L, max_pages=3, max_len=200) == INVALID   # 3 pages of 64 < 200 keys
    assert paged(L, dtype=F32) == UNSUPPORTED
    assert paged(L, d=96) == UNSUPPORTED
    assert paged(L, Hq=6, Hkv=4) == INVALID
    assert paged(L, S=201) == INVALID             # more segments than keys
    assert paged(L, S=4) == INVALID               # several segments need a workspace
    assert paged(L, num_pages=0) == INVALID
    # one segment of 100000 keys in pages of 16 would need > 4096 table entries
    assert paged(L, ps=16, max_pages=7000, max_len=100000, S=1) == UNSUPPORTED
    assert paged(L, B=0) == OK


def test_paged_decode_declares_its_auto_split_rule():
    # pages a segment touches must fit the 4096-entry staging area; the rule is host arithmetic
    assert pkg.attn_decode_workspace_bytes(2, 8, 2, 200, 128, 3) == \
        (3 * 16 * 128 * 4 + 255) // 256 * 256 + 3 * 16 * 4


def bwd(L, B=1, Hq=2, Hkv=1, Nq=8, Nk=8, d=64, causal=0, scale=0.125, ws=FAKE, wbytes=1 << 20,
        dtype=BF16):
    return L.attn_bwd(FAKE, FAKE, FAKE, FAKE, FAKE_LSE, FAKE, FAKE, FAKE, FAKE, B, Hq, Hkv, Nq, Nk,
                      d, causal, scale, ws, wbytes, dtype, None)


def test_bwd_rejects_bad_arguments(L):
    assert bwd(L, d=96) == UNSUPPORTED
    assert bwd(L, dtype=F32) == UNSUPPORTED
    assert bwd(L, Hq=3, Hkv=2) == INVALID
    assert bwd(L, causal=2) == INVALID
    assert bwd(L, scale=float("nan")) == INVALID
    assert bwd(L, ws=None) == INVALID
    assert bwd(L, wbytes=16) == INVALID          # D needs B*Hq*Nq floats
    assert bwd(L, B=0) == OK
    assert pkg.attn_bwd_workspace_bytes(2, 3, 100) == (2 * 3 * 100 * 4 + 255) // 256 * 256


def test_fwd_host_rejects_bad_arguments(L):
    H = ctypes.c_void_p(0x10000)   # host pointers are never touched either
    def host(B=2, d=64, chunks=0, q_h=H, q_d=FAKE, scale=0.125, causal=0):
        return L.attn_fwd_host(q_h, H, H, H, H, q_d, FAKE, FAKE, FAKE, FAKE_LSE, B, 2, 1, 8, 8, d, causal,
                               scale, BF16, chunks, None, None, None)
    assert host(d=96) == UNSUPPORTED
    assert host(q_h=None) == INVALID
    assert host(q_d=None) == INVALID
    assert host(q_d=ctypes.c_void_p(0x7f0000000008)) == INVALID   # device buffer not 16-byte aligned
    assert host(scale=float("inf")) == INVALID
    assert host(causal=2) == INVALID
    assert host(chunks=-1) == INVALID
    assert host(B=20, chunks=17) == UNSUPPORTED   # at most 16 chunks
    assert host(B=0) == OK


def test_fp8_entry_points_reject_bad_arguments(L):
    assert L.attn_quantize_fp8(FAKE, FAKE, FAKE_LSE, 1, 8, 2, 7, None) == INVALID   # odd d
    assert L.attn_quantize_fp8(None, FAKE, FAKE_LSE, 1, 8, 2, 64, None) == INVALID
    assert L.attn_quantize_fp8(FAKE, FAKE, FAKE_LSE, 0, 8, 2, 64, None) == OK
    rot = lambda x=FAKE, signs=FAKE_LSE, B=1, d=128: L.attn_quantize_fp8_rotated(
        x, signs, FAKE, FAKE_LSE, B, 8, 2, d, None)
    assert rot(d=96) == UNSUPPORTED          # the Hadamard transform needs d = 64 or 128
    assert rot(d=0) == INVALID
    assert rot(signs=None) == INVALID
    assert rot(x=None) == INVALID
    assert rot(B=0) == OK
    f8 = lambda d=128, causal=0, Hq=2, Hkv=1, B=1: L.attn_fwd_fp8(
        FAKE, FAKE, FAKE, FAKE_LSE, FAKE_LSE, FAKE, FAKE_LSE, B, Hq, Hkv, 8, 8, d, causal, 0.1, None)
    assert f8(d=64) == UNSUPPORTED
    assert f8(causal=3) == INVALID
    assert f8(Hq=3, Hkv=2) == INVALID
    assert f8(B=0) == OK
    qv = lambda v=FAKE, vt=FAKE, sc=FAKE_LSE, B=1, d=128: L.attn_quantize_fp8_v(v, vt, sc, B, 8, 2, d, None)
    assert qv(d=96) == UNSUPPORTED           # transposed tiles of 64 or 128 rows
    assert qv(d=0) == INVALID
    assert qv(v=None) == INVALID
    assert qv(sc=None) == INVALID
    assert qv(B=0) == OK
    pv = lambda d=128, causal=0, Hq=2, Hkv=1, B=1, vt=FAKE, vs=FAKE_LSE, Nq=8: L.attn_fwd_fp8_pv(
        FAKE, FAKE, vt, FAKE_LSE, FAKE_LSE, vs, FAKE, FAKE_LSE, B, Hq, Hkv, Nq, 8, d, causal, 0.1, None)
    assert pv(d=64) == UNSUPPORTED
    assert pv(causal=2) == INVALID
    assert pv(Hq=3, Hkv=2) == INVALID
    assert pv(vt=None) == INVALID
    assert pv(vs=None) == INVALID
    assert pv(B=0) == OK
    assert pv(Nq=0) == OK


def test_test_entry_points_reject_bad_arguments(L):
    """The test-only entry points check their options and then their
    arguments as the production calls do, before any launch."""
    opt = pkg.AttnTestOptions()
    f = lambda o=ctypes.byref(opt), d=64, Hq=2, Hkv=1, scale=0.125: L.attn_fwd_test(
        FAKE, FAKE, FAKE, FAKE, FAKE_LSE, 1, Hq, Hkv, 8, 8, d, 0, scale, o, None)
    assert f(o=None) == INVALID
    assert f(d=96) == UNSUPPORTED
    assert f(Hq=3, Hkv=2) == INVALID
    assert f(scale=0.0) == INVALID
    for bad in (pkg.AttnTestOptions(rescale_threshold=9.0), pkg.AttnTestOptions(rescale_threshold=-1.0),
                pkg.AttnTestOptions(rescale_threshold=float("nan")),
                pkg.AttnTestOptions(wait_limit_cycles=-5)):
        assert f(o=ctypes.byref(bad)) == INVALID
    dt = lambda o=ctypes.byref(opt), S=4, ws=None: L.attn_decode_test(
        FAKE, FAKE, FAKE, FAKE, FAKE_LSE, 1, 8, 2, 100, 128, 0.1, S, ws, 0, o, None)
    assert dt(o=None) == INVALID
    assert dt(o=ctypes.byref(pkg.AttnTestOptions(wait_limit_cycles=-1))) == INVALID
    assert dt(S=101) == INVALID    # more segments than keys
    assert dt(S=4) == INVALID      # several segments need a workspace


def test_static_decode_reports_invalid_arguments_before_scratch_size(L):
    """attn_decode_splitkv_static runs the argument checks of
    attn_decode_splitkv first: a call that is invalid is reported as invalid
    even when its partials would not fit the built-in scratch area."""
    st = lambda B=64, Hq=32, Hkv=8, Nk=1000, S=2000, scale=0.1, q=FAKE: L.attn_decode_splitkv_static(
        q, FAKE, FAKE, FAKE, FAKE_LSE, B, Hq, Hkv, Nk, 128, scale, S, BF16, None)
    assert st() == INVALID                          # num_splits > Nk
    assert st(S=64, scale=float("nan")) == INVALID  # bad scale
    assert st(S=64, q=None) == INVALID
    assert st(S=64, Hq=30, Hkv=8) == INVALID        # Hq % Hkv != 0
    # a valid call whose partials exceed the scratch area is refused as unsupported
    need = pkg.attn_decode_workspace_bytes(64, 32, 8, 100000, 128, 64)
    assert need > pkg.DECODE_STATIC_SCRATCH_BYTES
    assert st(Nk=100000, S=64) == UNSUPPORTED
