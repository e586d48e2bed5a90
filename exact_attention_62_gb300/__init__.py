"""exact_attention_62_gb300 -- fused exact attention and flash-decoding for GB300.

Thin Python binding over the C ABI of ``libattn.so`` (declared in
``include/attn.h``).  The functions below carry the same names as the C entry
points and only marshal arguments: they take CUDA torch tensors, pass their
device pointers and the current CUDA stream, and raise ``AttnError`` on a
non-OK status.  Every step of the computation runs in the library's CUDA
kernels; there is no CPU or PyTorch fallback, and a missing library is an
error.

PyTorch is used only for device memory and streams.
"""
from __future__ import annotations

import ctypes
import os

__all__ = [
    "AttnError", "ATTN_BF16", "ATTN_F32", "lib", "ensure_built", "library_path", "load_library",
    "use_library",
    "attn_fwd", "attn_fwd_host", "attn_decode_num_splits", "attn_decode_workspace_bytes",
    "attn_decode_splitkv", "attn_merge_lse", "attn_status_string",
    "attn_check_device_status", "attn_read_tile_counter", "attn_version",
    "attn_decode_splitkv_static", "attn_decode_paged", "attn_decode_paged_num_splits",
    "attn_bwd", "attn_bwd_workspace_bytes", "attn_quantize_fp8", "attn_quantize_fp8_rotated",
    "attn_fwd_fp8", "attn_quantize_fp8_v", "attn_fwd_fp8_pv", "DECODE_STATIC_SCRATCH_BYTES",
    "EXPORTED_SYMBOLS", "TEST_SYMBOLS",
    "AttnTestOptions", "attn_fwd_test", "attn_decode_test",
]

ATTN_OK, ATTN_ERR_INVALID, ATTN_ERR_UNSUPPORTED, ATTN_ERR_CUDA, ATTN_ERR_TIMEOUT, ATTN_ERR_BOUNDS = range(6)
ATTN_BF16, ATTN_F32 = 0, 1

# Every symbol include/attn.h declares.
EXPORTED_SYMBOLS = (
    "attn_fwd", "attn_fwd_host", "attn_decode_num_splits", "attn_decode_workspace_bytes",
    "attn_decode_splitkv", "attn_merge_lse", "attn_status_string",
    "attn_check_device_status", "attn_read_tile_counter", "attn_version",
    "attn_decode_splitkv_static", "attn_decode_paged", "attn_decode_paged_num_splits",
    "attn_bwd", "attn_bwd_workspace_bytes", "attn_quantize_fp8", "attn_quantize_fp8_rotated",
    "attn_fwd_fp8", "attn_quantize_fp8_v", "attn_fwd_fp8_pv",
)

# The test-only entry points include/attn_test.h declares.
TEST_SYMBOLS = ("attn_fwd_test", "attn_decode_test", "attn_decode_model_time", "attn_decode_model_best")

# Size of the scratch area built into the library for attn_decode_splitkv_static.
DECODE_STATIC_SCRATCH_BYTES = 8 << 20

_PKG = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_PKG, "libattn.so")
_lib = None


class AttnTestOptions(ctypes.Structure):
    """attn_test_options_t of include/attn_test.h (tests and measurements only)."""
    _fields_ = [("p_in_smem", ctypes.c_int), ("exp2_poly", ctypes.c_int),
                ("rescale_threshold", ctypes.c_float), ("wait_limit_cycles", ctypes.c_longlong),
                ("skip_load", ctypes.c_int), ("o_extent_slack", ctypes.c_longlong)]

    def __init__(self, p_in_smem=0, exp2_poly=0, rescale_threshold=0.0, wait_limit_cycles=0,
                 skip_load=-1, o_extent_slack=0):
        super().__init__(int(p_in_smem), int(exp2_poly), float(rescale_threshold),
                         int(wait_limit_cycles), int(skip_load), int(o_extent_slack))


class AttnError(RuntimeError):
    """A libattn entry point returned a non-OK status."""

    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__("%s failed: %s (status %d)" % (fn, _status_text(status), status))


def library_path() -> str:
    return _LIB_PATH


def ensure_built() -> str:
    """Builds libattn.so if it is missing; returns its path."""
    if not os.path.exists(_LIB_PATH):
        from . import build as _build
        _build.build()
    return _LIB_PATH


def lib() -> ctypes.CDLL:
    """The loaded libattn.so.  Raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(_LIB_PATH):
        raise RuntimeError(
            "libattn.so is not built (%s); run `python -m exact_attention_62_gb300.build` "
            "or __graft_entry__.build()" % _LIB_PATH)
    _lib = load_library(_LIB_PATH)
    return _lib


def use_library(L):
    """Makes every entry point of this module call the library L (a handle
    from load_library) and returns the one in use before.  For tests that run
    the same calls on the bounds-checked debug build, libattn_bounds.so."""
    global _lib
    old = _lib
    _lib = L
    return old


def load_library(path: str) -> ctypes.CDLL:
    """Loads a build of the library (libattn.so or the bounds-checked
    libattn_bounds.so) with the argument types of every entry point."""
    L = ctypes.CDLL(path)
    P, I, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    LL, SZ = ctypes.c_longlong, ctypes.c_size_t
    L.attn_fwd.argtypes = [P, P, P, P, P, I, I, I, I, I, I, I, F, I, P]
    L.attn_fwd.restype = I
    L.attn_fwd_host.argtypes = [P, P, P, P, P, P, P, P, P, P, I, I, I, I, I, I, I, F, I, I, P, P, P]
    L.attn_fwd_host.restype = I
    L.attn_decode_num_splits.argtypes = [I, I, I, I, I]
    L.attn_decode_num_splits.restype = I
    L.attn_decode_workspace_bytes.argtypes = [I, I, I, I, I, I]
    L.attn_decode_workspace_bytes.restype = SZ
    L.attn_decode_splitkv.argtypes = [P, P, P, P, P, I, I, I, I, I, F, I, P, SZ, I, P]
    L.attn_decode_splitkv.restype = I
    L.attn_merge_lse.argtypes = [P, P, I, LL, I, P, P, I, P]
    L.attn_merge_lse.restype = I
    L.attn_status_string.argtypes = [I]
    L.attn_status_string.restype = ctypes.c_char_p
    L.attn_check_device_status.argtypes = []
    L.attn_check_device_status.restype = I
    L.attn_read_tile_counter.argtypes = [ctypes.POINTER(ctypes.c_ulonglong), I]
    L.attn_read_tile_counter.restype = I
    L.attn_version.argtypes = []
    L.attn_version.restype = ctypes.c_char_p
    L.attn_decode_splitkv_static.argtypes = [P, P, P, P, P, I, I, I, I, I, F, I, I, P]
    L.attn_decode_paged.argtypes = [P, P, P, P, P, P, P, I, I, I, I, I, I, I, I, F, I, P, SZ, I, P]
    L.attn_decode_paged.restype = I
    L.attn_decode_paged_num_splits.argtypes = [I, I, I, I, I, I]
    L.attn_decode_paged_num_splits.restype = I
    L.attn_bwd_workspace_bytes.argtypes = [I, I, I]
    L.attn_bwd_workspace_bytes.restype = SZ
    L.attn_bwd.argtypes = [P, P, P, P, P, P, P, P, P, I, I, I, I, I, I, I, F, P, SZ, I, P]
    L.attn_bwd.restype = I
    L.attn_quantize_fp8.argtypes = [P, P, P, I, I, I, I, P]
    L.attn_quantize_fp8.restype = I
    L.attn_quantize_fp8_rotated.argtypes = [P, P, P, P, I, I, I, I, P]
    L.attn_quantize_fp8_rotated.restype = I
    L.attn_fwd_fp8.argtypes = [P, P, P, P, P, P, P, I, I, I, I, I, I, I, F, P]
    L.attn_fwd_fp8.restype = I
    L.attn_quantize_fp8_v.argtypes = [P, P, P, I, I, I, I, P]
    L.attn_quantize_fp8_v.restype = I
    L.attn_fwd_fp8_pv.argtypes = [P, P, P, P, P, P, P, P, I, I, I, I, I, I, I, F, P]
    L.attn_fwd_fp8_pv.restype = I
    L.attn_decode_splitkv_static.restype = I
    OPT = ctypes.POINTER(AttnTestOptions)
    L.attn_fwd_test.argtypes = [P, P, P, P, P, I, I, I, I, I, I, I, F, OPT, P]
    L.attn_fwd_test.restype = I
    L.attn_decode_test.argtypes = [P, P, P, P, P, I, I, I, I, I, F, I, P, SZ, OPT, P]
    L.attn_decode_test.restype = I
    DB = ctypes.c_double
    L.attn_decode_model_time.argtypes = [I, I, I, I, I, DB, DB, DB, DB]
    L.attn_decode_model_time.restype = DB
    L.attn_decode_model_best.argtypes = [I, I, I, I, DB, DB, DB, DB, I]
    L.attn_decode_model_best.restype = I
    return L


def _status_text(status: int) -> str:
    try:
        return lib().attn_status_string(int(status)).decode()
    except Exception:  # library not loadable: still report the code
        return "status %d" % status


def _check(fn: str, status: int):
    if status != ATTN_OK:
        raise AttnError(fn, status)


def _dtype_code(t) -> int:
    import torch
    if t.dtype == torch.bfloat16:
        return ATTN_BF16
    if t.dtype == torch.float32:
        return ATTN_F32
    raise TypeError("unsupported dtype %s (bfloat16 or float32)" % t.dtype)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream, device=None):
    import torch
    s = torch.cuda.current_stream(device) if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _used_on(stream, *tensors):
    """The call's kernels use these device tensors on `stream`.  When that is
    not the current stream (the one torch's caching allocator associates
    with tensors allocated here), record the use, so that memory freed by
    the caller, or by this module on return, is not handed out again before
    the stream's work is done."""
    if stream is None:
        return
    import torch
    if stream == torch.cuda.current_stream(stream.device):
        return
    for t in tensors:
        if t is not None and t.is_cuda:
            t.record_stream(stream)


def _need_cuda_contig(name, t, device=None):
    if not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % name)
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    if device is not None and t.device != device:
        raise ValueError("%s is on %s, the call's tensors on %s" % (name, t.device, device))


def _need_buffer(name, t, shape, dtype, device):
    """A caller-provided output or input buffer: the kernels index it from the
    sizes alone, so its shape, dtype and device must be exactly these."""
    _need_cuda_contig(name, t, device)
    if tuple(t.shape) != tuple(shape):
        raise ValueError("%s must have shape %s, got %s" % (name, tuple(shape), tuple(t.shape)))
    if t.dtype != dtype:
        raise ValueError("%s must be %s, got %s" % (name, dtype, t.dtype))


def _need_workspace(t, device):
    import torch
    _need_cuda_contig("workspace", t, device)
    if t.dtype != torch.uint8:
        raise ValueError("workspace must be a uint8 tensor")


def attn_fwd(q, k, v, causal: bool = False, scale: float | None = None, o=None, lse=None,
             stream=None):
    """O = softmax(scale q k^T) v per head, with LSE = log-sum-exp of the scores.

    q [B, Nq, Hq, d], k/v [B, Nk, Hkv, d]; bf16 (tensor cores) or fp32.
    Returns (o [B, Nq, Hq, d], lse [B, Hq, Nq] float32).
    """
    import torch
    B, Nq, Hq, d = q.shape
    Bk, Nk, Hkv, dk = k.shape
    if Bk != B or dk != d or tuple(v.shape) != tuple(k.shape):
        raise ValueError("shape mismatch: q %s k %s v %s" % (tuple(q.shape), tuple(k.shape), tuple(v.shape)))
    if not (q.dtype == k.dtype == v.dtype):
        raise ValueError("q, k, v must share a dtype")
    dev = q.device
    for n, t in (("q", q), ("k", k), ("v", v)):
        _need_cuda_contig(n, t, dev)
    if scale is None:
        scale = d ** -0.5
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, Hq, Nq), dtype=torch.float32, device=dev)
    _need_buffer("o", o, q.shape, q.dtype, dev)
    _need_buffer("lse", lse, (B, Hq, Nq), torch.float32, dev)
    with torch.cuda.device(dev):
        st = lib().attn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, Hq, Hkv, Nq, Nk, d,
                            int(bool(causal)), float(scale), _dtype_code(q), _stream(stream, dev))
    _check("attn_fwd", st)
    _used_on(stream, q, k, v, o, lse)
    return o, lse


def attn_fwd_host(q, k, v, causal: bool = False, scale: float | None = None, o=None, lse=None,
                  device_buffers=None, chunks: int = 0, stream=None, h2d_stream=None, d2h_stream=None):
    """attn_fwd on CPU tensors (page-locked for asynchronous copies): the batch
    is copied in, computed and copied back in chunks (the chunks' forwards on
    `stream` and a second compute stream by turns) so the transfers overlap
    the computation.  Returns (o, lse) CPU tensors (pinned
    when allocated here); they hold the results once `stream` (default: the
    current stream) has completed.  device_buffers = (q_d, k_d, v_d, o_d,
    lse_d) reuses device memory across calls; h2d_stream / d2h_stream default
    to two streams created here (pass the same stream as `stream` for no
    overlap)."""
    import torch
    B, Nq, Hq, d = q.shape
    Bk, Nk, Hkv, dk = k.shape
    if Bk != B or dk != d or tuple(v.shape) != tuple(k.shape):
        raise ValueError("shape mismatch: q %s k %s v %s" % (tuple(q.shape), tuple(k.shape), tuple(v.shape)))
    if not (q.dtype == k.dtype == v.dtype):
        raise ValueError("q, k, v must share a dtype")
    for n, t in (("q", q), ("k", k), ("v", v)):
        if t.is_cuda or not t.is_contiguous():
            raise ValueError("%s must be a contiguous CPU tensor" % n)
    dev = torch.device("cuda", torch.cuda.current_device())
    if scale is None:
        scale = d ** -0.5
    if o is None:
        o = torch.empty(q.shape, dtype=q.dtype, pin_memory=True)
    if lse is None:
        lse = torch.empty((B, Hq, Nq), dtype=torch.float32, pin_memory=True)
    for n, t, shape, dt in (("o", o, q.shape, q.dtype), ("lse", lse, (B, Hq, Nq), torch.float32)):
        if t.is_cuda or not t.is_contiguous() or tuple(t.shape) != tuple(shape) or t.dtype != dt:
            raise ValueError("%s must be a contiguous CPU %s tensor of shape %s" % (n, dt, tuple(shape)))
    if device_buffers is None:
        device_buffers = (torch.empty(q.shape, dtype=q.dtype, device=dev),
                          torch.empty(k.shape, dtype=k.dtype, device=dev),
                          torch.empty(v.shape, dtype=v.dtype, device=dev),
                          torch.empty(q.shape, dtype=q.dtype, device=dev),
                          torch.empty((B, Hq, Nq), dtype=torch.float32, device=dev))
    q_d, k_d, v_d, o_d, lse_d = device_buffers
    for n, t, ref in (("q_d", q_d, q), ("k_d", k_d, k), ("v_d", v_d, v), ("o_d", o_d, q)):
        _need_buffer(n, t, ref.shape, ref.dtype, dev)
    _need_buffer("lse_d", lse_d, (B, Hq, Nq), torch.float32, dev)
    if h2d_stream is None:
        h2d_stream = torch.cuda.Stream(dev)
    if d2h_stream is None:
        d2h_stream = torch.cuda.Stream(dev)
    with torch.cuda.device(dev):
        st = lib().attn_fwd_host(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(q_d), _ptr(k_d),
                                 _ptr(v_d), _ptr(o_d), _ptr(lse_d), B, Hq, Hkv, Nq, Nk, d,
                                 int(bool(causal)), float(scale), _dtype_code(q), int(chunks),
                                 _stream(stream, dev), _stream(h2d_stream, dev), _stream(d2h_stream, dev))
    _check("attn_fwd_host", st)
    _used_on(stream, *device_buffers)
    return o, lse


def attn_decode_num_splits(B: int, Hq: int, Hkv: int, Nk: int, d: int) -> int:
    return int(lib().attn_decode_num_splits(B, Hq, Hkv, Nk, d))


def attn_decode_workspace_bytes(B: int, Hq: int, Hkv: int, Nk: int, d: int,
                                num_splits: int = 0) -> int:
    return int(lib().attn_decode_workspace_bytes(B, Hq, Hkv, Nk, d, num_splits))


def attn_decode_splitkv(q, k_cache, v_cache, scale: float | None = None, num_splits: int = 0,
                        workspace=None, o=None, lse=None, stream=None):
    """Flash-decoding: q [B, 1, Hq, d], caches [B, Nk, Hkv, d] (bf16).

    Returns (o [B, 1, Hq, d], lse [B, Hq]).  ``workspace`` is a CUDA uint8
    tensor of at least attn_decode_workspace_bytes(...) bytes; it is
    allocated here when not given.
    """
    import torch
    B, one, Hq, d = q.shape
    if one != 1:
        raise ValueError("decode takes one query per sequence (q.shape[1] == 1)")
    Bk, Nk, Hkv, dk = k_cache.shape
    if Bk != B or dk != d or tuple(v_cache.shape) != tuple(k_cache.shape):
        raise ValueError("shape mismatch")
    if not (q.dtype == k_cache.dtype == v_cache.dtype):
        raise ValueError("q and the caches must share a dtype")
    dev = q.device
    for n, t in (("q", q), ("k_cache", k_cache), ("v_cache", v_cache)):
        _need_cuda_contig(n, t, dev)
    if scale is None:
        scale = d ** -0.5
    if num_splits == 0 and Nk > 0 and B > 0 and Hq > 0:
        with torch.cuda.device(dev):
            num_splits = attn_decode_num_splits(B, Hq, Hkv, Nk, d)
    wbytes = attn_decode_workspace_bytes(B, Hq, Hkv, Nk, d, num_splits) if Nk > 0 and B > 0 and Hq > 0 else 0
    if workspace is None and wbytes > 0:
        workspace = torch.empty(wbytes, dtype=torch.uint8, device=dev)
    if workspace is not None:
        _need_workspace(workspace, dev)
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, Hq), dtype=torch.float32, device=dev)
    _need_buffer("o", o, q.shape, q.dtype, dev)
    _need_buffer("lse", lse, (B, Hq), torch.float32, dev)
    wsize = 0 if workspace is None else workspace.numel() * workspace.element_size()
    with torch.cuda.device(dev):
        st = lib().attn_decode_splitkv(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(o), _ptr(lse),
                                       B, Hq, Hkv, Nk, d, float(scale), int(num_splits),
                                       _ptr(workspace), wsize, _dtype_code(q), _stream(stream, dev))
    _check("attn_decode_splitkv", st)
    _used_on(stream, q, k_cache, v_cache, workspace, o, lse)
    return o, lse


def attn_decode_splitkv_static(q, k_cache, v_cache, scale: float | None = None,
                               num_splits: int = 0, o=None, lse=None, stream=None):
    """Flash-decoding for callers that cannot allocate device memory.

    Same arguments and results as attn_decode_splitkv without the workspace:
    the partials go to a fixed scratch area inside the library
    (DECODE_STATIC_SCRATCH_BYTES, shared by every call).  Calls that overlap
    on the GPU race on that area.  The output tensors are allocated here only
    when not given; pass o and lse to allocate nothing at all.
    """
    import torch
    B, one, Hq, d = q.shape
    if one != 1:
        raise ValueError("decode takes one query per sequence (q.shape[1] == 1)")
    Bk, Nk, Hkv, dk = k_cache.shape
    if Bk != B or dk != d or tuple(v_cache.shape) != tuple(k_cache.shape):
        raise ValueError("shape mismatch")
    if not (q.dtype == k_cache.dtype == v_cache.dtype):
        raise ValueError("q and the caches must share a dtype")
    dev = q.device
    for n, t in (("q", q), ("k_cache", k_cache), ("v_cache", v_cache)):
        _need_cuda_contig(n, t, dev)
    if scale is None:
        scale = d ** -0.5
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, Hq), dtype=torch.float32, device=dev)
    _need_buffer("o", o, q.shape, q.dtype, dev)
    _need_buffer("lse", lse, (B, Hq), torch.float32, dev)
    with torch.cuda.device(dev):
        st = lib().attn_decode_splitkv_static(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(o),
                                              _ptr(lse), B, Hq, Hkv, Nk, d, float(scale),
                                              int(num_splits), _dtype_code(q), _stream(stream, dev))
    _check("attn_decode_splitkv_static", st)
    _used_on(stream, q, k_cache, v_cache, o, lse)
    return o, lse


def attn_merge_lse(o_parts, lse_parts, out_dtype=None, o=None, lse=None, stream=None):
    """Merges partials o_parts [P, rows, d] / lse_parts [P, rows] (float32)."""
    import torch
    P, rows, d = o_parts.shape
    if tuple(lse_parts.shape) != (P, rows):
        raise ValueError("lse_parts must be [P, rows]")
    if o_parts.dtype != torch.float32 or lse_parts.dtype != torch.float32:
        raise ValueError("o_parts and lse_parts must be float32")
    dev = o_parts.device
    for n, t in (("o_parts", o_parts), ("lse_parts", lse_parts)):
        _need_cuda_contig(n, t, dev)
    if out_dtype is None:
        out_dtype = o.dtype if o is not None else torch.float32
    if o is None:
        o = torch.empty((rows, d), dtype=out_dtype, device=dev)
    if lse is None:
        lse = torch.empty((rows,), dtype=torch.float32, device=dev)
    _need_buffer("o", o, (rows, d), out_dtype, dev)
    _need_buffer("lse", lse, (rows,), torch.float32, dev)
    with torch.cuda.device(dev):
        st = lib().attn_merge_lse(_ptr(o_parts), _ptr(lse_parts), P, rows, d, _ptr(o), _ptr(lse),
                                  _dtype_code(o), _stream(stream, dev))
    _check("attn_merge_lse", st)
    _used_on(stream, o_parts, lse_parts, o, lse)
    return o, lse


def attn_status_string(status: int) -> str:
    return lib().attn_status_string(int(status)).decode()


def attn_check_device_status() -> int:
    """Reads and clears the kernels' device status words (synchronises)."""
    return int(lib().attn_check_device_status())


def attn_read_tile_counter(reset: bool = False) -> int:
    """(query tile, key tile) pairs the bf16 forward computed since the last reset."""
    c = ctypes.c_ulonglong(0)
    _check("attn_read_tile_counter", lib().attn_read_tile_counter(ctypes.byref(c), int(bool(reset))))
    return int(c.value)


def attn_version() -> str:
    return lib().attn_version().decode()


def attn_decode_paged_num_splits(B: int, Hq: int, Hkv: int, d: int, page_size: int,
                                 max_seq_len: int) -> int:
    return int(lib().attn_decode_paged_num_splits(B, Hq, Hkv, d, page_size, max_seq_len))


def attn_decode_paged(q, k_pages, v_pages, block_table, seq_lens, max_seq_len: int,
                      scale: float | None = None, num_splits: int = 0, workspace=None, o=None,
                      lse=None, stream=None):
    """Flash-decoding over a paged KV cache.

    q [B, 1, Hq, d]; k_pages, v_pages [num_pages, page_size, Hkv, d] (bf16);
    block_table [B, max_pages] and seq_lens [B] int32 on the device;
    max_seq_len >= every seq_lens[b].  Returns (o [B, 1, Hq, d], lse [B, Hq]).
    """
    import torch
    B, one, Hq, d = q.shape
    if one != 1:
        raise ValueError("decode takes one query per sequence (q.shape[1] == 1)")
    num_pages, page_size, Hkv, dk = k_pages.shape
    if dk != d or tuple(v_pages.shape) != tuple(k_pages.shape):
        raise ValueError("shape mismatch")
    if block_table.dim() != 2 or block_table.shape[0] != B or tuple(seq_lens.shape) != (B,):
        raise ValueError("block_table must be [B, max_pages] and seq_lens [B]")
    if block_table.dtype != torch.int32 or seq_lens.dtype != torch.int32:
        raise ValueError("block_table and seq_lens must be int32")
    if not (q.dtype == k_pages.dtype == v_pages.dtype):
        raise ValueError("q and the page pools must share a dtype")
    dev = q.device
    for n, t in (("q", q), ("k_pages", k_pages), ("v_pages", v_pages),
                 ("block_table", block_table), ("seq_lens", seq_lens)):
        _need_cuda_contig(n, t, dev)
    if scale is None:
        scale = d ** -0.5
    max_pages = block_table.shape[1]
    if num_splits == 0 and max_seq_len > 0 and B > 0 and Hq > 0:
        with torch.cuda.device(dev):
            num_splits = attn_decode_paged_num_splits(B, Hq, Hkv, d, page_size, max_seq_len)
    wbytes = (attn_decode_workspace_bytes(B, Hq, Hkv, max_seq_len, d, num_splits)
              if max_seq_len > 0 and B > 0 and Hq > 0 and num_splits > 0 else 0)
    if workspace is None and wbytes > 0:
        workspace = torch.empty(wbytes, dtype=torch.uint8, device=dev)
    if workspace is not None:
        _need_workspace(workspace, dev)
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, Hq), dtype=torch.float32, device=dev)
    _need_buffer("o", o, q.shape, q.dtype, dev)
    _need_buffer("lse", lse, (B, Hq), torch.float32, dev)
    wsize = 0 if workspace is None else workspace.numel() * workspace.element_size()
    with torch.cuda.device(dev):
        st = lib().attn_decode_paged(_ptr(q), _ptr(k_pages), _ptr(v_pages), _ptr(block_table),
                                     _ptr(seq_lens), _ptr(o), _ptr(lse), B, Hq, Hkv, d, num_pages,
                                     page_size, max_pages, int(max_seq_len), float(scale),
                                     int(num_splits), _ptr(workspace), wsize, _dtype_code(q),
                                     _stream(stream, dev))
    _check("attn_decode_paged", st)
    _used_on(stream, q, k_pages, v_pages, block_table, seq_lens, workspace, o, lse)
    return o, lse


def attn_bwd_workspace_bytes(B: int, Hq: int, Nq: int) -> int:
    return int(lib().attn_bwd_workspace_bytes(B, Hq, Nq))


def attn_bwd(q, k, v, o, lse, dout, causal: bool, scale: float | None = None, dq=None, dk=None,
             dv=None, workspace=None, stream=None):
    """Backward of attn_fwd: q, o, dout [B, Nq, Hq, d]; k, v [B, Nk, Hkv, d] (bf16);
    lse [B, Hq, Nq] float32 from the forward.  Returns (dq, dk, dv)."""
    import torch
    B, Nq, Hq, d = q.shape
    Bk, Nk, Hkv, dk_ = k.shape
    if Bk != B or dk_ != d or tuple(v.shape) != tuple(k.shape):
        raise ValueError("shape mismatch between q and k/v")
    if tuple(o.shape) != tuple(q.shape) or tuple(dout.shape) != tuple(q.shape):
        raise ValueError("o and dout must have q's shape")
    if tuple(lse.shape) != (B, Hq, Nq):
        raise ValueError("lse must be [B, Hq, Nq]")
    if not (q.dtype == k.dtype == v.dtype == o.dtype == dout.dtype):
        raise ValueError("q, k, v, o and dout must share a dtype")
    dev = q.device
    for n, t in (("q", q), ("k", k), ("v", v), ("o", o), ("dout", dout)):
        _need_cuda_contig(n, t, dev)
    _need_buffer("lse", lse, (B, Hq, Nq), torch.float32, dev)
    if scale is None:
        scale = d ** -0.5
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    _need_buffer("dq", dq, q.shape, q.dtype, dev)
    _need_buffer("dk", dk, k.shape, k.dtype, dev)
    _need_buffer("dv", dv, v.shape, v.dtype, dev)
    wbytes = attn_bwd_workspace_bytes(B, Hq, Nq)
    if workspace is None:
        workspace = torch.empty(max(16, wbytes), dtype=torch.uint8, device=dev)
    _need_workspace(workspace, dev)
    wsize = workspace.numel() * workspace.element_size()
    with torch.cuda.device(dev):
        st = lib().attn_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dout), _ptr(dq),
                            _ptr(dk), _ptr(dv), B, Hq, Hkv, Nq, Nk, d, int(bool(causal)),
                            float(scale), _ptr(workspace), wsize, _dtype_code(q), _stream(stream, dev))
    _check("attn_bwd", st)
    _used_on(stream, q, k, v, o, lse, dout, dq, dk, dv, workspace)
    return dq, dk, dv


def attn_quantize_fp8(x, codes=None, scales=None, stream=None):
    """Block quantisation of a bf16 [B, N, H, d] tensor to e4m3 codes (uint8)
    with one float32 scale per (batch, head, 128-row block).  Returns
    (codes [B, N, H, d] uint8, scales [B, H, ceil(N/128)] float32)."""
    import torch
    B, N, H, d = x.shape
    dev = x.device
    _need_cuda_contig("x", x, dev)
    if x.dtype != torch.bfloat16:
        raise ValueError("x must be bfloat16")
    codes = torch.empty(x.shape, dtype=torch.uint8, device=dev) if codes is None else codes
    nb = (N + 127) // 128
    scales = torch.empty((B, H, nb), dtype=torch.float32, device=dev) if scales is None else scales
    _need_buffer("codes", codes, x.shape, torch.uint8, dev)
    _need_buffer("scales", scales, (B, H, nb), torch.float32, dev)
    with torch.cuda.device(dev):
        st = lib().attn_quantize_fp8(_ptr(x), _ptr(codes), _ptr(scales), B, N, H, d, _stream(stream, dev))
    _check("attn_quantize_fp8", st)
    _used_on(stream, x, codes, scales)
    return codes, scales


def attn_quantize_fp8_rotated(x, signs, codes=None, scales=None, stream=None):
    """attn_quantize_fp8 of x R, R = diag(signs) H / sqrt(d) (H the Sylvester
    Hadamard matrix): a random orthogonal transform that spreads outlier
    features before quantisation.  signs: float32 [d] of +-1 on x's device,
    the same for Q and K (then (qR)(kR)^T = qk^T and attn_fwd_fp8 takes the
    result unchanged).  d is 64 or 128.  Returns (codes, scales) as
    attn_quantize_fp8."""
    import torch
    B, N, H, d = x.shape
    dev = x.device
    _need_cuda_contig("x", x, dev)
    if x.dtype != torch.bfloat16:
        raise ValueError("x must be bfloat16")
    _need_buffer("signs", signs, (d,), torch.float32, dev)
    codes = torch.empty(x.shape, dtype=torch.uint8, device=dev) if codes is None else codes
    nb = (N + 127) // 128
    scales = torch.empty((B, H, nb), dtype=torch.float32, device=dev) if scales is None else scales
    _need_buffer("codes", codes, x.shape, torch.uint8, dev)
    _need_buffer("scales", scales, (B, H, nb), torch.float32, dev)
    with torch.cuda.device(dev):
        st = lib().attn_quantize_fp8_rotated(_ptr(x), _ptr(signs), _ptr(codes), _ptr(scales), B, N, H, d,
                                             _stream(stream, dev))
    _check("attn_quantize_fp8_rotated", st)
    _used_on(stream, x, signs, codes, scales)
    return codes, scales


def attn_fwd_fp8(q8, k8, v, q_scales, k_scales, causal: bool, scale: float | None = None, o=None,
                 lse=None, stream=None):
    """Forward with e4m3 Q and K codes and their block scales (from
    attn_quantize_fp8), bf16 V.  Returns (o [B, Nq, Hq, d] bf16, lse [B, Hq, Nq])."""
    import torch
    B, Nq, Hq, d = q8.shape
    Bk, Nk, Hkv, dk = k8.shape
    if Bk != B or dk != d or tuple(v.shape) != tuple(k8.shape):
        raise ValueError("shape mismatch")
    if q8.dtype != torch.uint8 or k8.dtype != torch.uint8 or v.dtype != torch.bfloat16:
        raise ValueError("q8 and k8 must be uint8 e4m3 codes and v bfloat16")
    dev = q8.device
    for n, t in (("q8", q8), ("k8", k8), ("v", v)):
        _need_cuda_contig(n, t, dev)
    _need_buffer("q_scales", q_scales, (B, Hq, (Nq + 127) // 128), torch.float32, dev)
    _need_buffer("k_scales", k_scales, (B, Hkv, (Nk + 127) // 128), torch.float32, dev)
    if scale is None:
        scale = d ** -0.5
    o = torch.empty((B, Nq, Hq, d), dtype=torch.bfloat16, device=dev) if o is None else o
    lse = torch.empty((B, Hq, Nq), dtype=torch.float32, device=dev) if lse is None else lse
    _need_buffer("o", o, (B, Nq, Hq, d), torch.bfloat16, dev)
    _need_buffer("lse", lse, (B, Hq, Nq), torch.float32, dev)
    with torch.cuda.device(dev):
        st = lib().attn_fwd_fp8(_ptr(q8), _ptr(k8), _ptr(v), _ptr(q_scales), _ptr(k_scales), _ptr(o),
                                _ptr(lse), B, Hq, Hkv, Nq, Nk, d, int(bool(causal)), float(scale),
                                _stream(stream, dev))
    _check("attn_fwd_fp8", st)
    _used_on(stream, q8, k8, v, q_scales, k_scales, o, lse)
    return o, lse


def fp8_v_ld(N: int) -> int:
    """Row length (keys) of attn_quantize_fp8_v's transposed codes: N rounded
    up to a multiple of 16."""
    return (N + 15) // 16 * 16


def attn_quantize_fp8_v(v, vt8=None, scales=None, stream=None):
    """e4m3 quantisation of V for attn_fwd_fp8_pv: one float32 scale per
    (batch, head) over the whole sequence, codes written transposed.  v: bf16
    [B, N, H, d], d 64 or 128.  Returns (vt8 [B, H, d, fp8_v_ld(N)] uint8,
    scales [B, H] float32); vt8[b, h, c, n] is the code of v[b, n, h, c]."""
    import torch
    B, N, H, d = v.shape
    dev = v.device
    _need_cuda_contig("v", v, dev)
    if v.dtype != torch.bfloat16:
        raise ValueError("v must be bfloat16")
    shape = (B, H, d, fp8_v_ld(N))
    vt8 = torch.empty(shape, dtype=torch.uint8, device=dev) if vt8 is None else vt8
    scales = torch.empty((B, H), dtype=torch.float32, device=dev) if scales is None else scales
    _need_buffer("vt8", vt8, shape, torch.uint8, dev)
    _need_buffer("scales", scales, (B, H), torch.float32, dev)
    with torch.cuda.device(dev):
        st = lib().attn_quantize_fp8_v(_ptr(v), _ptr(vt8), _ptr(scales), B, N, H, d, _stream(stream, dev))
    _check("attn_quantize_fp8_v", st)
    _used_on(stream, v, vt8, scales)
    return vt8, scales


def attn_fwd_fp8_pv(q8, k8, vt8, q_scales, k_scales, v_scales, causal: bool, scale: float | None = None,
                    o=None, lse=None, stream=None):
    """Forward with e4m3 Q, K (attn_quantize_fp8) and V (attn_quantize_fp8_v),
    and P rounded to e4m3 for the P V product.  Returns (o [B, Nq, Hq, d]
    bf16, lse [B, Hq, Nq] float32)."""
    import torch
    B, Nq, Hq, d = q8.shape
    Bk, Nk, Hkv, dk = k8.shape
    if Bk != B or dk != d or tuple(vt8.shape) != (B, Hkv, d, fp8_v_ld(Nk)):
        raise ValueError("shape mismatch")
    if q8.dtype != torch.uint8 or k8.dtype != torch.uint8 or vt8.dtype != torch.uint8:
        raise ValueError("q8, k8 and vt8 must be uint8 e4m3 codes")
    dev = q8.device
    for n, t in (("q8", q8), ("k8", k8), ("vt8", vt8)):
        _need_cuda_contig(n, t, dev)
    _need_buffer("q_scales", q_scales, (B, Hq, (Nq + 127) // 128), torch.float32, dev)
    _need_buffer("k_scales", k_scales, (B, Hkv, (Nk + 127) // 128), torch.float32, dev)
    _need_buffer("v_scales", v_scales, (B, Hkv), torch.float32, dev)
    if scale is None:
        scale = d ** -0.5
    o = torch.empty((B, Nq, Hq, d), dtype=torch.bfloat16, device=dev) if o is None else o
    lse = torch.empty((B, Hq, Nq), dtype=torch.float32, device=dev) if lse is None else lse
    _need_buffer("o", o, (B, Nq, Hq, d), torch.bfloat16, dev)
    _need_buffer("lse", lse, (B, Hq, Nq), torch.float32, dev)
    with torch.cuda.device(dev):
        st = lib().attn_fwd_fp8_pv(_ptr(q8), _ptr(k8), _ptr(vt8), _ptr(q_scales), _ptr(k_scales),
                                   _ptr(v_scales), _ptr(o), _ptr(lse), B, Hq, Hkv, Nq, Nk, d,
                                   int(bool(causal)), float(scale), _stream(stream, dev))
    _check("attn_fwd_fp8_pv", st)
    _used_on(stream, q8, k8, vt8, q_scales, k_scales, v_scales, o, lse)
    return o, lse


# ----------------------------------------------------------------------------- tests only

def attn_fwd_test(q, k, v, causal: bool, scale: float, options: AttnTestOptions, o=None, lse=None,
                  stream=None):
    """attn_fwd_test of include/attn_test.h: the bf16 forward with test
    options (kernel variants, wait bound, load injection).  Tests and
    measurements only.  Returns (o, lse)."""
    import torch
    B, Nq, Hq, d = q.shape
    Bk, Nk, Hkv, dk = k.shape
    if Bk != B or dk != d or tuple(v.shape) != tuple(k.shape):
        raise ValueError("shape mismatch")
    if not (q.dtype == k.dtype == v.dtype == torch.bfloat16):
        raise ValueError("q, k, v must be bfloat16")
    dev = q.device
    for n, t in (("q", q), ("k", k), ("v", v)):
        _need_cuda_contig(n, t, dev)
    o = torch.empty_like(q) if o is None else o
    lse = torch.empty((B, Hq, Nq), dtype=torch.float32, device=dev) if lse is None else lse
    _need_buffer("o", o, q.shape, q.dtype, dev)
    _need_buffer("lse", lse, (B, Hq, Nq), torch.float32, dev)
    with torch.cuda.device(dev):
        st = lib().attn_fwd_test(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, Hq, Hkv, Nq, Nk,
                                 d, int(bool(causal)), float(scale), ctypes.byref(options),
                                 _stream(stream, dev))
    _check("attn_fwd_test", st)
    _used_on(stream, q, k, v, o, lse)
    return o, lse


def attn_decode_test(q, k_cache, v_cache, scale: float, num_splits: int, options: AttnTestOptions,
                     workspace=None, o=None, lse=None, stream=None):
    """attn_decode_test of include/attn_test.h: the split-KV decode with the
    wait bound and load injection of `options`.  Tests only.  Returns (o, lse)."""
    import torch
    B, one, Hq, d = q.shape
    Bk, Nk, Hkv, dk = k_cache.shape
    if one != 1 or Bk != B or dk != d or tuple(v_cache.shape) != tuple(k_cache.shape):
        raise ValueError("shape mismatch")
    dev = q.device
    for n, t in (("q", q), ("k_cache", k_cache), ("v_cache", v_cache)):
        _need_cuda_contig(n, t, dev)
    if num_splits == 0 and Nk > 0:
        with torch.cuda.device(dev):
            num_splits = attn_decode_num_splits(B, Hq, Hkv, Nk, d)
    wbytes = attn_decode_workspace_bytes(B, Hq, Hkv, Nk, d, num_splits) if Nk > 0 else 0
    if workspace is None and wbytes > 0:
        workspace = torch.empty(wbytes, dtype=torch.uint8, device=dev)
    o = torch.empty_like(q) if o is None else o
    lse = torch.empty((B, Hq), dtype=torch.float32, device=dev) if lse is None else lse
    _need_buffer("o", o, q.shape, q.dtype, dev)
    _need_buffer("lse", lse, (B, Hq), torch.float32, dev)
    wsize = 0 if workspace is None else workspace.numel() * workspace.element_size()
    with torch.cuda.device(dev):
        st = lib().attn_decode_test(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(o), _ptr(lse), B, Hq,
                                    Hkv, Nk, d, float(scale), int(num_splits), _ptr(workspace), wsize,
                                    ctypes.byref(options), _stream(stream, dev))
    _check("attn_decode_test", st)
    _used_on(stream, q, k_cache, v_cache, workspace, o, lse)
    return o, lse
