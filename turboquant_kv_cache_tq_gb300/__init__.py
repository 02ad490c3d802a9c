"""GB300 TurboQuant KV-cache codec: Python binding of the C ABI in include/tq.h.

This module only marshals torch tensors (device pointers, sizes and the
current CUDA stream) into ``libtq.so``; every step of encode and decode runs
in the library's CUDA kernels. There is no fallback: if the library is not
built, importing works but every call raises.

Names follow the C ABI: ``tq_packed_dim``, ``tq_encode_kv``, ``tq_decode_kv``,
``tq_lloyd_max_index``, ``tq_status_string``; ``alloc_cache`` allocates the
five packed-cache buffers with torch.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

__all__ = [
    "TQError", "lib", "tq_packed_dim", "tq_encode_kv", "tq_decode_kv", "tq_decode_kv_rotated",
    "tq_unrotate", "tq_lloyd_max_index", "tq_decode_attention", "tq_decode_attention_workspace_size",
    "tq_cache_assemble", "merge_rows", "extend_rows", "extract_row", "filter_rows", "tq_lloyd_max_fit",
    "tq_lloyd_max_fit_status",
    "tq_status_string", "alloc_cache", "HEAD_DIMS", "VALUE_BITS", "KEY_MODES",
]

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libtq.so")
HEAD_DIMS = (64, 128, 256, 512)
VALUE_BITS = (2, 3, 4, 5, 8)
KEY_MODES = ((2, False), (4, False), (5, False), (8, False), (8, True))
GROUP = 32
TQ_F32, TQ_BF16 = 0, 1
_DTYPE = {torch.float32: TQ_F32, torch.bfloat16: TQ_BF16}
_NAMES = ("TQ_OK", "TQ_ERR_INVALID_ARG", "TQ_ERR_HEAD_DIM", "TQ_ERR_BITS", "TQ_ERR_ALIGNMENT",
          "TQ_ERR_DTYPE", "TQ_ERR_CUDA", "TQ_ERR_TIMEOUT", "TQ_ERR_DEVICE_CHECK")

_lock = threading.Lock()
_lib = None


class TQError(RuntimeError):
    """A non-OK tq_status from the library."""

    def __init__(self, status: int, what: str):
        self.status = status
        name = _NAMES[status] if 0 <= status < len(_NAMES) else str(status)
        super().__init__("%s: %s (%s)" % (what, name, tq_status_string(status)))


def lib() -> ctypes.CDLL:
    """The loaded libtq.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    "libtq.so is not built (%s); run python -m turboquant_kv_cache_tq_gb300.build" % LIB_PATH)
            _lib = load_library(LIB_PATH)
    return _lib


def load_library(path: str) -> ctypes.CDLL:
    """A build of the C ABI at `path` (libtq.so or its debug variant
    libtq_debug.so) with every entry point's argument types declared."""
    L = ctypes.CDLL(path)
    P, I, I64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64
    L.tq_packed_dim.restype = I64
    L.tq_packed_dim.argtypes = [I64, I]
    L.tq_encode_kv.restype = I
    L.tq_encode_kv.argtypes = [P, P, I, I64, I64, I64, I64, I, I, I, P, P, P, P, P, I64, I64, P]
    L.tq_decode_kv.restype = I
    L.tq_decode_kv.argtypes = [P, P, P, P, P, I64, I64, I64, I64, I64, I, I, I, P, P, I, P]
    L.tq_decode_kv_rotated.restype = I
    L.tq_decode_kv_rotated.argtypes = [P, P, P, P, P, I64, I64, I64, I64, I64, I, I, I, P, P, I, P]
    L.tq_unrotate.restype = I
    L.tq_unrotate.argtypes = [P, I, I64, I64, P, P]
    L.tq_lloyd_max_index.restype = I
    L.tq_lloyd_max_index.argtypes = [P, I64, I, P, P]
    L.tq_decode_attention.restype = I
    L.tq_decode_attention.argtypes = [P, I64, I64, I64, P, P, P, P, P, I64, I64, I64, I64, I, I, I, P,
                                      ctypes.c_float, P, I, P, I64, P]
    L.tq_decode_attention_noalloc.restype = I
    L.tq_decode_attention_noalloc.argtypes = [P, I64, I64, I64, P, P, P, P, P, I64, I64, I64, I64, I, I,
                                              I, P, ctypes.c_float, P, I, P]
    L.tq_decode_attention_workspace_size.restype = I64
    L.tq_decode_attention_workspace_size.argtypes = [I64, I64, I64, I64]
    L.tq_cache_assemble.restype = I
    L.tq_cache_assemble.argtypes = [P, I64, I64, I64, I, I, P, P, P, P, P, I64, I64, P]
    L.tq_lloyd_max_fit.restype = I
    L.tq_lloyd_max_fit.argtypes = [P, I64, I, I, P, P, P, P, I64, P]
    L.tq_lloyd_max_fit_bounded.restype = I
    L.tq_lloyd_max_fit_bounded.argtypes = [P, I64, I, I, P, P, P, P, I64, I64, I, P]
    L.tq_lloyd_max_fit_status.restype = I
    L.tq_lloyd_max_fit_status.argtypes = [P, P]
    L.tq_lloyd_max_fit_workspace_size.restype = I64
    L.tq_lloyd_max_fit_workspace_size.argtypes = [I]
    L.tq_device_status.restype = I
    L.tq_device_status.argtypes = [P]
    L.tq_debug_checks.restype = I
    L.tq_debug_checks.argtypes = []
    L.tq_status_string.restype = ctypes.c_char_p
    L.tq_status_string.argtypes = [I]
    return L


def tq_status_string(status: int) -> str:
    return lib().tq_status_string(int(status)).decode()


def _stream_handle(stream, device) -> int:
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return stream.cuda_stream


def _check(status: int, what: str) -> None:
    if status != 0:
        raise TQError(status, what)


def tq_packed_dim(dim: int, bits: int) -> int:
    """Bytes of one packed row of `dim` codes at `bits` bits (raises if not byte-aligned)."""
    r = int(lib().tq_packed_dim(int(dim), int(bits)))
    if r < 0:
        raise TQError(-r, "tq_packed_dim(%d, %d)" % (dim, bits))
    return r


def alloc_cache(B: int, H: int, t_cap: int, D: int, k_bits: int, v_bits: int, device="cuda") -> dict:
    """The five packed-cache buffers [B,H,t_cap,X] (codes uint8, scales/zeros fp16)."""
    G = D // GROUP
    return dict(
        k_codes=torch.zeros((B, H, t_cap, tq_packed_dim(D, k_bits)), dtype=torch.uint8, device=device),
        k_scales=torch.zeros((B, H, t_cap, G), dtype=torch.float16, device=device),
        k_zeros=torch.zeros((B, H, t_cap, G), dtype=torch.float16, device=device),
        v_codes=torch.zeros((B, H, t_cap, tq_packed_dim(D, v_bits)), dtype=torch.uint8, device=device),
        v_scales=torch.zeros((B, H, t_cap, G), dtype=torch.float16, device=device),
    )


def _cache_ptrs(cache: dict):
    for name in ("k_codes", "k_scales", "k_zeros", "v_codes", "v_scales"):
        t = cache[name]
        if not t.is_contiguous():
            raise ValueError("cache buffer %s must be contiguous" % name)
    return [cache[n].data_ptr() for n in ("k_codes", "k_scales", "k_zeros", "v_codes", "v_scales")]


def tq_encode_kv(k: torch.Tensor, v: torch.Tensor, k_bits: int, k_signed: bool, v_bits: int,
                 cache: dict, t_off: int = 0, stream=None) -> dict:
    """Encode K, V [B,H,T,D] (fp32 or bf16, contiguous, on the GPU) into tokens
    [t_off, t_off+T) of `cache` (capacity = its token axis). Asynchronous on
    `stream` (default: the current stream)."""
    if k.shape != v.shape or k.dtype != v.dtype or k.dim() != 4:
        raise ValueError("K and V must be [B,H,T,D] tensors of one shape and dtype")
    if k.dtype not in _DTYPE:
        raise ValueError("K/V dtype must be float32 or bfloat16, got %s" % k.dtype)
    if not (k.is_contiguous() and v.is_contiguous()):
        raise ValueError("K and V must be contiguous")
    B, H, T, D = k.shape
    t_cap = cache["k_codes"].shape[2]
    st = lib().tq_encode_kv(k.data_ptr(), v.data_ptr(), _DTYPE[k.dtype], B, H, T, D, int(k_bits),
                            int(bool(k_signed)), int(v_bits), *_cache_ptrs(cache), t_cap, int(t_off),
                            _stream_handle(stream, k.device))
    _check(st, "tq_encode_kv")
    return cache


def _decode(fn, name, cache, T, k_bits, k_signed, v_bits, out_dtype, k_out, v_out, stream):
    B, H, t_cap, _ = cache["k_codes"].shape
    D = cache["k_scales"].shape[-1] * GROUP
    dev = cache["k_codes"].device
    if out_dtype not in _DTYPE:
        raise ValueError("out_dtype must be float32 or bfloat16")
    if k_out is None:
        k_out = torch.empty((B, H, T, D), dtype=out_dtype, device=dev)
    if v_out is None:
        v_out = torch.empty((B, H, T, D), dtype=out_dtype, device=dev)
    for t in (k_out, v_out):
        if t.dtype != out_dtype or tuple(t.shape) != (B, H, T, D) or not t.is_contiguous():
            raise ValueError("k_out/v_out must be contiguous [B,H,T,D] tensors of out_dtype")
    st = fn(*_cache_ptrs(cache), B, H, T, D, t_cap, int(k_bits), int(bool(k_signed)), int(v_bits),
            k_out.data_ptr(), v_out.data_ptr(), _DTYPE[out_dtype], _stream_handle(stream, dev))
    _check(st, name)
    return k_out, v_out


def tq_decode_kv(cache: dict, T: int, k_bits: int, k_signed: bool, v_bits: int,
                 out_dtype=torch.bfloat16, k_out=None, v_out=None, stream=None):
    """Decode tokens [0,T) of `cache` into K, V [B,H,T,D] of `out_dtype`
    (allocated when not given). Asynchronous on `stream`."""
    return _decode(lib().tq_decode_kv, "tq_decode_kv", cache, T, k_bits, k_signed, v_bits, out_dtype,
                   k_out, v_out, stream)


def tq_decode_kv_rotated(cache: dict, T: int, k_bits: int, k_signed: bool, v_bits: int,
                         out_dtype=torch.bfloat16, k_out=None, v_out=None, stream=None):
    """As tq_decode_kv, but V stays in the rotated domain (centroid * scale,
    no inverse transform); undo it on an attention output with tq_unrotate."""
    return _decode(lib().tq_decode_kv_rotated, "tq_decode_kv_rotated", cache, T, k_bits, k_signed, v_bits,
                   out_dtype, k_out, v_out, stream)


def tq_unrotate(x: torch.Tensor, out=None, stream=None) -> torch.Tensor:
    """Inverse value rotation of the rows of `x` ([..., D], fp32 or bf16,
    contiguous), computed in fp32 and returned in x's dtype. `out` must not
    overlap x."""
    if x.dtype not in _DTYPE or not x.is_contiguous() or x.dim() < 1:
        raise ValueError("x must be a contiguous float32 or bfloat16 tensor")
    D = x.shape[-1]
    if out is None:
        out = torch.empty_like(x)
    if out.dtype != x.dtype or out.shape != x.shape or not out.is_contiguous():
        raise ValueError("out must be a contiguous tensor of x's shape and dtype")
    n = x.numel() // D if D else 0
    st = lib().tq_unrotate(x.data_ptr(), _DTYPE[x.dtype], n, D, out.data_ptr(), _stream_handle(stream, x.device))
    _check(st, "tq_unrotate")
    return out


def tq_lloyd_max_index(u: torch.Tensor, v_bits: int, out=None, stream=None) -> torch.Tensor:
    """count(boundaries < u) for each fp32 element of `u` (uint8 result)."""
    if u.dtype != torch.float32 or not u.is_contiguous():
        raise ValueError("u must be a contiguous float32 tensor")
    if out is None:
        out = torch.empty(u.shape, dtype=torch.uint8, device=u.device)
    st = lib().tq_lloyd_max_index(u.data_ptr(), u.numel(), int(v_bits), out.data_ptr(),
                                  _stream_handle(stream, u.device))
    _check(st, "tq_lloyd_max_index")
    return out


def tq_decode_attention_workspace_size(B: int, Hkv: int, T: int, D: int) -> int:
    """Bytes of scratch tq_decode_attention needs (on the current device)."""
    r = int(lib().tq_decode_attention_workspace_size(int(B), int(Hkv), int(T), int(D)))
    if r < 0:
        raise TQError(-r, "tq_decode_attention_workspace_size")
    return r


def tq_decode_attention(q: torch.Tensor, cache: dict, T: int, k_bits: int, k_signed: bool, v_bits: int,
                        left_pad=None, scale=None, out_dtype=torch.bfloat16, out=None, workspace=None,
                        stream=None) -> torch.Tensor:
    """Attention of bf16 queries q [B,Hq,Nq,D] over tokens [0,T) of a packed
    cache [B,Hkv,t_cap,*] (t_cap a multiple of 16), output unrotated
    [B,Hq,Nq,D] of out_dtype. left_pad: int32 device tensor [B] or None.
    workspace: a uint8 device tensor of at least
    tq_decode_attention_workspace_size bytes (allocated when None)."""
    if q.dtype != torch.bfloat16 or q.dim() != 4 or not q.is_contiguous():
        raise ValueError("q must be a contiguous [B,Hq,Nq,D] bfloat16 tensor")
    if out_dtype not in _DTYPE:
        raise ValueError("out_dtype must be float32 or bfloat16")
    B, Hq, Nq, D = q.shape
    Bc, Hkv, t_cap, _ = cache["k_codes"].shape
    if Bc != B:
        raise ValueError("q and the cache must have the same batch size")
    dev = q.device
    if scale is None:
        scale = D ** -0.5
    if out is None:
        out = torch.empty((B, Hq, Nq, D), dtype=out_dtype, device=dev)
    if out.dtype != out_dtype or tuple(out.shape) != (B, Hq, Nq, D) or not out.is_contiguous():
        raise ValueError("out must be a contiguous [B,Hq,Nq,D] tensor of out_dtype")
    lp = 0
    if left_pad is not None:
        if left_pad.dtype != torch.int32 or tuple(left_pad.shape) != (B,) or not left_pad.is_contiguous():
            raise ValueError("left_pad must be a contiguous int32 tensor [B]")
        lp = left_pad.data_ptr()
    need = tq_decode_attention_workspace_size(B, Hkv, T, D)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=dev)
    st = lib().tq_decode_attention(q.data_ptr(), B, Hq, Nq, *_cache_ptrs(cache), Hkv, int(T), D, t_cap,
                                   int(k_bits), int(bool(k_signed)), int(v_bits), lp or None, float(scale),
                                   out.data_ptr(), _DTYPE[out_dtype], workspace.data_ptr(),
                                   workspace.numel() * workspace.element_size(), _stream_handle(stream, dev))
    _check(st, "tq_decode_attention")
    return out


# ---- batched packed-cache rows (batched-quant.ts) ---------------------------------
class TQRowSource(ctypes.Structure):
    """tq_row_source of include/tq.h."""
    _fields_ = [("k_codes", ctypes.c_void_p), ("k_scales", ctypes.c_void_p), ("k_zeros", ctypes.c_void_p),
                ("v_codes", ctypes.c_void_p), ("v_scales", ctypes.c_void_p), ("B", ctypes.c_int64),
                ("b", ctypes.c_int64), ("t_cap", ctypes.c_int64), ("t_start", ctypes.c_int64),
                ("len", ctypes.c_int64)]


def _cache_geometry(cache: dict):
    B, H, t_cap, xk = cache["k_codes"].shape
    D = cache["k_scales"].shape[-1] * GROUP
    return B, H, t_cap, D, xk * 8 // D, cache["v_codes"].shape[-1] * 8 // D


def tq_cache_assemble(sources, dst: dict, width: int, stream=None) -> dict:
    """Assemble destination batch row r from sources[r] = (cache, b, t_start,
    length) or None (an all-padding row): width - length zero tokens, then the
    source's tokens [t_start, t_start + length), for every head and buffer."""
    n, H, t_cap, D, kb, vb = _cache_geometry(dst)
    if len(sources) != n:
        raise ValueError("one source per destination batch row")
    arr = (TQRowSource * max(n, 1))()
    for r, src in enumerate(sources):
        if src is None:
            arr[r] = TQRowSource(None, None, None, None, None, 0, 0, 0, 0, 0)
            continue
        cache, b, t0, length = src
        Bs, Hs, tcs, Ds, kbs, vbs = _cache_geometry(cache)
        if (Hs, Ds, kbs, vbs) != (H, D, kb, vb):
            raise ValueError("source and destination caches differ in heads, head_dim or bit widths")
        arr[r] = TQRowSource(*_cache_ptrs(cache), Bs, int(b), tcs, int(t0), int(length))
    st = lib().tq_cache_assemble(ctypes.cast(arr, ctypes.c_void_p), n, H, D, kb, vb, *_cache_ptrs(dst), t_cap,
                                 int(width), _stream_handle(stream, dst["k_codes"].device))
    _check(st, "tq_cache_assemble")
    return dst


def _alloc_like(cache: dict, B: int, t_cap: int) -> dict:
    _, H, _, D, kb, vb = _cache_geometry(cache)
    return alloc_cache(B, H, t_cap, D, kb, vb, device=cache["k_codes"].device)


def merge_rows(rows, t_cap=None, stream=None):
    """mergeQuantRows: rows = [(cache, length)] single-row caches ([1,H,*,X],
    tokens [0, length) valid) -> (batch cache [N,H,t_cap,X], left pads, width)
    with every row right-justified in width = max length."""
    width = max(int(n) for _, n in rows)
    pads = [width - int(n) for _, n in rows]
    dst = _alloc_like(rows[0][0], len(rows), width if t_cap is None else t_cap)
    tq_cache_assemble([(c, 0, 0, n) for c, n in rows], dst, width, stream)
    return dst, pads, width


def extend_rows(batch, S: int, pads, row, t_cap=None, stream=None):
    """extendQuantRows: append row = (cache, length) to a batch whose window
    is S tokens wide; the narrower side is padded on the left."""
    rc, n = row
    width = max(int(S), int(n))
    B = batch["k_codes"].shape[0]
    dst = _alloc_like(batch, B + 1, width if t_cap is None else t_cap)
    srcs = [(batch, b, 0, S) for b in range(B)] + [(rc, 0, 0, n)]
    tq_cache_assemble(srcs, dst, width, stream)
    return dst, [p + (width - S) for p in pads] + [width - int(n)], width


def extract_row(batch, S: int, pad: int, i: int, stream=None) -> dict:
    """extractQuantRow: batch row i past its left pad as a fresh single-row
    cache [1, H, S - pad, X]."""
    dst = _alloc_like(batch, 1, int(S) - int(pad))
    tq_cache_assemble([(batch, i, pad, int(S) - int(pad))], dst, int(S) - int(pad), stream)
    return dst


def filter_rows(batch, S: int, keep, stream=None) -> dict:
    """filterQuantRows: the batch rows `keep`, in that order, same window."""
    dst = _alloc_like(batch, len(keep), batch["k_codes"].shape[2])
    tq_cache_assemble([(batch, int(b), 0, S) for b in keep], dst, S, stream)
    return dst


# ---- Lloyd-Max table fit (turboquant-tables.ts) -----------------------------------
def tq_lloyd_max_fit(x: torch.Tensor, init: torch.Tensor, iters: int, workspace=None, stream=None,
                     spin_limit: int = 0, absent_block: int = -1):
    """Lloyd-Max fit of len(init) levels to the fp32 samples x (device), from
    the ascending centroids init -> (centroids, boundaries), fp32 tensors.
    spin_limit / absent_block: see tq_lloyd_max_fit_bounded (0 / -1: the
    plain fit); tq_lloyd_max_fit_status(workspace) reports a give-up."""
    if x.dtype != torch.float32 or init.dtype != torch.float32 or not (x.is_contiguous() and init.is_contiguous()):
        raise ValueError("x and init must be contiguous float32 tensors")
    K = init.numel()
    r = int(lib().tq_lloyd_max_fit_workspace_size(K))
    if r < 0:
        raise TQError(-r, "tq_lloyd_max_fit_workspace_size")
    if workspace is None:
        workspace = torch.empty(r, dtype=torch.uint8, device=x.device)
    c = torch.empty(K, dtype=torch.float32, device=x.device)
    b = torch.empty(max(K - 1, 1), dtype=torch.float32, device=x.device)
    st = lib().tq_lloyd_max_fit_bounded(x.data_ptr(), x.numel(), K, int(iters), init.data_ptr(), c.data_ptr(),
                                        b.data_ptr(), workspace.data_ptr(), workspace.numel(), int(spin_limit),
                                        int(absent_block), _stream_handle(stream, x.device))
    _check(st, "tq_lloyd_max_fit")
    return c, b[: K - 1]


def tq_lloyd_max_fit_status(workspace: torch.Tensor, stream=None) -> int:
    """Waits for `stream`, then returns the status of the last fit run with
    `workspace`: 0 (TQ_OK) or 7 (TQ_ERR_TIMEOUT: a grid-barrier wait gave up)."""
    st = int(lib().tq_lloyd_max_fit_status(workspace.data_ptr(), _stream_handle(stream, workspace.device)))
    if st not in (0, 7):
        raise TQError(st, "tq_lloyd_max_fit_status")
    return st
