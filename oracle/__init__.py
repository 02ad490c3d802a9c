"""Python access to the plain CPU oracle of the TurboQuant KV-cache codec.

TEST INFRASTRUCTURE ONLY. This package is imported by the tests, by the
package's smoke check and by the benchmark's CPU-baseline leg; the product
path (``turboquant_kv_cache_tq_gb300``) never imports it and shares no code
with it. The arithmetic lives in ``tq_oracle.c`` (single-threaded C, IEEE
binary32, one rounding per operation); this module only builds it with gcc
and marshals numpy arrays through ctypes.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SOURCES = ("tq_oracle.c", "tq_oracle_tables.c", "tq_oracle_attention.c")
LIB_PATH = os.path.join(_HERE, "libtq_oracle.so")
CFLAGS = ("-O2", "-std=c11", "-Wall", "-Wextra", "-ffp-contract=off", "-fno-fast-math", "-fPIC")

F32, BF16 = 0, 1
GROUP = 32
HEAD_DIMS = (64, 128, 256, 512)
VALUE_BITS = (2, 3, 4, 5, 8)
KEY_MODES = ((2, 0), (4, 0), (5, 0), (8, 0), (8, 1))  # (bits, signed)

_lock = threading.Lock()
_lib = None


def _stale() -> bool:
    if not os.path.exists(LIB_PATH):
        return True
    t = os.path.getmtime(LIB_PATH)
    return any(os.path.getmtime(os.path.join(_HERE, s)) > t for s in _SOURCES + ("tq_oracle.h",))


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/libtq_oracle.so`` (gcc, no SIMD flags)."""
    if force or _stale():
        tmp = LIB_PATH + ".tmp%d" % os.getpid()
        cmd = ["gcc", *CFLAGS, "-shared", "-o", tmp] + [os.path.join(_HERE, s) for s in _SOURCES] + ["-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, LIB_PATH)
    return LIB_PATH


def lib() -> ctypes.CDLL:
    global _lib
    with _lock:
        if _lib is None:
            build()
            _lib = _declare(ctypes.CDLL(LIB_PATH))
    return _lib


def _declare(L: ctypes.CDLL) -> ctypes.CDLL:
    P, I, I64, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float
    sig = {
        "oracle_sign_vector": (P, [I]),
        "oracle_lloyd_max": (I, [I, ctypes.POINTER(P), ctypes.POINTER(P)]),
        "oracle_packed_dim": (I64, [I64, I]),
        "oracle_f32_to_f16": (ctypes.c_uint16, [F]),
        "oracle_f16_to_f32": (F, [ctypes.c_uint16]),
        "oracle_f32_to_bf16": (ctypes.c_uint16, [F]),
        "oracle_bf16_to_f32": (F, [ctypes.c_uint16]),
        "oracle_round": (F, [F]),
        "oracle_f32_to_f16_n": (None, [P, I64, P]),
        "oracle_f16_to_f32_n": (None, [P, I64, P]),
        "oracle_f32_to_bf16_n": (None, [P, I64, P]),
        "oracle_hadamard_rows": (None, [P, I64, I, I]),
        "oracle_fwht_rows": (I, [P, I64, I, I]),
        "oracle_searchsorted": (None, [P, I, P, I64, P]),
        "oracle_pack_bits": (I, [P, I64, I, P]),
        "oracle_unpack_bits": (I, [P, I64, I, P]),
        "oracle_encode_keys_row": (I, [P, I, I, I, P, P, P]),
        "oracle_decode_keys_row": (I, [P, I, I, P, P, P]),
        "oracle_encode_values_row": (I, [P, I, I, P, P]),
        "oracle_decode_values_row": (I, [P, I, I, P, P]),
        "oracle_decode_values_rotated_row": (I, [P, I, I, P, P]),
        "oracle_encode_kv": (I, [P, P, I, I64, I64, I64, I64, I, I, I, P, P, P, P, P, I64, I64]),
        "oracle_decode_kv": (I, [P, P, P, P, P, I64, I64, I64, I64, I64, I, I, I, P, P, I, I]),
        "oracle_unrotate_rows": (I, [P, I64, I, P]),
        "oracle_decode_attention": (I, [P, I64, I64, I64, P, P, P, P, P, I64, I64, I64, I64, I, I, I, P,
                                        ctypes.c_double, P]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(L, name)
        fn.restype = res
        fn.argtypes = args
    return L


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data


class OracleError(RuntimeError):
    pass


def _check(status: int, what: str) -> None:
    if status != 0:
        raise OracleError("%s failed with oracle status %d" % (what, status))


# ---- tables ------------------------------------------------------------------
def sign_vector(d: int) -> np.ndarray:
    p = lib().oracle_sign_vector(d)
    if not p:
        raise OracleError("no sign vector for head_dim %d" % d)
    return np.ctypeslib.as_array((ctypes.c_byte * d).from_address(p)).astype(np.int8).copy()


def lloyd_max(bits: int) -> tuple[np.ndarray, np.ndarray]:
    c, b = ctypes.c_void_p(), ctypes.c_void_p()
    n = lib().oracle_lloyd_max(bits, ctypes.byref(c), ctypes.byref(b))
    if n == 0:
        raise OracleError("no Lloyd-Max table for bits=%d" % bits)
    cent = np.ctypeslib.as_array((ctypes.c_float * n).from_address(c.value)).copy()
    bnd = np.ctypeslib.as_array((ctypes.c_float * (n - 1)).from_address(b.value)).copy()
    return cent, bnd


def packed_dim(dim: int, bits: int) -> int:
    return int(lib().oracle_packed_dim(dim, bits))


# ---- conversions ---------------------------------------------------------------
def f32_to_f16_bits(x) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, np.uint16)
    lib().oracle_f32_to_f16_n(_ptr(x), x.size, _ptr(out))
    return out


def f16_bits_to_f32(h) -> np.ndarray:
    h = np.ascontiguousarray(h, dtype=np.uint16)
    out = np.empty(h.shape, np.float32)
    lib().oracle_f16_to_f32_n(_ptr(h), h.size, _ptr(out))
    return out


def f32_to_bf16_bits(x) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, np.uint16)
    lib().oracle_f32_to_bf16_n(_ptr(x), x.size, _ptr(out))
    return out


def bf16_bits_to_f32(h) -> np.ndarray:
    h = np.ascontiguousarray(h, dtype=np.uint16)
    return (h.astype(np.uint32) << 16).view(np.float32)


def round_half_even(x: float) -> float:
    return float(lib().oracle_round(float(x)))


# ---- rotation -------------------------------------------------------------------
def hadamard(x, normalised: bool = True) -> np.ndarray:
    """Hadamard transform of each row (last axis, a power of two)."""
    y = np.array(x, dtype=np.float32, order="C", copy=True)
    n = y.shape[-1]
    lib().oracle_hadamard_rows(_ptr(y), y.size // n, n, int(normalised))
    return y


def fwht(x, encode: bool) -> np.ndarray:
    y = np.array(x, dtype=np.float32, order="C", copy=True)
    d = y.shape[-1]
    _check(lib().oracle_fwht_rows(_ptr(y), y.size // d, d, int(encode)), "fwht")
    return y


def searchsorted(boundaries, x) -> np.ndarray:
    b = np.ascontiguousarray(boundaries, dtype=np.float32)
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, np.uint8)
    lib().oracle_searchsorted(_ptr(b), b.size, _ptr(x), x.size, _ptr(out))
    return out


# ---- packing ----------------------------------------------------------------------
def pack_bits(codes, bits: int) -> np.ndarray:
    """Pack each row (last axis) independently."""
    c = np.ascontiguousarray(codes, dtype=np.uint8)
    n = c.shape[-1]
    pd = packed_dim(n, bits)
    if pd < 0:
        raise OracleError("packed_dim(%d, %d) is not byte-aligned" % (n, bits))
    rows = c.reshape(-1, n)
    out = np.empty((rows.shape[0], pd), np.uint8)
    for r in range(rows.shape[0]):
        _check(lib().oracle_pack_bits(_ptr(rows[r]), n, bits, _ptr(out[r])), "pack_bits")
    return out.reshape(c.shape[:-1] + (pd,))


def unpack_bits(packed, bits: int, n: int) -> np.ndarray:
    p = np.ascontiguousarray(packed, dtype=np.uint8)
    pd = p.shape[-1]
    rows = p.reshape(-1, pd)
    out = np.empty((rows.shape[0], n), np.uint8)
    for r in range(rows.shape[0]):
        _check(lib().oracle_unpack_bits(_ptr(rows[r]), n, bits, _ptr(out[r])), "unpack_bits")
    return out.reshape(p.shape[:-1] + (n,))


# ---- rows -------------------------------------------------------------------------
def encode_keys(x, bits: int, signed: bool):
    """Rows of the last axis -> (codes uint8 [...,d], scales f16 bits, zeros f16 bits)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    d = x.shape[-1]
    rows = x.reshape(-1, d)
    codes = np.empty(rows.shape, np.uint8)
    sc = np.empty((rows.shape[0], d // GROUP), np.uint16)
    zr = np.empty_like(sc)
    for r in range(rows.shape[0]):
        _check(lib().oracle_encode_keys_row(_ptr(rows[r]), d, bits, int(signed), _ptr(codes[r]),
                                            _ptr(sc[r]), _ptr(zr[r])), "encode_keys")
    lead = x.shape[:-1]
    return codes.reshape(lead + (d,)), sc.reshape(lead + (d // GROUP,)), zr.reshape(lead + (d // GROUP,))


def decode_keys(codes, scales, zeros, signed: bool) -> np.ndarray:
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    d = codes.shape[-1]
    c = codes.reshape(-1, d)
    s = np.ascontiguousarray(scales, dtype=np.uint16).reshape(c.shape[0], -1)
    z = np.ascontiguousarray(zeros, dtype=np.uint16).reshape(c.shape[0], -1)
    out = np.empty(c.shape, np.float32)
    for r in range(c.shape[0]):
        _check(lib().oracle_decode_keys_row(_ptr(c[r]), d, int(signed), _ptr(s[r]), _ptr(z[r]),
                                            _ptr(out[r])), "decode_keys")
    return out.reshape(codes.shape)


def encode_values(x, bits: int):
    x = np.ascontiguousarray(x, dtype=np.float32)
    d = x.shape[-1]
    rows = x.reshape(-1, d)
    idx = np.empty(rows.shape, np.uint8)
    sc = np.empty((rows.shape[0], d // GROUP), np.uint16)
    for r in range(rows.shape[0]):
        _check(lib().oracle_encode_values_row(_ptr(rows[r]), d, bits, _ptr(idx[r]), _ptr(sc[r])),
               "encode_values")
    lead = x.shape[:-1]
    return idx.reshape(lead + (d,)), sc.reshape(lead + (d // GROUP,))


def decode_values(idx, scales, bits: int, rotated: bool = False) -> np.ndarray:
    idx = np.ascontiguousarray(idx, dtype=np.uint8)
    d = idx.shape[-1]
    c = idx.reshape(-1, d)
    s = np.ascontiguousarray(scales, dtype=np.uint16).reshape(c.shape[0], -1)
    out = np.empty(c.shape, np.float32)
    fn = lib().oracle_decode_values_rotated_row if rotated else lib().oracle_decode_values_row
    for r in range(c.shape[0]):
        _check(fn(_ptr(c[r]), d, bits, _ptr(s[r]), _ptr(out[r])), "decode_values")
    return out.reshape(idx.shape)


def unrotate(x) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    d = x.shape[-1]
    out = np.empty_like(x)
    _check(lib().oracle_unrotate_rows(_ptr(x), x.size // d, d, _ptr(out)), "unrotate")
    return out


# ---- whole tensors -----------------------------------------------------------------
def _as_raw(x):
    """numpy fp32 array -> (array, F32); uint16 array of bf16 bits -> (array, BF16)."""
    x = np.ascontiguousarray(x)
    if x.dtype == np.float32:
        return x, F32
    if x.dtype == np.uint16:
        return x, BF16
    raise OracleError("K/V must be float32 or uint16 (bf16 bit patterns), got %s" % x.dtype)


def alloc_cache(B, H, t_cap, D, k_bits, v_bits):
    G = D // GROUP
    return dict(
        k_codes=np.zeros((B, H, t_cap, packed_dim(D, k_bits)), np.uint8),
        k_scales=np.zeros((B, H, t_cap, G), np.uint16),
        k_zeros=np.zeros((B, H, t_cap, G), np.uint16),
        v_codes=np.zeros((B, H, t_cap, packed_dim(D, v_bits)), np.uint8),
        v_scales=np.zeros((B, H, t_cap, G), np.uint16),
    )


def encode_kv(k, v, k_bits: int, k_signed: bool, v_bits: int, cache=None, t_cap=None, t_off=0):
    """Encode K, V [B,H,T,D] into a packed cache dict (allocated when None)."""
    k, dt = _as_raw(k)
    v, dv = _as_raw(v)
    if dt != dv or k.shape != v.shape:
        raise OracleError("K and V must share dtype and shape")
    B, H, T, D = k.shape
    if cache is None:
        cache = alloc_cache(B, H, t_cap if t_cap is not None else T, D, k_bits, v_bits)
    t_cap = cache["k_codes"].shape[2]
    st = lib().oracle_encode_kv(_ptr(k), _ptr(v), dt, B, H, T, D, k_bits, int(k_signed), v_bits,
                                _ptr(cache["k_codes"]), _ptr(cache["k_scales"]), _ptr(cache["k_zeros"]),
                                _ptr(cache["v_codes"]), _ptr(cache["v_scales"]), t_cap, t_off)
    _check(st, "encode_kv")
    return cache


def decode_kv(cache, T: int, k_bits: int, k_signed: bool, v_bits: int, out_dtype: int = F32,
              rotated_v: bool = False):
    """Decode tokens [0,T) of a packed cache -> (K, V) [B,H,T,D] (fp32, or bf16 bits)."""
    B, H, t_cap, _ = cache["k_codes"].shape
    D = cache["k_scales"].shape[-1] * GROUP
    odt = np.float32 if out_dtype == F32 else np.uint16
    ko = np.empty((B, H, T, D), odt)
    vo = np.empty((B, H, T, D), odt)
    st = lib().oracle_decode_kv(_ptr(cache["k_codes"]), _ptr(cache["k_scales"]), _ptr(cache["k_zeros"]),
                                _ptr(cache["v_codes"]), _ptr(cache["v_scales"]), B, H, T, D, t_cap,
                                k_bits, int(k_signed), v_bits, _ptr(ko), _ptr(vo), out_dtype,
                                int(rotated_v))
    _check(st, "decode_kv")
    return ko, vo


def decode_attention(q_bits, cache, T: int, k_bits: int, k_signed: bool, v_bits: int,
                     left_pad=None, scale=None) -> np.ndarray:
    """Attention of bf16 queries q [B,Hq,Nq,D] (uint16 bit patterns) over tokens
    [0,T) of a packed cache (tryDecodePackedKv with deferV, softmax attention,
    unrotateValues), in double precision -> float64 [B,Hq,Nq,D]."""
    q_bits = np.ascontiguousarray(q_bits, dtype=np.uint16)
    B, Hq, Nq, D = q_bits.shape
    Bc, Hkv, t_cap, _ = cache["k_codes"].shape
    if Bc != B:
        raise OracleError("q and cache batch differ")
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    lp = None
    if left_pad is not None:
        lp = np.ascontiguousarray(left_pad, dtype=np.int32)
        if lp.shape != (B,):
            raise OracleError("left_pad must have one entry per batch row")
    out = np.empty((B, Hq, Nq, D), np.float64)
    st = lib().oracle_decode_attention(_ptr(q_bits), B, Hq, Nq, _ptr(cache["k_codes"]), _ptr(cache["k_scales"]),
                                       _ptr(cache["k_zeros"]), _ptr(cache["v_codes"]), _ptr(cache["v_scales"]),
                                       Hkv, T, D, t_cap, k_bits, int(k_signed), v_bits,
                                       None if lp is None else _ptr(lp), float(scale), _ptr(out))
    _check(st, "decode_attention")
    return out
