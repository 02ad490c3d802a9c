"""Helpers shared by the GPU parity tests: run the CUDA path through the C ABI
and the oracle on the same seeded inputs, and compare.

Acceptance (element by element):
- packed K codes, K scales, K zeros and V scales: bit-exact (an fp16 NaN
  equals any other NaN: IEEE arithmetic fixes that a result is NaN, not its
  payload or sign);
- packed V codes: bit-exact, except indices whose normalised rotated value u
  lies within 1e-5 of a Lloyd-Max boundary (at most 1e-4 of the elements);
- decoded tensors: within 1e-5 relative error in fp32 (NaN where the oracle
  has NaN), and bf16 outputs equal to the round-to-nearest-even of the
  oracle's fp32 result (ties of that rounding are not reachable off by one:
  the fp32 values must already agree to 1e-5).
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import turboquant_kv_cache_tq_gb300 as tq
from turboquant_kv_cache_tq_gb300.workloads import to_oracle

V_TOL = 1e-5
V_MAX_FRAC = 1e-4
DEC_RTOL = 1e-5

CACHE_KEYS = ("k_codes", "k_scales", "k_zeros", "v_codes", "v_scales")


def f16_is_nan(h: np.ndarray) -> np.ndarray:
    """fp16 bit patterns that encode a NaN (any sign or payload)."""
    h = np.asarray(h).astype(np.uint16)
    return ((h & 0x7C00) == 0x7C00) & ((h & 0x03FF) != 0)


def require_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from turboquant_kv_cache_tq_gb300 import build

    build.build()
    return tq.lib()


def cache_to_numpy(cache: dict) -> dict:
    out = {}
    for k in CACHE_KEYS:
        t = cache[k].detach().cpu().contiguous()
        out[k] = t.numpy() if t.dtype == torch.uint8 else t.view(torch.int16).numpy().view(np.uint16)
    return out


def cache_from_numpy(c: dict, device="cuda") -> dict:
    out = {}
    for k in CACHE_KEYS:
        a = np.ascontiguousarray(c[k])
        t = torch.from_numpy(a.view(np.int16) if a.dtype == np.uint16 else a)
        out[k] = (t.view(torch.float16) if a.dtype == np.uint16 else t).to(device)
    return out


def gpu_encode(k, v, k_bits, k_signed, v_bits, t_cap=None, t_off=0, cache=None, fill=None):
    kd, vd = k.cuda(), v.cuda()
    B, H, T, D = k.shape
    if cache is None:
        cache = tq.alloc_cache(B, H, T if t_cap is None else t_cap, D, k_bits, v_bits)
        if fill is not None:
            for t in cache.values():
                t.view(torch.uint8).fill_(fill)
    tq.tq_encode_kv(kd, vd, k_bits, k_signed, v_bits, cache, t_off=t_off)
    torch.cuda.synchronize()
    return cache


def _unpack_rows(packed, bits, d):
    return oracle.unpack_bits(packed.reshape(-1, packed.shape[-1]), bits, d)


def rotated_normalised(v_np, d):
    """u = fwht(v) / (rms + eps) per element, in float64 from the oracle's
    rotation (only used to classify index mismatches; the fp32 values of the
    codec agree with these to ~1e-7 relative)."""
    x = v_np if v_np.dtype == np.float32 else oracle.bf16_bits_to_f32(v_np)
    y = oracle.fwht(x.reshape(-1, d), encode=True).astype(np.float64)
    g = y.reshape(y.shape[0], d // 32, 32)
    r = np.sqrt((g * g).mean(-1))
    return y / (np.repeat(r, 32, axis=1) + 1e-8)


def compare_encoded(gpu: dict, ref: dict, D: int, v_bits: int, v_input=None, rows=None):
    """Assert the acceptance rules on two packed caches (numpy dicts), either on
    all rows or on the selected cache rows `rows` (indices into B*H*t_cap)."""
    def sel(a):
        a = a.reshape(-1, a.shape[-1])
        return a if rows is None else a[rows]

    for key in ("k_codes", "k_scales", "k_zeros", "v_scales"):
        g, r = sel(gpu[key]), sel(ref[key])
        ne = g != r
        if key != "k_codes":
            ne &= ~(f16_is_nan(g) & f16_is_nan(r))  # IEEE leaves a NaN's payload open
        if ne.any():
            bad = np.argwhere(ne)
            raise AssertionError("%s differs at %d places, first %s: gpu %s ref %s"
                                 % (key, len(bad), bad[0].tolist(), g[tuple(bad[0])], r[tuple(bad[0])]))
    g, r = sel(gpu["v_codes"]), sel(ref["v_codes"])
    if np.array_equal(g, r):
        return 0
    gi = _unpack_rows(g, v_bits, D)
    ri = _unpack_rows(r, v_bits, D)
    mism = np.argwhere(gi != ri)
    assert v_input is not None, "V codes differ and no input given to classify them"
    u = rotated_normalised(v_input, D)
    _, bnd = oracle.lloyd_max(v_bits)
    for (row, e) in mism:
        dist = np.min(np.abs(u[row, e] - bnd.astype(np.float64)))
        assert dist <= V_TOL, "V index differs at row %d elem %d (gpu %d, ref %d, |u-b| = %g)" % (
            row, e, gi[row, e], ri[row, e], dist)
    assert len(mism) <= max(1, V_MAX_FRAC * gi.size), "%d V index mismatches" % len(mism)
    return len(mism)


def compare_decoded(gpu: np.ndarray, ref: np.ndarray, what: str):
    """fp32: NaN positions equal, |g - r| <= 1e-5 |r| elsewhere."""
    g = gpu.astype(np.float64)
    r = ref.astype(np.float64)
    gn, rn = np.isnan(g), np.isnan(r)
    assert np.array_equal(gn, rn), "%s: NaN positions differ (%d vs %d)" % (what, gn.sum(), rn.sum())
    inf = np.isinf(r)
    assert np.array_equal(g[inf], r[inf]), "%s: infinities differ" % what
    ok = ~rn & ~inf
    err = np.abs(g[ok] - r[ok])
    lim = DEC_RTOL * np.abs(r[ok])
    if not np.all((err <= lim) | (err == 0)):
        i = np.argmax(err - lim)
        raise AssertionError("%s: relative error above 1e-5 (gpu %r ref %r)" % (what, g[ok][i], r[ok][i]))
    return int(np.count_nonzero(err))


def oracle_encode(k, v, k_bits, k_signed, v_bits, t_cap=None, t_off=0, cache=None):
    return oracle.encode_kv(to_oracle(k), to_oracle(v), k_bits, k_signed, v_bits, cache=cache,
                            t_cap=t_cap, t_off=t_off)


def check_roundtrip(k, v, k_bits, k_signed, v_bits, t_cap=None, t_off=0):
    """Encode on both sides, compare; decode the oracle's bytes on both sides
    (fp32 and bf16), compare. Returns (#V index exceptions, #inexact decodes)."""
    B, H, T, D = k.shape
    gcache = gpu_encode(k, v, k_bits, k_signed, v_bits, t_cap=t_cap, t_off=t_off)
    rcache = oracle_encode(k, v, k_bits, k_signed, v_bits, t_cap=t_cap, t_off=t_off)
    g = cache_to_numpy(gcache)
    cap = T if t_cap is None else t_cap
    rows = None
    if cap != T or t_off:
        rows = (np.arange(B * H)[:, None] * cap + t_off + np.arange(T)[None, :]).reshape(-1)
    n_exc = compare_encoded(g, rcache, D, v_bits, v_input=to_oracle(v).reshape(-1, D), rows=rows)
    # decode the oracle's bytes (tokens [t_off, t_off+T) are what we wrote;
    # decode reads tokens [0, T_dec) with T_dec = t_off + T)
    Td = t_off + T
    inexact = 0
    dev = cache_from_numpy(rcache)
    for dt, odt in ((torch.float32, oracle.F32), (torch.bfloat16, oracle.BF16)):
        kg, vg = tq.tq_decode_kv(dev, Td, k_bits, k_signed, v_bits, out_dtype=dt)
        torch.cuda.synchronize()
        kr, vr = oracle.decode_kv(rcache, Td, k_bits, k_signed, v_bits, out_dtype=odt)
        if dt == torch.float32:
            inexact += compare_decoded(kg.cpu().numpy(), kr, "K decode")
            inexact += compare_decoded(vg.cpu().numpy(), vr, "V decode")
        else:
            kf, vf = oracle.decode_kv(rcache, Td, k_bits, k_signed, v_bits, out_dtype=oracle.F32)
            compare_decoded_bf16(kg.cpu().view(torch.int16).numpy().view(np.uint16), kr, kf, "K bf16")
            compare_decoded_bf16(vg.cpu().view(torch.int16).numpy().view(np.uint16), vr, vf, "V bf16")
    return n_exc, inexact


def compare_decoded_bf16(gpu_bits: np.ndarray, ref_bits: np.ndarray, ref_f32: np.ndarray, what: str):
    """bf16 outputs: equal to the oracle's bf16 bits, except where the fp32
    results already differ within the decode tolerance (then one bf16 step)."""
    if np.array_equal(gpu_bits, ref_bits):
        return
    gf = oracle.bf16_bits_to_f32(gpu_bits)
    rbf = oracle.bf16_bits_to_f32(ref_bits)
    nan = np.isnan(rbf)
    assert np.array_equal(np.isnan(gf), nan), what
    inf = np.isinf(rbf)
    assert np.array_equal(gf[inf], rbf[inf]), what
    fin = ~nan & ~inf
    d = np.abs(gf[fin].astype(np.float64) - rbf[fin])
    assert np.all(d <= 2.0 ** -7 * np.abs(ref_f32[fin]) + 1e-30), what
