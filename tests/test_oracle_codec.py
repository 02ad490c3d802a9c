"""Pins of the oracle's key and value codec (page "@mlx-bun/inference
0.0.0-stage -> 1.0.0", file package/src/kernels/turboquant/ops.ts: encodeKeys,
decodeKeys, encodeValues, dequantScaled, decodeValues, decodeValuesRotated,
unrotateValues) and of its whole-tensor cache addressing.

Pins used:
- the page's stated special case: a constant 32-group of keys gives scale
  exactly 0 and a zero point of +Inf in fp16 (ops.ts header comment);
- closed forms: integer ramps whose codes follow by hand; one-hot rotated
  inputs whose Lloyd-Max indices follow from the table alone;
- error bounds of affine quantisation (half a step, one step at the clipped
  ends) and the range the codes must span;
- the distortion of each table for the RMS-normalised coordinate of a
  Gaussian row, computed by quadrature, which the value round trip must
  reproduce;
- invariants: groups never mix tokens, a token-at-a-time encode equals one
  whole encode byte for byte, bf16 input equals its exact fp32 upcast.
"""
import math

import numpy as np
import pytest
import scipy.linalg

from tests.test_oracle_tables import gaussian_mse

RNG = np.random.default_rng(7)
KEY_MODES = [(2, False), (4, False), (5, False), (8, False), (8, True)]


def _kmax(bits, signed):
    return (1 << (bits - 1)) - 1 if signed else (1 << bits) - 1


def _codes_as_int(codes, signed):
    return codes.view(np.int8).astype(np.int64) if signed else codes.astype(np.int64)


# ---- keys -----------------------------------------------------------------------
@pytest.mark.parametrize("bits,signed", KEY_MODES)
@pytest.mark.parametrize("value", [0.5, -0.5, 3.0])
def test_constant_key_group_gives_zero_scale_and_infinite_zero(oracle_mod, bits, signed, value):
    x = np.full((1, 64), value, np.float32)
    x[0, 32:] = RNG.standard_normal(32)
    codes, sc, zr = oracle_mod.encode_keys(x, bits, signed)
    assert sc[0, 0] == 0x0000
    assert zr[0, 0] == (0x7C00 if value > 0 else 0xFC00)  # +Inf / -Inf in fp16
    assert np.all(codes[0, :32] == 0)
    dec = oracle_mod.decode_keys(codes, sc, zr, signed)
    # (q + Inf) * 0 is NaN for the whole constant group, the other group is finite
    assert np.all(np.isnan(dec[0, :32])) and np.all(np.isfinite(dec[0, 32:]))


def _f16_nan(h):
    return (int(h) & 0x7C00) == 0x7C00 and (int(h) & 0x03FF) != 0


# ---- keys and values with Inf / NaN: the IEEE special cases of the page's formulas ----
@pytest.mark.parametrize("bits,signed", KEY_MODES)
@pytest.mark.parametrize("pos", [0, 17, 31])
def test_key_group_with_nan(oracle_mod, bits, signed, pos):
    """A NaN anywhere in a group (also first, where a plain < scan would keep
    it, and last) makes min and max NaN: scale, zero point and every quotient
    are NaN and every code converts to 0; the other group is untouched."""
    x = RNG.standard_normal((1, 64)).astype(np.float32)
    c0, s0, z0 = oracle_mod.encode_keys(x, bits, signed)
    x[0, pos] = np.nan
    codes, sc, zr = oracle_mod.encode_keys(x, bits, signed)
    assert np.all(codes[0, :32] == 0)
    assert _f16_nan(sc[0, 0]) and _f16_nan(zr[0, 0])
    assert np.array_equal(codes[0, 32:], c0[0, 32:]) and sc[0, 1] == s0[0, 1] and zr[0, 1] == z0[0, 1]
    dec = oracle_mod.decode_keys(codes, sc, zr, signed)
    assert np.all(np.isnan(dec[0, :32])) and np.all(np.isfinite(dec[0, 32:]))


@pytest.mark.parametrize("bits,signed", KEY_MODES)
@pytest.mark.parametrize("lo", [-1.0, 0.5])
def test_key_group_with_positive_inf(oracle_mod, bits, signed, lo):
    """max = +Inf, min finite: range and scale are +Inf, scale + eps = Inf.
    Unsigned: zero point round(min / Inf) = a zero with min's sign; signed:
    (Inf + min) / (2 Inf) = NaN. Every finite x gives x / Inf = +-0, Inf gives
    NaN, so every code is 0 either way; the decode (0 + zero) * Inf is NaN."""
    x = np.linspace(lo, 1.0, 32, dtype=np.float32)[None]
    x[0, 5] = np.inf
    codes, sc, zr = oracle_mod.encode_keys(x, bits, signed)
    assert sc[0, 0] == 0x7C00
    if signed:
        assert _f16_nan(zr[0, 0])
    else:
        assert zr[0, 0] == (0x8000 if lo < 0 else 0x0000)
    assert np.all(codes == 0)
    assert np.all(np.isnan(oracle_mod.decode_keys(codes, sc, zr, signed)))


@pytest.mark.parametrize("bits,signed", KEY_MODES)
def test_key_group_with_both_infinities_or_overflowing_range(oracle_mod, bits, signed):
    """-Inf and +Inf: range +Inf, and the zero point's numerator (-Inf, or
    -Inf + Inf) makes it NaN. A finite group +-3e38 overflows the range to
    +Inf: the signed zero point is round(0 / Inf) = 0, the unsigned one
    round(-3e38 / Inf) = -0; all codes 0."""
    x = np.zeros((2, 32), np.float32)
    x[0] = np.linspace(-1, 1, 32)
    x[0, 3], x[0, 20] = np.inf, -np.inf
    x[1, 0::2], x[1, 1::2] = 3e38, -3e38
    codes, sc, zr = oracle_mod.encode_keys(x, bits, signed)
    assert sc[0, 0] == 0x7C00 and _f16_nan(zr[0, 0])
    assert sc[1, 0] == 0x7C00 and zr[1, 0] == (0x0000 if signed else 0x8000)
    assert np.all(codes == 0)


@pytest.mark.parametrize("d", [64, 128, 256, 512])
@pytest.mark.parametrize("bits", [2, 3, 5, 8])
def test_value_row_with_inf_or_nan(oracle_mod, d, bits):
    """One Inf (or NaN) in a value row reaches every coordinate of the
    normalised Hadamard transform, so every group's RMS is Inf (NaN), every
    normalised value Inf / Inf (NaN / NaN) = NaN, and searchsorted counts no
    boundary: all indices 0, every scale +Inf (NaN)."""
    x = RNG.standard_normal((3, d)).astype(np.float32)
    x[0, 3] = np.inf
    x[1, d - 1] = np.nan
    x[2, 11] = -np.inf
    idx, sc = oracle_mod.encode_values(x, bits)
    assert np.all(idx == 0)
    assert np.all(sc[0] == 0x7C00) and np.all(sc[2] == 0x7C00)
    assert all(_f16_nan(h) for h in sc[1])


@pytest.mark.parametrize("bits", [2, 3, 4, 5, 8])
def test_value_row_whose_sum_of_squares_overflows(oracle_mod, bits):
    """One element 1e38 in a row of 128: every rotated coordinate is finite
    (+-1e38 / sqrt(128)), but 32 squares of ~8.8e36 overflow, so the RMS is
    +Inf, every normalised value y / Inf is a signed zero and every index is
    count(boundaries < 0) (a boundary equal to 0 is not below -0 or +0)."""
    x = np.zeros((1, 128), np.float32)
    x[0, 7] = 1e38
    _, b = oracle_mod.lloyd_max(bits)
    idx, sc = oracle_mod.encode_values(x, bits)
    assert np.all(sc == 0x7C00)
    assert np.all(idx == np.count_nonzero(b < 0.0))


def test_unsigned_ramp_closed_form(oracle_mod):
    # x_i = i on one group, 5 bits: scale = 31/31 = 1, scale+eps rounds to 1 in
    # fp32, zero point round(0/1) = 0, codes = i exactly
    x = np.arange(32, dtype=np.float32)[None]
    codes, sc, zr = oracle_mod.encode_keys(x, 5, False)
    assert np.array_equal(codes[0], np.arange(32))
    assert sc[0, 0] == 0x3C00 and zr[0, 0] == 0x0000
    assert np.array_equal(oracle_mod.decode_keys(codes, sc, zr, False)[0], x[0])


def test_signed_ramp_closed_form(oracle_mod):
    # x_i = i - 15.5: symmetric, zero point 0, scale 31/254, codes round(254 (i-15.5)/31)
    x = (np.arange(32, dtype=np.float32) - np.float32(15.5))[None]
    codes, sc, zr = oracle_mod.encode_keys(x, 8, True)
    exact = 254.0 * (np.arange(32) - 15.5) / 31.0
    assert np.min(np.abs(exact - np.floor(exact) - 0.5)) > 1e-3  # no ties
    assert np.array_equal(codes[0].view(np.int8).astype(np.int64), np.rint(exact).astype(np.int64))
    assert codes[0].view(np.int8).min() == -127 and codes[0].view(np.int8).max() == 127
    assert zr[0, 0] == 0x0000
    assert sc[0, 0] == np.float16(31.0 / 254.0).view(np.uint16)


def _key_inputs():
    return [
        RNG.standard_normal((256, 128)).astype(np.float32),
        RNG.uniform(-3, 7, (128, 128)).astype(np.float32),
        (RNG.standard_normal((128, 128)) * np.where(RNG.random((128, 128)) < 0.01, 10, 1)).astype(np.float32),
        (RNG.standard_normal((64, 64)) * 1e-3 + 5.0).astype(np.float32),
    ]


@pytest.mark.parametrize("bits,signed", KEY_MODES)
def test_key_roundtrip_error_bound_and_range(oracle_mod, bits, signed):
    M = _kmax(bits, signed)
    lo, hi = (-M, M) if signed else (0, M)
    for x in _key_inputs():
        codes, sc, zr = oracle_mod.encode_keys(x, bits, signed)
        q = _codes_as_int(codes, signed)
        assert q.min() >= lo and q.max() <= hi
        s16 = sc.view(np.float16).astype(np.float64)
        z16 = zr.view(np.float16).astype(np.float64)
        dec = oracle_mod.decode_keys(codes, sc, zr, signed).astype(np.float64)
        G = x.shape[1] // 32
        xg = x.reshape(x.shape[0], G, 32).astype(np.float64)
        qg = q.reshape(x.shape[0], G, 32)
        err = np.abs(dec.reshape(xg.shape) - xg)
        rng = xg.max(-1) - xg.min(-1)
        s = rng / (2 * M if signed else M)
        # A zero point beyond the fp16 range becomes +-Inf, as it does for a
        # constant group: narrow groups far from 0 (the last input) hit this
        # at 8 bits. Those groups decode to non-finite values; the rest of the
        # bound applies to groups with a finite zero point.
        zp_est = (xg.min(-1) if not signed else (xg.max(-1) + xg.min(-1)) / 2) / s
        over = ~np.isfinite(z16)
        assert np.all(np.abs(zp_est[over]) > 65000)
        assert np.all(np.isfinite(z16[np.abs(zp_est) < 65000]))
        assert np.all(~np.isfinite(dec.reshape(xg.shape)[over]))
        if bits < 8:
            assert not over.any()
        keep = ~over
        err, qg, s16, z16, s = err[keep], qg[keep], s16[keep], z16[keep], s[keep]
        # the quantisation step is the range over the number of levels
        assert np.allclose(s16, s, rtol=2.0 ** -10, atol=1e-7)
        # half a step inside the range, one step where the clip acts, plus the
        # fp16 rounding of scale and zero point (a zero point above 2048 is
        # stored to within half an fp16 ulp), and eps, which the encoder adds
        # to the scale but the decoder does not
        q_plus_z = np.abs(qg + z16[..., None])
        zp_half_ulp = np.spacing(np.abs(z16).astype(np.float16)).astype(np.float64) / 2
        bound = (1.01 * s16[..., None]
                 + (q_plus_z + zp_half_ulp[..., None]) * (np.abs(s16 - s) + 1e-8)[..., None] * 1.01
                 + (zp_half_ulp * s16)[..., None] + 1e-6)
        assert np.all(err <= bound)
        # the codes span the whole level range in every group
        assert np.all(qg.min(-1) <= lo + 1) and np.all(qg.max(-1) >= hi - 1)


@pytest.mark.parametrize("bits,signed", KEY_MODES)
def test_key_groups_are_independent(oracle_mod, bits, signed):
    x = RNG.standard_normal((8, 128)).astype(np.float32)
    full = oracle_mod.encode_keys(x, bits, signed)
    for g in range(4):
        part = oracle_mod.encode_keys(np.ascontiguousarray(x[:, 32 * g:32 * g + 32]), bits, signed)
        assert np.array_equal(part[0], full[0][:, 32 * g:32 * g + 32])
        assert np.array_equal(part[1][:, 0], full[1][:, g]) and np.array_equal(part[2][:, 0], full[2][:, g])


# ---- values ---------------------------------------------------------------------
@pytest.mark.parametrize("d", [64, 128, 256, 512])
@pytest.mark.parametrize("bits", [2, 3, 4, 5, 8])
def test_value_one_hot_rotated_closed_form(oracle_mod, d, bits):
    """v = signs * H[:, j] rotates to sqrt(d) e_j exactly. Group j//32 then has
    RMS sqrt(d/32), so u_j = sqrt(32) (above every boundary) and every other
    coordinate is 0; all other groups are zero (scale 0, u = 0)."""
    H = scipy.linalg.hadamard(d)
    s = oracle_mod.sign_vector(d).astype(np.float32)
    _, bnd = oracle_mod.lloyd_max(bits)
    n_below_zero = int((bnd < 0).sum())
    for j in (0, 5, d // 2 + 3, d - 1):
        v = (s * H[:, j].astype(np.float32))[None]
        idx, sc = oracle_mod.encode_values(v, bits)
        expect = np.full(d, n_below_zero, np.int64)
        expect[j] = 2 ** bits - 1
        assert np.array_equal(idx[0].astype(np.int64), expect)
        r = np.float32(np.float32(d) * np.float32(1.0 / math.sqrt(d)))
        rms = np.float32(np.sqrt(np.float32(r * r) / np.float32(32)))
        exp_sc = np.zeros(d // 32, np.uint16)
        exp_sc[j // 32] = np.float16(rms).view(np.uint16)
        assert np.array_equal(sc[0], exp_sc)


@pytest.mark.parametrize("d", [64, 128, 256, 512])
@pytest.mark.parametrize("bits", [2, 3, 5, 8])
def test_value_decode_constant_index_closed_form(oracle_mod, d, bits):
    """All indices k with scale 1: the rotated vector is c_k * ones, whose
    inverse rotation is signs * c_k * sqrt(d) e_0."""
    cent, _ = oracle_mod.lloyd_max(bits)
    s = oracle_mod.sign_vector(d).astype(np.float64)
    for k in (0, 2 ** bits - 1, 2 ** (bits - 1)):
        idx = np.full((1, d), k, np.uint8)
        sc = np.full((1, d // 32), 0x3C00, np.uint16)
        out = oracle_mod.decode_values(idx, sc, bits)[0].astype(np.float64)
        expect = np.zeros(d)
        expect[0] = s[0] * float(cent[k]) * math.sqrt(d)
        assert np.allclose(out, expect, atol=1e-6 * abs(expect[0]) + 1e-7)
        rot = oracle_mod.decode_values(idx, sc, bits, rotated=True)[0]
        assert np.all(rot == cent[k])


def rms_normalised_distortion(cent, bnd, n=32):
    """E[(u - Q(u))^2] for u = one coordinate of an iid Gaussian n-vector
    divided by the vector's RMS: u is then a coordinate of a uniform point on
    the sphere of radius sqrt(n), with density proportional to
    (1 - u^2/n)^((n-3)/2) on |u| < sqrt(n)."""
    from scipy import integrate

    R = math.sqrt(n)
    f = lambda u: (1 - u * u / n) ** ((n - 3) / 2)
    Z = integrate.quad(f, -R, R)[0]
    edges = [-R] + [float(b) for b in bnd] + [R]
    total = 0.0
    for i, c in enumerate(cent):
        a, b = max(edges[i], -R), min(edges[i + 1], R)
        if a < b:
            total += integrate.quad(lambda u: (u - float(c)) ** 2 * f(u), a, b, epsabs=1e-13)[0]
    return total / Z


@pytest.mark.parametrize("bits", [2, 3, 4, 5, 8])
def test_value_distortion_matches_closed_form(oracle_mod, bits):
    """The rotation keeps iid N(0,1) rows iid N(0,1) and the norm of a Gaussian
    vector is independent of its direction, so the expected relative round-trip
    error equals the quantiser's distortion for the RMS-normalised coordinate
    (computed above by quadrature). 2^19 coordinates give < 1% standard error;
    fp16 scale rounding adds < 0.2% at 8 bits."""
    c, b = oracle_mod.lloyd_max(bits)
    D = rms_normalised_distortion(c, b)
    # normalising by the group's own RMS lowers the distortion a few percent
    # below the N(0,1) figure of the same table
    assert D < gaussian_mse(c, b)
    x = RNG.standard_normal((4096, 128)).astype(np.float32)
    idx, sc = oracle_mod.encode_values(x, bits)
    assert idx.max() < 2 ** bits
    y = oracle_mod.decode_values(idx, sc, bits).astype(np.float64)
    rel = np.sum((y - x) ** 2) / np.sum(x.astype(np.float64) ** 2)
    assert abs(rel / D - 1.0) < 0.025, (rel, D)


@pytest.mark.parametrize("d", [64, 256])
def test_value_scale_is_group_rms_of_rotation(oracle_mod, d):
    x = RNG.standard_normal((32, d)).astype(np.float32)
    idx, sc = oracle_mod.encode_values(x, 4)
    y = oracle_mod.fwht(x, encode=True).astype(np.float64).reshape(32, d // 32, 32)
    rms = np.sqrt((y ** 2).mean(-1))
    assert np.allclose(sc.view(np.float16).astype(np.float64), rms, rtol=2.0 ** -11)


def test_unrotate_inverts_rotation(oracle_mod):
    x = RNG.standard_normal((16, 128)).astype(np.float32)
    y = oracle_mod.fwht(x, encode=True)
    assert np.max(np.abs(oracle_mod.unrotate(y) - x)) < 1e-5


def test_deferred_decode_matches_eager(oracle_mod):
    """Unrotating the rotated-domain decode gives the eager decode (the page
    notes the two are both valid decodes, equal up to rounding)."""
    x = RNG.standard_normal((64, 128)).astype(np.float32)
    idx, sc = oracle_mod.encode_values(x, 3)
    eager = oracle_mod.decode_values(idx, sc, 3)
    deferred = oracle_mod.unrotate(oracle_mod.decode_values(idx, sc, 3, rotated=True))
    assert np.allclose(eager, deferred, rtol=1e-6, atol=1e-6)


# ---- whole tensors -----------------------------------------------------------------
def _bf16_bits(x):
    import torch

    return torch.from_numpy(np.ascontiguousarray(x, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


@pytest.mark.parametrize("bits,signed", KEY_MODES)
def test_tensor_encode_matches_rows(oracle_mod, bits, signed):
    B, H, T, D = 2, 3, 5, 128
    k = RNG.standard_normal((B, H, T, D)).astype(np.float32)
    v = RNG.standard_normal((B, H, T, D)).astype(np.float32)
    cache = oracle_mod.encode_kv(k, v, bits, signed, 3)
    kc, ks, kz = oracle_mod.encode_keys(k, bits, signed)
    vi, vs = oracle_mod.encode_values(v, 3)
    assert np.array_equal(cache["k_codes"], oracle_mod.pack_bits(kc, bits))
    assert np.array_equal(cache["k_scales"], ks) and np.array_equal(cache["k_zeros"], kz)
    assert np.array_equal(cache["v_codes"], oracle_mod.pack_bits(vi, 3))
    assert np.array_equal(cache["v_scales"], vs)
    kd, vd = oracle_mod.decode_kv(cache, T, bits, signed, 3)
    assert np.array_equal(kd, oracle_mod.decode_keys(kc, ks, kz, signed))
    assert np.array_equal(vd, oracle_mod.decode_values(vi, vs, 3))


def test_bf16_input_equals_fp32_upcast(oracle_mod):
    x = RNG.standard_normal((1, 2, 7, 64)).astype(np.float32)
    xb = _bf16_bits(x)
    up = oracle_mod.bf16_bits_to_f32(xb)
    a = oracle_mod.encode_kv(xb, xb, 8, True, 4)
    b = oracle_mod.encode_kv(up, up, 8, True, 4)
    for key in a:
        assert np.array_equal(a[key], b[key])
    ko, vo = oracle_mod.decode_kv(a, 7, 8, True, 4, out_dtype=oracle_mod.BF16)
    kf, vf = oracle_mod.decode_kv(a, 7, 8, True, 4)
    assert np.array_equal(ko, _bf16_bits(kf)) and np.array_equal(vo, _bf16_bits(vf))


def test_token_appends_equal_one_encode(oracle_mod):
    """Groups run along head_dim only, so encoding T tokens one at a time at
    increasing offsets writes the same bytes as one T-token encode; bytes
    outside the written token range are left untouched."""
    B, H, T, D, cap = 2, 2, 9, 64, 13
    k = RNG.standard_normal((B, H, T, D)).astype(np.float32)
    v = RNG.standard_normal((B, H, T, D)).astype(np.float32)
    whole = oracle_mod.alloc_cache(B, H, cap, D, 8, 3)
    for a in whole.values():
        a.view(np.uint8).fill(0xA5)
    oracle_mod.encode_kv(k, v, 8, True, 3, cache=whole, t_off=2)
    step = oracle_mod.alloc_cache(B, H, cap, D, 8, 3)
    for a in step.values():
        a.view(np.uint8).fill(0xA5)
    for t in range(T):
        oracle_mod.encode_kv(np.ascontiguousarray(k[:, :, t:t + 1]), np.ascontiguousarray(v[:, :, t:t + 1]),
                             8, True, 3, cache=step, t_off=2 + t)
    for key in whole:
        assert np.array_equal(whole[key], step[key])
        untouched = np.concatenate([whole[key][:, :, :2], whole[key][:, :, 2 + T:]], axis=2)
        assert np.all(untouched.view(np.uint8) == 0xA5)
    ref = oracle_mod.encode_kv(k, v, 8, True, 3)
    for key in whole:
        assert np.array_equal(whole[key][:, :, 2:2 + T], ref[key])


def test_oracle_argument_errors(oracle_mod):
    L = oracle_mod.lib()
    k = np.zeros((1, 1, 2, 96), np.float32)
    buf = np.zeros(4096, np.uint8)
    p = buf.ctypes.data
    assert L.oracle_encode_kv(k.ctypes.data, k.ctypes.data, 0, 1, 1, 2, 96, 8, 1, 3, p, p, p, p, p, 2, 0) == 2
    assert L.oracle_encode_kv(k.ctypes.data, k.ctypes.data, 0, 1, 1, 2, 64, 8, 1, 6, p, p, p, p, p, 2, 0) == 3
    assert L.oracle_encode_kv(k.ctypes.data, k.ctypes.data, 0, 1, 1, 2, 64, 4, 1, 3, p, p, p, p, p, 2, 0) == 3
    assert L.oracle_encode_kv(k.ctypes.data, k.ctypes.data, 0, 1, 1, 2, 64, 3, 0, 3, p, p, p, p, p, 2, 0) == 3
    assert L.oracle_encode_kv(k.ctypes.data, k.ctypes.data, 0, 1, 1, 2, 64, 8, 1, 3, p, p, p, p, p, 2, 1) == 1
    assert L.oracle_encode_kv(k.ctypes.data, k.ctypes.data, 7, 1, 1, 2, 64, 8, 1, 3, p, p, p, p, p, 2, 0) == 5
