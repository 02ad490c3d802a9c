"""Pins of the oracle's primitives against library routines, closed forms,
brute force and hand-evaluated page formulas.

- fp16 / bf16 casts and round-half-even: numpy's IEEE float16 cast, torch's
  bfloat16 cast, numpy.rint.
- fwht (page "@mlx-bun/inference 0.0.0-stage -> 1.0.0", ops.ts, fwht): the
  Sylvester Hadamard matrix of scipy.linalg.hadamard in float64, one-hot
  inputs (exact), the d=2 textbook case, self-inverse and Parseval.
- searchsorted (ops.ts, searchsorted): numpy.searchsorted(side="left"), which
  returns the number of boundaries strictly below x.
- packBits / unpackBits (ops.ts, bit packing): the per-width byte formulas of
  pack2bit, pack3bit, pack4bit and pack5bit, evaluated independently here, the
  hand-evaluated bytes in tests/golden/pack_examples.txt, and brute force.
- packedDim (ops.ts, packedDim): values and the misalignment error.
"""
import os

import numpy as np
import pytest
import scipy.linalg
import torch

RNG = np.random.default_rng(20260)


# ---- conversions ---------------------------------------------------------------
def _interesting_floats():
    parts = [
        RNG.standard_normal(100000).astype(np.float32),
        (RNG.choice([-1, 1], 100000) * 10.0 ** RNG.uniform(-9, 6, 100000)).astype(np.float32),
        np.array([0.0, -0.0, np.inf, -np.inf, 65504, 65519.996, 65520, 65536, 1e9, -65520,
                  2.0 ** -14, 2.0 ** -24, 2.0 ** -25, 2.0 ** -25 * 1.0000001, 2.0 ** -26,
                  6.0e-8, 5.9604645e-08, 1e-45, 3.0e-38, 5e7, -5e7], np.float32),
    ]
    # exact fp16 rounding ties: midpoints between consecutive fp16 values
    h = np.arange(0, 0x7BFF, 7, dtype=np.uint16)
    lo = h.view(np.float16).astype(np.float32)
    hi = (h + 1).view(np.float16).astype(np.float32)
    mids = ((lo.astype(np.float64) + hi.astype(np.float64)) / 2).astype(np.float32)
    parts += [mids, -mids]
    return np.concatenate(parts)


def test_f32_to_f16_matches_numpy(oracle_mod):
    x = _interesting_floats()
    ours = oracle_mod.f32_to_f16_bits(x)
    with np.errstate(over="ignore"):
        ref = x.astype(np.float16).view(np.uint16)
    assert np.array_equal(ours, ref)


def test_f32_to_f16_nan(oracle_mod):
    h = oracle_mod.f32_to_f16_bits(np.array([np.nan, -np.nan], np.float32))
    assert np.all(np.isnan(h.view(np.float16)))


def test_f16_to_f32_all_patterns(oracle_mod):
    h = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ours = oracle_mod.f16_bits_to_f32(h)
    ref = h.view(np.float16).astype(np.float32)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan].view(np.uint32), ref[~nan].view(np.uint32))


def test_f32_to_bf16_matches_torch(oracle_mod):
    x = _interesting_floats()
    # bf16 ties: low 16 bits exactly 0x8000
    ties = (RNG.integers(0, 2 ** 15, 20000, dtype=np.uint32) << 16 | 0x8000).view(np.float32)
    x = np.concatenate([x, ties, -ties])
    x = x[np.isfinite(x)]
    ours = oracle_mod.f32_to_bf16_bits(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)


def test_round_half_even(oracle_mod):
    vals = [0.5, 1.5, 2.5, -0.5, -1.5, -2.5, 3.49999, 3.5000002, 1e7 + 0.5, 8388607.5, -0.3]
    vals += list(RNG.uniform(-300, 300, 2000)) + list(np.arange(-20, 20) + 0.5)
    for v in vals:
        v32 = float(np.float32(v))
        assert oracle_mod.round_half_even(v32) == float(np.rint(np.float32(v32)))


# ---- Hadamard / fwht ----------------------------------------------------------
@pytest.mark.parametrize("n", [2, 4, 8, 16, 32, 64, 128, 256, 512])
def test_hadamard_matches_sylvester_matrix(oracle_mod, n):
    x = RNG.standard_normal((64, n)).astype(np.float32)
    ours = oracle_mod.hadamard(x).astype(np.float64)
    H = scipy.linalg.hadamard(n).astype(np.float64)
    ref = x.astype(np.float64) @ H.T / np.sqrt(n)
    err = np.abs(ours - ref).max(axis=1)
    norm = np.linalg.norm(x.astype(np.float64), axis=1)
    # log2(n) rounded adds plus one rounded multiply, each <= 2^-24 relative
    assert np.all(err <= (np.log2(n) + 2) * 2.0 ** -23 * norm)


@pytest.mark.parametrize("n", [2, 8, 64, 128, 256, 512])
def test_hadamard_one_hot_is_exact(oracle_mod, n):
    H = scipy.linalg.hadamard(n)
    c = np.float32(1.0 / np.sqrt(float(n)))
    for j in range(0, n, max(1, n // 16)):
        e = np.zeros(n, np.float32)
        e[j] = 1.0
        ours = oracle_mod.hadamard(e[None])[0]
        assert np.array_equal(ours, H[:, j].astype(np.float32) * c)


def test_hadamard_two_point_textbook(oracle_mod):
    a, b = np.float32(0.75), np.float32(-2.5)
    out = oracle_mod.hadamard(np.array([[a, b]], np.float32))[0]
    r2 = np.float32(1.0 / np.sqrt(2.0))
    assert out[0] == np.float32(np.float32(a + b) * r2) and out[1] == np.float32(np.float32(a - b) * r2)
    assert abs(float(out[0]) - (0.75 - 2.5) / np.sqrt(2)) < 1e-6


@pytest.mark.parametrize("n", [64, 128, 256, 512])
def test_hadamard_self_inverse_and_parseval(oracle_mod, n):
    x = RNG.standard_normal((256, n)).astype(np.float32)
    y = oracle_mod.hadamard(x)
    z = oracle_mod.hadamard(y)
    assert np.max(np.abs(z - x)) < 1e-5
    assert np.allclose(np.linalg.norm(y, axis=1), np.linalg.norm(x, axis=1), rtol=1e-5)
    # the unnormalised transform applied twice is n times the identity
    u = oracle_mod.hadamard(oracle_mod.hadamard(x, normalised=False), normalised=False)
    assert np.allclose(u / n, x, atol=1e-5)


@pytest.mark.parametrize("d", [64, 128, 256, 512])
def test_fwht_encode_decode(oracle_mod, d):
    x = RNG.standard_normal((128, d)).astype(np.float32)
    s = oracle_mod.sign_vector(d).astype(np.float64)
    H = scipy.linalg.hadamard(d).astype(np.float64) / np.sqrt(d)
    enc = oracle_mod.fwht(x, encode=True)
    # encode = H (s * x): signs first, then the transform
    assert np.max(np.abs(enc - (x.astype(np.float64) * s) @ H.T)) < 1e-5
    dec = oracle_mod.fwht(enc, encode=False)
    # decode = s * (H y): the transform first, then the signs
    assert np.max(np.abs(dec - s * (enc.astype(np.float64) @ H.T))) < 1e-5
    assert np.max(np.abs(dec - x)) < 1e-5
    with pytest.raises(oracle_mod.OracleError):
        oracle_mod.fwht(np.zeros((1, 96), np.float32), True)


# ---- searchsorted --------------------------------------------------------------
@pytest.mark.parametrize("bits", [2, 3, 4, 5, 8])
def test_searchsorted_matches_numpy(oracle_mod, bits):
    _, b = oracle_mod.lloyd_max(bits)
    x = [RNG.standard_normal(20000).astype(np.float32) * 2, b, np.nextafter(b, np.float32(np.inf)),
         np.nextafter(b, np.float32(-np.inf)), np.array([np.inf, -np.inf, 0.0, -0.0, 100.0, -100.0], np.float32)]
    x = np.concatenate(x).astype(np.float32)
    ours = oracle_mod.searchsorted(b, x)
    ref = np.searchsorted(b, x, side="left")
    assert np.array_equal(ours.astype(np.int64), ref)
    # x equal to a boundary is not counted (strict comparison)
    assert np.array_equal(oracle_mod.searchsorted(b, b).astype(np.int64), np.arange(len(b)))


def test_searchsorted_nan_counts_nothing(oracle_mod):
    _, b = oracle_mod.lloyd_max(4)
    assert oracle_mod.searchsorted(b, np.array([np.nan], np.float32))[0] == 0


# ---- packing ----------------------------------------------------------------------
def _page_pack(codes, bits):
    """The page's per-width byte formulas (pack2bit/3bit/4bit/5bit), evaluated
    independently of the oracle's flat-bitstream loop."""
    v = [int(c) for c in codes]
    out = []
    if bits == 8:
        return bytes(v)
    if bits == 2:
        for i in range(0, len(v), 4):
            a = [x & 3 for x in v[i:i + 4]]
            out.append(a[0] | a[1] << 2 | a[2] << 4 | a[3] << 6)
    elif bits == 4:
        for i in range(0, len(v), 2):
            out.append((v[i] & 15) | (v[i + 1] & 15) << 4)
    elif bits == 3:
        for i in range(0, len(v), 8):
            m = [x & 7 for x in v[i:i + 8]]
            b0 = m[0] | m[1] << 3 | m[2] << 6
            b1 = m[2] >> 2 | m[3] << 1 | m[4] << 4 | m[5] << 7
            b2 = m[5] >> 1 | m[6] << 2 | m[7] << 5
            out += [b0 & 255, b1 & 255, b2 & 255]
    elif bits == 5:
        for i in range(0, len(v), 8):
            lanes = v[i:i + 8]
            for byte in range(5):
                val = 0
                for lane in range(8):
                    lo, hi = max(5 * lane, 8 * byte), min(5 * lane + 5, 8 * byte + 8)
                    if lo < hi:
                        w = hi - lo
                        val |= ((lanes[lane] >> (lo - 5 * lane)) & ((1 << w) - 1)) << (lo - 8 * byte)
                out.append(val)
    return bytes(out)


def test_pack_golden_examples(oracle_mod):
    path = os.path.join(os.path.dirname(__file__), "golden", "pack_examples.txt")
    n = 0
    for line in open(path):
        if line.startswith("#") or not line.strip():
            continue
        bits, codes, packed = [p.strip() for p in line.split("|")]
        bits = int(bits)
        codes = np.array([int(t) for t in codes.split()], np.uint8)
        packed = bytes(int(t, 16) for t in packed.split())
        assert oracle_mod.pack_bits(codes, bits).tobytes() == packed
        assert _page_pack(codes, bits) == packed
        assert np.array_equal(oracle_mod.unpack_bits(np.frombuffer(packed, np.uint8), bits, len(codes)), codes)
        n += 1
    assert n == 9


@pytest.mark.parametrize("bits", [2, 3, 4, 5, 8])
def test_pack_matches_page_formulas(oracle_mod, bits):
    codes = RNG.integers(0, 2 ** bits, (64, 128), dtype=np.uint8)
    ours = oracle_mod.pack_bits(codes, bits)
    assert ours.shape == (64, 128 * bits // 8)
    for r in range(codes.shape[0]):
        assert ours[r].tobytes() == _page_pack(codes[r], bits)


@pytest.mark.parametrize("bits", [2, 3, 4, 5, 8])
def test_pack_roundtrip_brute_force(oracle_mod, bits):
    # every value at every lane position of an 8-code block
    for pos in range(8):
        for val in range(2 ** bits):
            codes = np.zeros(8, np.uint8)
            codes[pos] = val
            p = oracle_mod.pack_bits(codes, bits)
            assert np.array_equal(oracle_mod.unpack_bits(p, bits, 8), codes)
            # only the bits of this lane are set
            total = int.from_bytes(p.tobytes(), "little")
            assert total == val << (pos * bits)


def test_packed_dim(oracle_mod):
    for d in (64, 128, 256, 512):
        for b in (2, 3, 4, 5, 8):
            assert oracle_mod.packed_dim(d, b) == d * b // 8
    assert oracle_mod.packed_dim(512, 5) == 320 and oracle_mod.packed_dim(128, 3) == 48
    assert oracle_mod.packed_dim(512, 2) == 128 and oracle_mod.packed_dim(64, 3) == 24
    assert oracle_mod.packed_dim(3, 3) == -1 and oracle_mod.packed_dim(5, 5) == -1
    with pytest.raises(oracle_mod.OracleError):
        oracle_mod.pack_bits(np.zeros(8, np.uint8), 6)
