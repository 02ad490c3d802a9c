"""Pins of the oracle's decode attention over a packed cache (page
"@mlx-bun/inference 0.0.0-stage -> 1.0.0": ops.ts tryDecodePackedKv with
deferV, decodeValuesRotated, unrotateValues; batched-mask.ts, the left-pad
key mask of batched decode).

Pins used:
- a library routine: torch's scaled_dot_product_attention in float64 on the
  eagerly rotated-back values, with the grouped-query head map and the
  left-pad / causal mask written out as a boolean matrix. It pins the score
  scale, the softmax, the head map, the mask and, through the linearity the
  decodeValuesRotated comment states, the deferred inverse rotation;
- closed forms: one valid key gives back that key's value row rotated back
  (scipy's Hadamard matrix, the signs after it); a zero query gives the plain
  mean of the valid rows; a row with no valid key is zero;
- the page's special case: a constant key group decodes to NaN, which makes
  exactly the rows that can see that token NaN.
"""
import numpy as np
import pytest
import scipy.linalg
import torch

RNG = np.random.default_rng(11)


def _cache(oracle_mod, B, Hkv, T, D, kb, ks, vb, t_cap=None, k=None, seed=0):
    rng = np.random.default_rng(seed)
    if k is None:
        k = rng.standard_normal((B, Hkv, T, D)).astype(np.float32)
    v = rng.standard_normal((B, Hkv, T, D)).astype(np.float32)
    return oracle_mod.encode_kv(k, v, kb, ks, vb, t_cap=t_cap if t_cap else T)


def _queries(oracle_mod, B, Hq, Nq, D, seed=1, scale=1.0):
    x = (scale * np.random.default_rng(seed).standard_normal((B, Hq, Nq, D))).astype(np.float32)
    return oracle_mod.f32_to_bf16_bits(x)


def _rotate_back(oracle_mod, rows):
    """Inverse rotation in float64: Hadamard matrix / sqrt(d), then the signs."""
    D = rows.shape[-1]
    Hm = scipy.linalg.hadamard(D).astype(np.float64) / np.sqrt(D)
    return (rows @ Hm.T) * oracle_mod.sign_vector(D).astype(np.float64)


def _decoded(oracle_mod, cache, T, kb, ks, vb):
    """bf16 keys and bf16 rotated values, as float64 [B,H,T,D]."""
    kd, vd = oracle_mod.decode_kv(cache, T, kb, ks, vb, out_dtype=oracle_mod.BF16, rotated_v=True)
    return (oracle_mod.bf16_bits_to_f32(kd).astype(np.float64),
            oracle_mod.bf16_bits_to_f32(vd).astype(np.float64))


def _mask(B, Nq, T, left_pad):
    """[B, Nq, T] validity: left_pad[b] <= t <= T - Nq + n."""
    t = np.arange(T)[None, None, :]
    n = np.arange(Nq)[None, :, None]
    lp = np.zeros(B, np.int64) if left_pad is None else np.asarray(left_pad, np.int64)
    return (t >= lp[:, None, None]) & (t <= T - Nq + n)


@pytest.mark.parametrize("D,kb,ks,vb,Hkv,G,Nq,T,pad", [
    (64, 8, True, 3, 2, 4, 1, 37, None),
    (128, 8, True, 3, 2, 4, 1, 50, [0, 7]),
    (128, 4, False, 2, 1, 8, 3, 41, [5, 0]),
    (256, 5, False, 4, 2, 2, 2, 33, [1, 3]),
    (512, 2, False, 5, 1, 1, 1, 20, None),
    (128, 8, False, 8, 3, 1, 4, 19, [0, 15]),
])
def test_matches_library_sdpa(oracle_mod, D, kb, ks, vb, Hkv, G, Nq, T, pad):
    B, Hq = 2, Hkv * G
    cache = _cache(oracle_mod, B, Hkv, T, D, kb, ks, vb, t_cap=T + 3, seed=D + vb)
    qb = _queries(oracle_mod, B, Hq, Nq, D, seed=D)
    got = oracle_mod.decode_attention(qb, cache, T, kb, ks, vb, left_pad=pad)

    kd, vrot = _decoded(oracle_mod, cache, T, kb, ks, vb)
    v_eager = _rotate_back(oracle_mod, vrot)
    q = torch.from_numpy(oracle_mod.bf16_bits_to_f32(qb).astype(np.float64))
    K = torch.from_numpy(kd).repeat_interleave(G, dim=1)   # head hq reads kv head hq // G
    V = torch.from_numpy(v_eager).repeat_interleave(G, dim=1)
    m = torch.from_numpy(_mask(B, Nq, T, pad))[:, None]     # [B, 1, Nq, T]
    want = torch.nn.functional.scaled_dot_product_attention(q, K, V, attn_mask=m).numpy()
    assert np.allclose(got, want, rtol=1e-11, atol=1e-12)


def test_single_key_gives_its_row_rotated_back(oracle_mod):
    D, T = 128, 1
    cache = _cache(oracle_mod, 1, 1, T, D, 8, True, 3)
    qb = _queries(oracle_mod, 1, 2, 1, D)
    got = oracle_mod.decode_attention(qb, cache, T, 8, True, 3)
    _, vrot = _decoded(oracle_mod, cache, T, 8, True, 3)
    want = _rotate_back(oracle_mod, vrot[0, 0, 0])
    assert np.allclose(got[0, 0, 0], want, rtol=0, atol=1e-14)
    assert np.allclose(got[0, 1, 0], want, rtol=0, atol=1e-14)


@pytest.mark.parametrize("Nq,pad", [(1, [0, 4]), (3, [2, 0])])
def test_zero_query_gives_mean_of_valid_rows(oracle_mod, Nq, pad):
    D, T, B = 64, 23, 2
    cache = _cache(oracle_mod, B, 1, T, D, 4, False, 5)
    qb = np.zeros((B, 1, Nq, D), np.uint16)  # +0.0 in bf16
    got = oracle_mod.decode_attention(qb, cache, T, 4, False, 5, left_pad=pad)
    _, vrot = _decoded(oracle_mod, cache, T, 4, False, 5)
    for b in range(B):
        for n in range(Nq):
            rows = vrot[b, 0, pad[b]:T - Nq + n + 1]
            want = _rotate_back(oracle_mod, rows.mean(axis=0))
            assert np.allclose(got[b, 0, n], want, rtol=1e-12, atol=1e-14)


def test_row_without_valid_key_is_zero(oracle_mod):
    D, T = 64, 8
    cache = _cache(oracle_mod, 2, 1, T, D, 8, True, 2)
    qb = _queries(oracle_mod, 2, 1, 2, D)
    got = oracle_mod.decode_attention(qb, cache, T, 8, True, 2, left_pad=[7, 8])
    # batch 0: query 0 sits at position 6 < pad 7 (no key), query 1 at 7 sees key 7
    assert np.all(got[0, 0, 0] == 0) and np.any(got[0, 0, 1] != 0)
    assert np.all(got[1] == 0)


def test_constant_key_group_poisons_exactly_the_rows_that_see_it(oracle_mod):
    D, T, B, Hkv, G, Nq = 64, 16, 2, 2, 2, 2
    k = np.random.default_rng(3).standard_normal((B, Hkv, T, D)).astype(np.float32)
    k[0, 0, 5, :32] = 0.5  # decodes to NaN (scale 0, zero point +Inf)
    cache = _cache(oracle_mod, B, Hkv, T, D, 8, True, 3, k=k)
    qb = _queries(oracle_mod, B, Hkv * G, Nq, D)
    got = oracle_mod.decode_attention(qb, cache, T, 8, True, 3, left_pad=[0, 0])
    nan_rows = np.isnan(got).any(axis=-1)
    assert np.all(np.isnan(got[nan_rows]))
    want = np.zeros_like(nan_rows)
    want[0, 0:G, :] = True  # kv head 0 of batch 0, both query tokens see token 5
    assert np.array_equal(nan_rows, want)
    got_pad = oracle_mod.decode_attention(qb, cache, T, 8, True, 3, left_pad=[6, 0])
    assert np.all(np.isfinite(got_pad))  # the pad hides token 5


def test_dominant_key(oracle_mod):
    """A query along one key with a large scale puts (almost) all weight on it."""
    D, T = 128, 12
    cache = _cache(oracle_mod, 1, 1, T, D, 8, True, 4)
    kd, vrot = _decoded(oracle_mod, cache, T, 8, True, 4)
    qv = oracle_mod.f32_to_bf16_bits((kd[0, 0, 9] * 4.0).astype(np.float32))[None, None, None]
    got = oracle_mod.decode_attention(qv, cache, T, 8, True, 4, scale=1.0)
    want = _rotate_back(oracle_mod, vrot[0, 0, 9])
    assert np.allclose(got[0, 0, 0], want, rtol=0, atol=1e-9)
