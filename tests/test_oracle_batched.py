"""Pins of the oracle's batched packed-cache row operations (page
"@mlx-bun/inference 0.0.0-stage -> 1.0.0": batched-quant.ts mergeQuantRows,
extendQuantRows, extractQuantRow, filterQuantRows; batched-mask.ts, the
left-pad convention).

Pins used:
- hand-evaluated pad bookkeeping of the pages' formulas (width = longest
  row, pad = width - length; extend grows existing pads by the batch side's
  pad);
- element-wise index checks written independently of the functions (pad
  columns are zero bytes, real columns are the source bytes shifted right);
- round trips and consistency between the operations (extract undoes merge;
  extending a merged batch by one row equals merging all rows; filter keeps
  rows unchanged);
- the codec and attention oracles: a merged row decodes to the same values
  as the row alone, and attention with the left-pad mask over the merged
  batch equals attention over each row alone, exactly.
"""
import numpy as np
import pytest

from oracle import batched_cache as bc


def _row(oracle_mod, L, seed, H=2, D=64, kb=8, ks=True, vb=3):
    rng = np.random.default_rng(seed)
    k = rng.standard_normal((1, H, L, D)).astype(np.float32)
    v = rng.standard_normal((1, H, L, D)).astype(np.float32)
    return oracle_mod.encode_kv(k, v, kb, ks, vb)


def test_merge_pad_bookkeeping(oracle_mod):
    rows = [_row(oracle_mod, n, i) for i, n in enumerate((3, 5, 2))]
    merged, pads, width = bc.merge_rows(rows)
    assert width == 5 and pads == [2, 0, 3]
    assert merged["k_codes"].shape == (3, 2, 5, 64) and merged["v_codes"].shape == (3, 2, 5, 24)
    # a wider joiner pads the batch side; a narrower one pads itself
    ext, pads2, w2 = bc.extend_rows(merged, pads, _row(oracle_mod, 7, 9))
    assert w2 == 7 and pads2 == [4, 2, 5, 0]
    ext, pads3, w3 = bc.extend_rows(merged, pads, _row(oracle_mod, 4, 10))
    assert w3 == 5 and pads3 == [2, 0, 3, 1]


def test_merge_elementwise(oracle_mod):
    lens = (6, 1, 4)
    rows = [_row(oracle_mod, n, 20 + i) for i, n in enumerate(lens)]
    merged, pads, width = bc.merge_rows(rows)
    for name in bc.BUFFERS:
        m = merged[name]
        for i, n in enumerate(lens):
            for t in range(width):
                if t < width - n:
                    assert np.all(m[i, :, t] == 0)
                else:
                    assert np.array_equal(m[i, :, t], rows[i][name][0, :, t - (width - n)])


def test_extract_undoes_merge(oracle_mod):
    rows = [_row(oracle_mod, n, 30 + i) for i, n in enumerate((9, 4, 9, 1))]
    merged, pads, _ = bc.merge_rows(rows)
    for i, r in enumerate(rows):
        got = bc.extract_row(merged, pads[i], i)
        for name in bc.BUFFERS:
            assert np.array_equal(got[name], r[name]) and got[name].flags["C_CONTIGUOUS"]


@pytest.mark.parametrize("lens", [(3, 8, 5), (8, 3, 2), (4, 4, 9)])
def test_extend_equals_merge(oracle_mod, lens):
    rows = [_row(oracle_mod, n, 40 + i) for i, n in enumerate(lens)]
    head, pads, _ = bc.merge_rows(rows[:-1])
    ext, pads_e, w_e = bc.extend_rows(head, pads, rows[-1])
    full, pads_m, w_m = bc.merge_rows(rows)
    assert w_e == w_m and pads_e == pads_m
    for name in bc.BUFFERS:
        assert np.array_equal(ext[name], full[name])


def test_filter_keeps_rows(oracle_mod):
    rows = [_row(oracle_mod, n, 50 + i) for i, n in enumerate((5, 2, 7, 3))]
    merged, pads, _ = bc.merge_rows(rows)
    keep = [3, 0, 2]
    f = bc.filter_rows(merged, keep)
    for j, i in enumerate(keep):
        for name in bc.BUFFERS:
            assert np.array_equal(f[name][j], merged[name][i])


def test_merged_rows_decode_and_attend_like_the_rows_alone(oracle_mod):
    H, D, G = 2, 64, 2
    lens = (11, 4, 7)
    rows = [_row(oracle_mod, n, 60 + i, H=H, D=D) for i, n in enumerate(lens)]
    merged, pads, width = bc.merge_rows(rows)
    dm_k, dm_v = oracle_mod.decode_kv(merged, width, 8, True, 3)
    rng = np.random.default_rng(5)
    q = oracle_mod.f32_to_bf16_bits(rng.standard_normal((len(lens), H * G, 1, D)).astype(np.float32))
    att = oracle_mod.decode_attention(q, merged, width, 8, True, 3, left_pad=pads)
    for i, n in enumerate(lens):
        rk, rv = oracle_mod.decode_kv(rows[i], n, 8, True, 3)
        assert np.array_equal(dm_k[i, :, pads[i]:], rk[0]) and np.array_equal(dm_v[i, :, pads[i]:], rv[0])
        alone = oracle_mod.decode_attention(q[i:i + 1], rows[i], n, 8, True, 3)
        assert np.array_equal(att[i], alone[0])
