"""GPU parity: the CUDA path (through the C ABI) against the oracle.

Small shapes cover every (head_dim, value bits, key mode, input dtype)
combination with ragged row counts that leave a partial last warp step; the
benchmark workloads run at reduced size element by element, and at full size
on sampled rows; edge cases cover empty inputs, cache offsets and bytes that
must stay untouched, and argument errors.
"""
import numpy as np
import pytest
import torch

import oracle
import turboquant_kv_cache_tq_gb300 as tq
from turboquant_kv_cache_tq_gb300.workloads import WORKLOADS, make_append_steps, make_kv, to_oracle
from tests.gpu_common import (cache_from_numpy, cache_to_numpy, check_roundtrip, compare_decoded,
                              compare_decoded_bf16, compare_encoded, gpu_encode, oracle_encode, require_gpu)

pytestmark = pytest.mark.gpu

KEY_MODES = [(2, False), (4, False), (5, False), (8, False), (8, True)]


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def _rand(shape, dtype, seed, scale=1.0):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(shape, generator=g) * scale
    return x.to(dtype).contiguous()


# ---- every combination, small ragged shapes ---------------------------------------
@pytest.mark.parametrize("D", [64, 128, 256, 512])
@pytest.mark.parametrize("v_bits", [2, 3, 4, 5, 8])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_all_combinations(D, v_bits, dtype):
    T = {64: 37, 128: 29, 256: 13, 512: 7}[D]
    for i, (kb, ks) in enumerate(KEY_MODES):
        k = _rand((2, 3, T, D), dtype, 100 + i + D + v_bits)
        v = _rand((2, 3, T, D), dtype, 200 + i + D + v_bits, scale=2.0)
        check_roundtrip(k, v, kb, ks, v_bits)


# ---- the bulk-copy decode (whole, 16-byte aligned tiles; bf16 outputs) ------------
@pytest.mark.parametrize("D", [64, 128, 256, 512])
@pytest.mark.parametrize("v_bits", [2, 3, 4, 5, 8])
def test_bulk_decode_all_combinations(D, v_bits):
    """Token counts that are whole tiles (multiples of 32 / (D / 32) rows) and
    caches whose rows keep every tile 16-byte aligned take the decode with
    bulk asynchronous copies: every key mode, full and spare capacity, eager
    and rotated values, against the oracle; the device error word stays
    clear."""
    rpw = 32 // (D // 32)
    T = rpw * {64: 7, 128: 9, 256: 5, 512: 6}[D]
    for i, (kb, ks) in enumerate(KEY_MODES):
        k = _rand((2, 3, T, D), torch.bfloat16, 500 + i + D + v_bits)
        v = _rand((2, 3, T, D), torch.bfloat16, 600 + i + D + v_bits, scale=2.0)
        check_roundtrip(k, v, kb, ks, v_bits)
        check_roundtrip(k, v, kb, ks, v_bits, t_cap=T + 2 * rpw)
        ref = oracle_encode(k, v, kb, ks, v_bits, t_cap=T + 2 * rpw)
        dev = cache_from_numpy(ref)
        kg, vg = tq.tq_decode_kv_rotated(dev, T, kb, ks, v_bits, out_dtype=torch.bfloat16)
        torch.cuda.synchronize()
        kr, vr = oracle.decode_kv(ref, T, kb, ks, v_bits, out_dtype=oracle.BF16, rotated_v=True)
        assert np.array_equal(vg.cpu().view(torch.int16).numpy().view(np.uint16), vr)
        assert np.array_equal(kg.cpu().view(torch.int16).numpy().view(np.uint16), kr)
    assert tq.lib().tq_device_status(None) == 0


# ---- workloads at reduced size, element by element --------------------------------
def test_tiny_workload_constant_group():
    w = WORKLOADS["tiny"]
    k, v = make_kv(w)
    for kb, ks in KEY_MODES:
        check_roundtrip(k, v, kb, ks, 3)
    g = cache_to_numpy(gpu_encode(k, v, 8, True, 3))
    # the constant group of K[0,0,0,0:32]: scale 0 and an fp16 +Inf zero point
    assert g["k_scales"][0, 0, 0, 0] == 0x0000 and g["k_zeros"][0, 0, 0, 0] == 0x7C00
    kd, _ = tq.tq_decode_kv(cache_from_numpy(g), w.T, 8, True, 3, out_dtype=torch.float32)
    kd = kd.cpu().numpy()
    assert np.all(np.isnan(kd[0, 0, 0, :32])) and np.isfinite(kd[0, 0, 0, 32:]).all()
    assert np.isfinite(kd.reshape(-1, 64)[1:]).all()


@pytest.mark.parametrize("name,T", [("llama3_8b_layer", 300), ("hd256", 40), ("hd512", 24), ("long_context", 50)])
def test_workload_reduced(name, T):
    w = WORKLOADS[name]
    B = min(w.B, 3)
    k, v = make_kv(w, B=B, T=T)
    for vb in w.v_bits:
        check_roundtrip(k, v, w.k_bits, w.k_signed, vb)
        # a second key mode on the same data
        check_roundtrip(k, v, 4, False, vb)


# ---- full-size workloads on sampled rows --------------------------------------------
def _sample_rows(R, n, seed, per_bh=None):
    rng = np.random.default_rng(seed)
    rows = set(rng.integers(0, R, n).tolist())
    rows |= {0, 1, 2, R - 3, R - 2, R - 1}
    if per_bh:
        rows |= {i * per_bh for i in range(0, R // per_bh, max(1, R // per_bh // 8))}
        rows |= {i * per_bh - 1 for i in range(1, R // per_bh, max(1, R // per_bh // 8))}
    return np.array(sorted(rows))


@pytest.mark.parametrize("name", ["llama3_8b_layer", "hd256", "hd512", "long_context"])
def test_workload_full_size_sampled(name):
    w = WORKLOADS[name]
    k, v = make_kv(w)
    D = w.D
    rows = _sample_rows(w.rows, 1500, w.seed, per_bh=w.T)
    ko = to_oracle(k).reshape(-1, D)[rows].reshape(1, 1, -1, D)
    vo = to_oracle(v).reshape(-1, D)[rows].reshape(1, 1, -1, D)
    for vb in w.v_bits:
        gcache = gpu_encode(k, v, w.k_bits, w.k_signed, vb)
        ref = oracle.encode_kv(ko, vo, w.k_bits, w.k_signed, vb)
        g = {key: val.reshape(-1, val.shape[-1])[rows][None, None] for key, val in cache_to_numpy(gcache).items()}
        compare_encoded(g, ref, D, vb, v_input=vo.reshape(-1, D))
        # decode at full size, compare the sampled rows with the oracle's decode
        kd, vd = tq.tq_decode_kv(gcache, w.T, w.k_bits, w.k_signed, vb, out_dtype=torch.float32)
        torch.cuda.synchronize()
        # the oracle decodes the same packed bytes (a value index may differ
        # from the oracle's encode inside the boundary band)
        kr, vr = oracle.decode_kv(g, len(rows), w.k_bits, w.k_signed, vb)
        sel = torch.from_numpy(rows).cuda()
        compare_decoded(kd.reshape(-1, D)[sel].cpu().numpy(), kr.reshape(-1, D), "K")
        compare_decoded(vd.reshape(-1, D)[sel].cpu().numpy(), vr.reshape(-1, D), "V")
        del kd, vd
        # bf16 outputs, as the bench decodes them
        kb16, vb16 = tq.tq_decode_kv(gcache, w.T, w.k_bits, w.k_signed, vb, out_dtype=torch.bfloat16)
        torch.cuda.synchronize()
        kr16, vr16 = oracle.decode_kv(g, len(rows), w.k_bits, w.k_signed, vb, out_dtype=oracle.BF16)
        _bits = lambda t: t.reshape(-1, D)[sel].cpu().view(torch.int16).numpy().view(np.uint16)
        compare_decoded_bf16(_bits(kb16), kr16.reshape(-1, D), kr.reshape(-1, D), "K bf16")
        compare_decoded_bf16(_bits(vb16), vr16.reshape(-1, D), vr.reshape(-1, D), "V bf16")
        del gcache, kb16, vb16
        torch.cuda.empty_cache()


# ---- launches long enough for the interleaved work order -------------------------------
@pytest.mark.parametrize("D", [64, 128, 256, 512])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_long_launches_sampled(D, dtype):
    """Launches of more than 4 items per warp take the interleaved work order
    (short ones the snake order, which every small test covers). 4 * 9728 *
    rows-per-warp + 1 rows exceed 4 steps per warp at any occupancy (at most
    64 warps per SM on 152 SMs); sampled rows are compared with the oracle,
    and the decode of the whole launch on the same rows."""
    rpw = 32 // (D // 32)
    R = 4 * 152 * 64 * rpw + 1
    H = 4
    T = (R + H - 1) // H
    g = torch.Generator(device="cuda").manual_seed(D + (dtype == torch.float32))
    k = (torch.randn((1, H, T, D), generator=g, device="cuda") * 1.5).to(dtype)
    v = torch.randn((1, H, T, D), generator=g, device="cuda").to(dtype)
    rows = _sample_rows(H * T, 300, D, per_bh=T)
    kr = to_oracle(k.reshape(-1, D)[torch.from_numpy(rows).cuda()].cpu()).reshape(1, 1, -1, D)
    vr = to_oracle(v.reshape(-1, D)[torch.from_numpy(rows).cuda()].cpu()).reshape(1, 1, -1, D)
    for i, vb in enumerate([2, 3, 4, 5, 8]):
        kb, ks = KEY_MODES[(i + D // 64) % len(KEY_MODES)]
        cache = tq.alloc_cache(1, H, T, D, kb, vb)
        tq.tq_encode_kv(k, v, kb, ks, vb, cache)
        torch.cuda.synchronize()
        ref = oracle.encode_kv(kr, vr, kb, ks, vb)
        got = {n: t.reshape(-1, t.shape[-1])[rows][None, None] for n, t in cache_to_numpy(cache).items()}
        compare_encoded(got, ref, D, vb, v_input=vr.reshape(-1, D))
        kd, vd = tq.tq_decode_kv(cache, T, kb, ks, vb, out_dtype=torch.float32)
        torch.cuda.synchronize()
        # the oracle decodes the same packed bytes (a value index may differ
        # from the oracle's encode inside the boundary band)
        kref, vref = oracle.decode_kv(got, len(rows), kb, ks, vb)
        sel = torch.from_numpy(rows).cuda()
        compare_decoded(kd.reshape(-1, D)[sel].cpu().numpy(), kref.reshape(-1, D), "K")
        compare_decoded(vd.reshape(-1, D)[sel].cpu().numpy(), vref.reshape(-1, D), "V")
        del kd, vd
        # bf16 outputs (long launches keep each lane's sign words in registers there)
        kb16, vb16 = tq.tq_decode_kv(cache, T, kb, ks, vb, out_dtype=torch.bfloat16)
        torch.cuda.synchronize()
        kr16, vr16 = oracle.decode_kv(got, len(rows), kb, ks, vb, out_dtype=oracle.BF16)
        _bits = lambda t: t.reshape(-1, D)[sel].cpu().view(torch.int16).numpy().view(np.uint16)
        compare_decoded_bf16(_bits(kb16), kr16.reshape(-1, D), kref.reshape(-1, D), "K bf16")
        compare_decoded_bf16(_bits(vb16), vr16.reshape(-1, D), vref.reshape(-1, D), "V bf16")
        del cache, kb16, vb16
    torch.cuda.empty_cache()


# ---- appends into a preallocated cache ---------------------------------------------
def test_long_context_appends_equal_one_encode():
    """The serving mix: a prefix encode into a cache of capacity T + 64, then
    64 single-token appends at t_off = T + s; the bytes equal one encode of
    all T + 64 tokens and the oracle's bytes for the same tokens."""
    w = WORKLOADS["long_context"]
    B, T = 4, 96
    k, v = make_kv(w, B=B, T=T)
    steps = make_append_steps(w)
    cap = T + len(steps)
    for vb in w.v_bits:
        cache = gpu_encode(k, v, w.k_bits, w.k_signed, vb, t_cap=cap)
        for s, (ks_, vs_) in enumerate(steps):
            tq.tq_encode_kv(ks_[:B].contiguous().cuda(), vs_[:B].contiguous().cuda(), w.k_bits, w.k_signed, vb,
                            cache, t_off=T + s)
        torch.cuda.synchronize()
        kall = torch.cat([k] + [s_[0][:B] for s_ in steps], dim=2).contiguous()
        vall = torch.cat([v] + [s_[1][:B] for s_ in steps], dim=2).contiguous()
        whole = cache_to_numpy(gpu_encode(kall, vall, w.k_bits, w.k_signed, vb))
        got = cache_to_numpy(cache)
        for key in got:
            assert np.array_equal(got[key], whole[key]), key
        ref = oracle_encode(kall, vall, w.k_bits, w.k_signed, vb)
        compare_encoded(got, ref, w.D, vb, v_input=to_oracle(vall).reshape(-1, w.D))


def test_offsets_touch_only_written_tokens():
    k = _rand((2, 2, 9, 128), torch.bfloat16, 5)
    v = _rand((2, 2, 9, 128), torch.bfloat16, 6)
    cache = gpu_encode(k, v, 8, True, 3, t_cap=16, t_off=5, fill=0xA5)
    g = cache_to_numpy(cache)
    ref = oracle_encode(k, v, 8, True, 3, t_cap=16, t_off=5)
    for key in g:
        assert np.all(g[key][:, :, :5].view(np.uint8) == 0xA5), key
        assert np.all(g[key][:, :, 14:].view(np.uint8) == 0xA5), key
        assert np.array_equal(g[key][:, :, 5:14], ref[key][:, :, 5:14]), key
    check_roundtrip(k, v, 5, False, 5, t_cap=12, t_off=3)


def _key_groups(groups, D=64):
    """A [1,1,T,D] fp32 K tensor whose rows are the given 32-element groups."""
    g = np.asarray(groups, np.float32).reshape(-1, D)
    return torch.from_numpy(g.copy()).view(1, 1, -1, D)


def test_key_rounding_ties():
    """Groups whose x / (scale + eps) - zero lands exactly on half-integers:
    the quotient must be the correctly rounded one and round() half to even,
    like the page's."""
    half = np.arange(32, dtype=np.float32) + np.float32(0.5)  # 5-bit: scale 1, zero 0, t = i + 0.5
    sym = np.concatenate([[-127.0, 127.0], np.arange(-15, 15) + 0.5]).astype(np.float32)  # int8: scale 1
    rows = [np.concatenate([half, half[::-1]]), np.concatenate([sym, -sym]),
            np.concatenate([half * 2, half - 16])]
    k = _key_groups(rows)
    v = torch.from_numpy(np.random.default_rng(0).standard_normal(k.shape).astype(np.float32))
    for kb, ks in KEY_MODES:
        check_roundtrip(k, v, kb, ks, 3)


@pytest.mark.parametrize("kb,ks", KEY_MODES)
def test_key_quotient_rounding_stress(kb, ks):
    """Groups on a power-of-two scale whose elements sit on, or one ulp
    beside, half-integer multiples of the scale, and groups whose scale is
    comparable to eps: every code depends on the exact rounding of
    x / (scale + eps) and of the subtraction of the zero point."""
    rng = np.random.default_rng(100 + kb + 10 * ks)
    M = 127 if ks else (1 << kb) - 1
    rows = []
    for g in range(512):
        e = int(rng.integers(-3, 12))
        h = np.float32(2.0 ** e)
        if ks:
            base = rng.integers(-2 * M, 2 * M + 1, 32).astype(np.float32) * np.float32(0.5)
            base[0], base[1] = -M, M
        else:
            base = rng.integers(0, 2 * M + 1, 32).astype(np.float32) * np.float32(0.5)
            base[0], base[1] = 0, M
        x = (base * h).astype(np.float32)
        nudge = rng.integers(-1, 2, 32)
        nudge[:2] = 0
        x = np.where(nudge > 0, np.nextafter(x, np.float32(np.inf)),
                     np.where(nudge < 0, np.nextafter(x, np.float32(-np.inf)), x)).astype(np.float32)
        if g % 8 == 7:  # scale near eps: range ~ M * 1e-8
            x = (rng.standard_normal(32) * M * 1e-8).astype(np.float32)
        rows.append(rng.permutation(x))
    k = _key_groups(np.concatenate(rows).reshape(-1, 64))
    v = torch.from_numpy(np.random.default_rng(3).standard_normal(k.shape).astype(np.float32))
    check_roundtrip(k, v, kb, ks, 3)


def test_key_signed_zero_extremes():
    """Groups whose min or max is +0 or -0: the zero point keeps the sign of
    the first such zero in element order, as the page's scan gives."""
    base = np.abs(np.random.default_rng(1).standard_normal(32)).astype(np.float32) + 0.1
    rows = []
    for first, second in ((0.0, -0.0), (-0.0, 0.0)):
        a = base.copy()
        a[3], a[17] = first, second  # min is a zero
        b = -base.copy()
        b[5], b[29] = first, second  # max is a zero
        rows += [np.concatenate([a, b])]
    rows += [np.concatenate([np.full(32, -0.0, np.float32), np.zeros(32, np.float32)])]
    k = _key_groups(rows)
    v = torch.from_numpy(np.random.default_rng(2).standard_normal(k.shape).astype(np.float32))
    for kb, ks in KEY_MODES:
        check_roundtrip(k, v, kb, ks, 2)


@pytest.mark.parametrize("T", [1, 2, 3, 7, 31, 64, 4097])
def test_row_to_token_mapping(T):
    """Rows map to (b*h, t) by a multiply-shift division by T; odd and
    power-of-two T, with a cache offset, against the oracle."""
    B, H = 3, 2
    k = _rand((B, H, T, 128), torch.bfloat16, 40 + T)
    v = _rand((B, H, T, 128), torch.bfloat16, 41 + T)
    check_roundtrip(k, v, 8, True, 4, t_cap=T + 5, t_off=2)


def test_decode_leaves_output_padding_untouched():
    k = _rand((1, 3, 11, 64), torch.bfloat16, 8)
    v = _rand((1, 3, 11, 64), torch.bfloat16, 9)
    cache = gpu_encode(k, v, 8, True, 2)
    big_k = torch.full((1 * 3 * 11 * 64 + 64,), 7.0, dtype=torch.float32, device="cuda")
    big_v = torch.full_like(big_k, 7.0)
    ko = big_k[:1 * 3 * 11 * 64].view(1, 3, 11, 64)
    vo = big_v[:1 * 3 * 11 * 64].view(1, 3, 11, 64)
    tq.tq_decode_kv(cache, 11, 8, True, 2, out_dtype=torch.float32, k_out=ko, v_out=vo)
    torch.cuda.synchronize()
    assert torch.all(big_k[-64:] == 7.0) and torch.all(big_v[-64:] == 7.0)


def test_empty_inputs_are_no_ops():
    cache = tq.alloc_cache(1, 2, 4, 128, 8, 3)
    for t in cache.values():
        t.view(torch.uint8).fill_(0x5A)
    k = torch.empty((1, 2, 0, 128), dtype=torch.bfloat16, device="cuda")
    tq.tq_encode_kv(k, k, 8, True, 3, cache, t_off=4)
    ko, vo = tq.tq_decode_kv(cache, 0, 8, True, 3)
    torch.cuda.synchronize()
    assert ko.numel() == 0 and vo.numel() == 0
    for t in cache.values():
        assert torch.all(t.view(torch.uint8) == 0x5A)


def test_argument_errors_on_device_tensors():
    k = torch.zeros((1, 2, 4, 96), dtype=torch.bfloat16, device="cuda")
    cache = tq.alloc_cache(1, 2, 4, 128, 8, 3)
    with pytest.raises(tq.TQError) as e:
        tq.tq_encode_kv(k, k, 8, True, 3, cache)
    assert e.value.status == 2
    k = torch.zeros((1, 2, 4, 128), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(tq.TQError) as e:
        tq.tq_encode_kv(k, k, 8, True, 6, cache)
    assert e.value.status == 3
    with pytest.raises(tq.TQError) as e:
        tq.tq_encode_kv(k, k, 8, True, 3, cache, t_off=1)
    assert e.value.status == 1
    # a K view that starts 2 bytes into its storage: 16-byte alignment fails
    flat = torch.zeros(1 * 2 * 4 * 128 + 8, dtype=torch.bfloat16, device="cuda")
    kv = flat[1:1 + 1024].view(1, 2, 4, 128)
    with pytest.raises(tq.TQError) as e:
        tq.tq_encode_kv(kv, k, 8, True, 3, cache)
    assert e.value.status == 4


# ---- the Lloyd-Max index routine ------------------------------------------------------
@pytest.mark.parametrize("bits", [2, 3, 4, 5, 8])
def test_lloyd_max_index_at_boundaries(bits):
    _, b = oracle.lloyd_max(bits)
    vals = [b]
    x = b.copy()
    y = b.copy()
    for _ in range(4):  # the 4 floats on each side of every boundary
        x = np.nextafter(x, np.float32(np.inf))
        y = np.nextafter(y, np.float32(-np.inf))
        vals += [x.copy(), y.copy()]
    rng = np.random.default_rng(bits)
    vals += [rng.standard_normal(200000).astype(np.float32) * 3,
             rng.uniform(-6, 6, 200000).astype(np.float32),
             np.array([np.inf, -np.inf, np.nan, 0.0, -0.0, 1e30, -1e30, 5.66, -5.66], np.float32)]
    # every cell edge of the device's lookup grid (cells are rint(u * S)) and its neighbours
    S = {2: 2, 3: 4, 4: 8, 5: 16, 8: 64}[bits]
    edges = ((np.arange(-8 * S, 8 * S) + 0.5) / S).astype(np.float32)
    vals += [edges, np.nextafter(edges, np.float32(np.inf)), np.nextafter(edges, np.float32(-np.inf))]
    u = np.concatenate(vals).astype(np.float32)
    got = tq.tq_lloyd_max_index(torch.from_numpy(u).cuda(), bits).cpu().numpy()
    ref = oracle.searchsorted(b, u)
    assert np.array_equal(got, ref), np.argwhere(got != ref)[:5]


# ---- non-finite inputs, element by element --------------------------------------------
# The page's formulas define a result for Inf and NaN inputs too (IEEE
# arithmetic): a NaN in a key group makes its min, max, scale and zero point
# NaN and every code 0 (NaN converts to 0); an Inf gives an Inf scale; one Inf
# or NaN in a value row reaches every rotated coordinate, so the RMS is Inf or
# NaN, every normalised value is NaN and every index 0 (searchsorted counts
# nothing below NaN); a finite row whose sum of squares overflows has RMS Inf
# and normalised values +-0.
def _k_pattern(x, i):
    """Plant key pattern i into the 32-element group view x (float32)."""
    p = i % 10
    if p == 0:
        x[0] = float("nan")
    elif p == 1:
        x[17] = float("nan")
    elif p == 2:
        x[:] = float("nan")
    elif p == 3:
        x[5] = float("inf")
    elif p == 4:
        x[9] = float("-inf")
    elif p == 5:
        x[3], x[20] = float("inf"), float("-inf")
    elif p == 6:
        x[:] = float("inf")
    elif p == 7:
        x[:] = 3e38
        x[1::2] = -3e38  # the range overflows
    elif p == 8:
        x[:] = 3e38  # range 0; the signed zero point's numerator overflows
    else:
        x[:] = x.abs() * 0.25 + 0.5
        x[7] = float("inf")  # positive minimum: zero point +0


def _v_pattern(x, i):
    """Plant value pattern i into the row view x (float32)."""
    p = i % 6
    if p == 0:
        x[3] = float("inf")
    elif p == 1:
        x[x.numel() - 1] = float("nan")
    elif p == 2:
        x[0], x[1] = float("inf"), float("-inf")
    elif p == 3:
        x[7] = 1e38  # finite rotation, the sum of squares overflows
    elif p == 4:
        x[:] = 3e38  # the rotation itself overflows
    else:
        x[11] = float("-inf")


def _non_finite_kv(B, H, T, D, dtype, seed, n_rows):
    k = _rand((B, H, T, D), torch.float32, seed)
    v = _rand((B, H, T, D), torch.float32, seed + 1)
    R = B * H * T
    rng = np.random.default_rng(seed)
    rows = sorted(set([0, R - 1, R // 2] + rng.choice(R, size=min(R, n_rows), replace=False).tolist()))
    kf, vf = k.view(-1, D), v.view(-1, D)
    for j, r in enumerate(rows):
        _k_pattern(kf[r, 32 * (j % (D // 32)): 32 * (j % (D // 32)) + 32], j)
        _v_pattern(vf[r], j)
    return k.to(dtype).contiguous(), v.to(dtype).contiguous()


@pytest.mark.parametrize("D,vb,dtype,T", [
    (128, 3, torch.bfloat16, 1000),    # single cell table, 256-thread blocks
    (64, 2, torch.float32, 777),
    (256, 4, torch.float32, 301),
    (512, 5, torch.bfloat16, 129),
    (128, 8, torch.bfloat16, 65544),   # >= 65536 rows: replicated cell tables (wide shape)
    (128, 3, torch.bfloat16, 65544),
    (64, 5, torch.bfloat16, 65544),
])
def test_non_finite_rows_match_oracle(D, vb, dtype, T):
    """Rows holding Inf, NaN and overflowing values, and the rows that share
    warps with them, match the oracle element by element: codes, scales and
    zero points (NaN equal to NaN), and decodes."""
    k, v = _non_finite_kv(1, 1, T, D, dtype, 900 + D + vb + T, 60)
    for kb, ks in ((8, True), (4, False)):
        check_roundtrip(k, v, kb, ks, vb)


# ---- buffers in pinned host memory (read and written over the CPU-GPU link) ------------
@pytest.mark.parametrize("D,vb", [(128, 8), (128, 3), (512, 5)])
def test_pinned_host_buffers(D, vb):
    """K, V read straight from pinned host memory and decoded outputs written
    straight to pinned host memory give the same bytes as device buffers
    (a decode with a host buffer takes the per-lane kernel, not bulk
    copies)."""
    rpw = 32 // (D // 32)
    k = _rand((2, 4, 16 * rpw, D), torch.bfloat16, 70 + D + vb)
    v = _rand((2, 4, 16 * rpw, D), torch.bfloat16, 71 + D + vb)
    kh, vh = k.pin_memory(), v.pin_memory()
    B, H, T, _ = k.shape
    c_dev = gpu_encode(k, v, 8, True, vb)
    c_host = tq.alloc_cache(B, H, T, D, 8, vb)
    s = torch.cuda.current_stream()
    tq.tq_encode_kv(kh, vh, 8, True, vb, c_host, stream=s)
    torch.cuda.synchronize()
    a, b = cache_to_numpy(c_dev), cache_to_numpy(c_host)
    for n in a:
        assert np.array_equal(a[n], b[n]), n
    for dt in (torch.bfloat16, torch.float32):
        kd, vd = tq.tq_decode_kv(c_dev, T, 8, True, vb, out_dtype=dt)
        ko = torch.empty((B, H, T, D), dtype=dt).pin_memory()
        vo = torch.empty((B, H, T, D), dtype=dt).pin_memory()
        tq.tq_decode_kv(c_dev, T, 8, True, vb, out_dtype=dt, k_out=ko, v_out=vo, stream=s)
        torch.cuda.synchronize()
        assert torch.equal(kd.cpu(), ko) and torch.equal(vd.cpu(), vo)


@pytest.mark.parametrize("D", [256, 512])
@pytest.mark.parametrize("vb", [2, 3, 4, 5, 8])
def test_wide_encode_every_row(D, vb):
    """bf16 launches of at least 65536 rows take the wide encode shape (cell
    tables replicated per lane, 512-thread blocks); at head_dim 256 and 512 a
    row spans 8 and 16 lanes (3 and 4 cross-lane Hadamard stages). Every row
    against the oracle at every width, with a ragged last tile."""
    T = 65536 + 2 * (32 // (D // 32)) + 1
    k = _rand((1, 1, T, D), torch.bfloat16, 40 + D + vb)
    v = _rand((1, 1, T, D), torch.bfloat16, 41 + D + vb, scale=2.0)
    check_roundtrip(k, v, 8, True, vb)
