"""GPU parity of the batched packed-cache row operations (tq_cache_assemble and
the merge / extend / extract / filter helpers built on it) against the
oracle's batched-quant.ts operations: byte equality of every buffer, bytes
outside the destination window untouched.

Page "@mlx-bun/inference 0.0.0-stage -> 1.0.0": batched-quant.ts
mergeQuantRows, extendQuantRows, extractQuantRow, filterQuantRows.
"""
import numpy as np
import pytest
import torch

import oracle
from oracle import batched_cache as bc
import turboquant_kv_cache_tq_gb300 as tq
from tests.gpu_common import CACHE_KEYS, cache_from_numpy, cache_to_numpy, require_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def _row_np(L, seed, H, D, kb, ks, vb):
    rng = np.random.default_rng(seed)
    k = rng.standard_normal((1, H, L, D)).astype(np.float32)
    v = rng.standard_normal((1, H, L, D)).astype(np.float32)
    return oracle.encode_kv(k, v, kb, ks, vb)


def _to_gpu_with_capacity(c: dict, t_cap: int, fill=0x5A) -> dict:
    """Upload an oracle cache into device buffers of a larger capacity whose
    tail holds a sentinel byte."""
    B, H, L, _ = c["k_codes"].shape
    dev = cache_from_numpy(c)
    out = {}
    for k in CACHE_KEYS:
        t = dev[k]
        big = torch.empty((B, H, t_cap, t.shape[-1]), dtype=t.dtype, device="cuda")
        big.view(torch.uint8).fill_(fill)
        big[:, :, :L] = t
        out[k] = big
    return out


def _window(gpu: dict, width: int) -> dict:
    return {k: v[:, :, :width] for k, v in cache_to_numpy(gpu).items()}


def _assert_same(got: dict, want: dict, what: str):
    for k in CACHE_KEYS:
        assert got[k].shape == want[k].shape, (what, k, got[k].shape, want[k].shape)
        assert np.array_equal(got[k], want[k]), "%s: %s differs" % (what, k)


def _assert_tail_untouched(gpu: dict, width: int, fill=0x5A):
    for k in CACHE_KEYS:
        tail = gpu[k][:, :, width:].contiguous().view(torch.uint8)
        assert torch.all(tail == fill), "bytes past the window were written (%s)" % k


GEOMS = [(2, 64, 8, True, 3), (2, 128, 8, True, 3), (3, 64, 5, False, 5), (1, 256, 4, False, 2),
         (2, 512, 2, False, 8)]


@pytest.mark.parametrize("H,D,kb,ks,vb", GEOMS)
def test_merge_extend_extract_filter(H, D, kb, ks, vb):
    lens = [7, 1, 12, 5, 12]
    rows_np = [_row_np(n, 100 + i, H, D, kb, ks, vb) for i, n in enumerate(lens)]
    rows_gpu = [(_to_gpu_with_capacity(r, n + 3), n) for r, n in zip(rows_np, lens)]

    # merge (destination with spare capacity: the tail must stay untouched)
    want, pads_w, width_w = bc.merge_rows(rows_np)
    got, pads, width = tq.merge_rows(rows_gpu, t_cap=16)
    torch.cuda.synchronize()
    assert (pads, width) == (pads_w, width_w)
    got_np = _window(got, width)
    _assert_same(got_np, want, "merge")

    # extend by a wider and by a narrower row
    for j, n in enumerate((15, 3)):
        r_np = _row_np(n, 200 + j, H, D, kb, ks, vb)
        e_want, e_pads_w, e_w = bc.extend_rows(want, pads_w, r_np)
        e_got, e_pads, e_width = tq.extend_rows(got, width, pads, (_to_gpu_with_capacity(r_np, n + 1), n))
        torch.cuda.synchronize()
        assert (e_pads, e_width) == (e_pads_w, e_w)
        _assert_same(_window(e_got, e_width), e_want, "extend by %d" % n)

    # extract every row back out
    for i in range(len(lens)):
        x = tq.extract_row(got, width, pads[i], i)
        torch.cuda.synchronize()
        _assert_same(cache_to_numpy(x), bc.extract_row(want, pads_w[i], i), "extract %d" % i)

    # filter (reordering, repeats allowed)
    keep = [4, 0, 2, 2]
    f = tq.filter_rows(got, width, keep)
    torch.cuda.synchronize()
    _assert_same(_window(f, width), bc.filter_rows(want, keep), "filter")


def test_destination_tail_untouched_and_many_rows():
    """More rows than one launch carries (48), a window inside a larger
    capacity, all-padding rows, and sources read from an offset."""
    H, D, kb, ks, vb = 2, 128, 8, True, 4
    rng = np.random.default_rng(3)
    src_np = _row_np(40, 7, H, D, kb, ks, vb)
    src = _to_gpu_with_capacity(src_np, 48)
    n_rows, width, t_cap = 61, 20, 29
    dst = tq.alloc_cache(n_rows, H, t_cap, D, kb, vb)
    for t in dst.values():
        t.view(torch.uint8).fill_(0x5A)
    plan = []
    for r in range(n_rows):
        if r % 9 == 4:
            plan.append(None)
            continue
        length = int(rng.integers(0, width + 1))
        t0 = int(rng.integers(0, 40 - length + 1))
        plan.append((src, 0, t0, length))
    tq.tq_cache_assemble(plan, dst, width)
    torch.cuda.synchronize()
    _assert_tail_untouched(dst, width)
    got = _window(dst, width)
    for r, pl in enumerate(plan):
        length = 0 if pl is None else pl[3]
        for k in CACHE_KEYS:
            row = got[k][r]
            assert np.all(row[:, :width - length] == 0)
            if length:
                assert np.array_equal(row[:, width - length:], src_np[k][0, :, pl[2]:pl[2] + length])


def test_merged_batch_attends_like_each_row_alone():
    """Continuous batching end to end on the GPU: rows encoded on the GPU,
    merged, attended with the left-pad mask, against the oracle's attention
    over each row alone."""
    from tests.test_gpu_attention import ATTN_TOL

    H, D, G, kb, ks, vb = 2, 128, 4, 8, True, 3
    lens = [37, 16, 64, 5]
    rows, rows_np = [], []
    for i, n in enumerate(lens):
        g = torch.Generator().manual_seed(300 + i)
        k = torch.randn((1, H, n, D), generator=g).to(torch.bfloat16)
        v = torch.randn((1, H, n, D), generator=g).to(torch.bfloat16)
        c = tq.alloc_cache(1, H, n, D, kb, vb)
        tq.tq_encode_kv(k.cuda(), v.cuda(), kb, ks, vb, c)
        rows.append((c, n))
    merged, pads, width = tq.merge_rows(rows, t_cap=64)
    q = torch.randn((len(lens), H * G, 1, D), generator=torch.Generator().manual_seed(9)).to(torch.bfloat16)
    lp = torch.tensor(pads, dtype=torch.int32, device="cuda")
    got = tq.tq_decode_attention(q.cuda(), merged, width, kb, ks, vb, left_pad=lp, out_dtype=torch.float32)
    torch.cuda.synchronize()
    qb = q.view(torch.int16).numpy().view(np.uint16)
    for i, (c, n) in enumerate(rows):
        cn = cache_to_numpy(c)
        want = oracle.decode_attention(qb[i:i + 1], cn, n, kb, ks, vb)
        _, vr = oracle.decode_kv(cn, n, kb, ks, vb, out_dtype=oracle.BF16, rotated_v=True)
        vmax = np.abs(oracle.bf16_bits_to_f32(vr)).max()
        err = np.abs(got[i].cpu().numpy().astype(np.float64) - want[0]).max()
        assert err <= ATTN_TOL * vmax, (i, err)


def test_host_checks():
    c = tq.alloc_cache(1, 2, 8, 128, 8, 3)
    d = tq.alloc_cache(2, 2, 8, 128, 8, 3)
    with pytest.raises(tq.TQError):  # reads past the source capacity
        tq.tq_cache_assemble([(c, 0, 4, 5), None], d, 6)
    with pytest.raises(tq.TQError):  # length longer than the window
        tq.tq_cache_assemble([(c, 0, 0, 7), None], d, 6)
    with pytest.raises(tq.TQError):  # batch row outside the source
        tq.tq_cache_assemble([(c, 1, 0, 3), None], d, 6)
    with pytest.raises(tq.TQError):  # window wider than the destination
        tq.tq_cache_assemble([(c, 0, 0, 3), None], d, 9)
