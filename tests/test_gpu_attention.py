"""GPU parity of the fused decode attention (tq_decode_attention) against the
oracle's decode_attention on the same packed cache bytes.

Page "@mlx-bun/inference 0.0.0-stage -> 1.0.0": ops.ts tryDecodePackedKv with
deferV (bf16 keys, bf16 rotated values), attention over them, unrotateValues
on the output; batched-mask.ts, the left-pad key mask.

Tolerance. The oracle is exact (double precision over the same bf16 decoded
rows). The kernel's products of bf16 operands are exact; what it rounds is
(1) the fp32 accumulation of each score over D products, (2) the softmax
weights, split into two bf16 parts (relative error <= 2^-18 each), (3) the
fp32 accumulation of the weighted values and of the chunk merge, (4) the
fp32 normalisation and inverse rotation. Every term is a relative error of a
weight or of a partial sum of weighted value rows, so the output error is
bounded by a small multiple of the largest decoded value magnitude
max|Vrot| (the weights sum to one): the tests require
|o_gpu - o_ref| <= ATTN_TOL * max|Vrot| per (batch, head) with
ATTN_TOL = 5e-6: the weight split alone can reach 2^-18 = 3.8e-6 if every
weight's rounding had the same sign, and the fp32 accumulations add a few
units of 2^-24 growing like the square root of the number of terms (measured
on GB300: at most 5e-7 over the cases below). NaN rows where the oracle has
NaN rows, and exact zeros where the oracle's row has no valid key.
"""
import numpy as np
import pytest
import torch

import oracle
import turboquant_kv_cache_tq_gb300 as tq
from tests.gpu_common import cache_from_numpy, cache_to_numpy, oracle_encode, require_gpu

pytestmark = pytest.mark.gpu

ATTN_TOL = 5e-6
KEY_MODES = [(2, False), (4, False), (5, False), (8, False), (8, True)]


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def _rand(shape, dtype, seed, scale=1.0):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(shape, generator=g) * scale).to(dtype).contiguous()


def _bits(t):
    return t.cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def _vrot_max(rc, T, kb, ks, vb):
    """max |Vrot| per (batch, kv head) over tokens [0, T) (bf16 decode, float64)."""
    _, vr = oracle.decode_kv(rc, T, kb, ks, vb, out_dtype=oracle.BF16, rotated_v=True)
    v = oracle.bf16_bits_to_f32(vr).astype(np.float64)
    return np.nan_to_num(np.abs(v), nan=0.0).max(axis=(2, 3)) if T else np.zeros(v.shape[:2])


def compare_attention(got, want, vmax, G, what, tol=ATTN_TOL):
    """got, want: [B, Hq, Nq, D]; vmax: [B, Hkv]. Returns the largest error
    relative to max|Vrot|."""
    g = got.astype(np.float64)
    gn, wn = np.isnan(g), np.isnan(want)
    assert np.array_equal(gn.any(-1), wn.any(-1)), "%s: NaN rows differ" % what
    assert np.array_equal(gn, wn), "%s: NaN positions differ" % what
    zero_rows = np.all(want == 0, axis=-1)
    assert np.all(g[zero_rows] == 0), "%s: rows without a valid key must be exactly zero" % what
    scale = np.repeat(vmax, G, axis=1)[:, :, None, None]
    err = np.where(wn, 0.0, np.abs(g - np.where(wn, 0.0, want)))
    rel = err / np.maximum(scale, 1e-30)
    worst = float(rel.max()) if rel.size else 0.0
    assert worst <= tol, "%s: error %.3g x max|Vrot| above %.1g" % (what, worst, tol)
    return worst


def run_case(B, Hkv, G, Nq, T, D, kb, ks, vb, t_cap=None, left_pad=None, seed=0, out_dtype=torch.float32,
             k=None, qscale=1.0):
    t_cap = t_cap if t_cap is not None else (T + 15) // 16 * 16
    if k is None:
        k = _rand((B, Hkv, T, D), torch.bfloat16, seed)
    v = _rand((B, Hkv, T, D), k.dtype, seed + 1, scale=1.5)
    rc = oracle_encode(k, v, kb, ks, vb, t_cap=t_cap)
    q = _rand((B, Hkv * G, Nq, D), torch.bfloat16, seed + 2, scale=qscale)
    dev = cache_from_numpy(rc)
    lp = None if left_pad is None else torch.tensor(left_pad, dtype=torch.int32, device="cuda")
    got = tq.tq_decode_attention(q.cuda(), dev, T, kb, ks, vb, left_pad=lp, out_dtype=out_dtype)
    torch.cuda.synchronize()
    want = oracle.decode_attention(_bits(q), rc, T, kb, ks, vb, left_pad=left_pad)
    vmax = _vrot_max(rc, T, kb, ks, vb)
    return got, want, vmax, rc, q


@pytest.mark.parametrize("D", [64, 128, 256, 512])
@pytest.mark.parametrize("vb", [2, 3, 4, 5, 8])
def test_matches_oracle_all_widths(D, vb):
    """Every key mode and value width; ragged token counts spanning several
    16-token tiles and several split blocks. At head_dim 256 and 512 two warps
    share each tile, one per half of head_dim."""
    T = {64: 203, 128: 141, 256: 77, 512: 53}[D]
    for i, (kb, ks) in enumerate(KEY_MODES):
        got, want, vmax, _, _ = run_case(2, 2, 4, 1, T, D, kb, ks, vb, seed=10 * i + D + vb)
        compare_attention(got.cpu().numpy(), want, vmax, 4, "D%d k%d%s v%d" % (D, kb, "s" if ks else "", vb))


@pytest.mark.parametrize("G,Nq", [(1, 1), (2, 3), (4, 2), (8, 1), (8, 2), (16, 1), (5, 3)])
def test_query_rows_and_causal_tail(G, Nq):
    """Grouped-query head map, several query tokens with the causal tail
    (query n sees keys <= T - Nq + n), one and two query-row tiles."""
    got, want, vmax, _, _ = run_case(2, 3, G, Nq, 90, 128, 8, True, 3, seed=G * 7 + Nq)
    compare_attention(got.cpu().numpy(), want, vmax, G, "G%d Nq%d" % (G, Nq))


@pytest.mark.parametrize("G,Nq,pads", [(4, 1, None), (8, 2, [0, 33, 70]), (16, 1, [5, 0, 90]), (3, 5, None)])
def test_head_dim_512_query_rows_and_pads(G, Nq, pads):
    """head_dim 512 (a warp pair per tile, partial scores added through shared
    memory) with one and two query-row tiles, causal tails and left pads."""
    got, want, vmax, _, _ = run_case(3, 2, G, Nq, 90, 512, 8, True, 4, left_pad=pads, seed=G * 11 + Nq)
    compare_attention(got.cpu().numpy(), want, vmax, G, "D512 G%d Nq%d pads %s" % (G, Nq, pads))
    got, want, vmax, _, _ = run_case(3, 2, G, Nq, 90, 512, 4, False, 3, left_pad=pads, seed=G * 13 + Nq,
                                     out_dtype=torch.bfloat16)
    ref = oracle.f32_to_bf16_bits(want.astype(np.float32))
    d = np.abs(oracle.bf16_bits_to_f32(_bits(got)).astype(np.float64) - oracle.bf16_bits_to_f32(ref))
    assert np.all(d <= 2.0 ** -7 * np.abs(want) + ATTN_TOL * np.repeat(vmax, G, axis=1)[:, :, None, None])


@pytest.mark.parametrize("B,Hkv,G,Nq,T,D,vb,pads", [
    (1, 1, 4, 1, 16384, 512, 2, None),
    (2, 1, 8, 2, 20000, 128, 3, [0, 2500]),
    (1, 2, 4, 1, 24000, 256, 4, None),
    (1, 1, 4, 1, 60000, 64, 5, None),
])
def test_heads_over_many_split_blocks(B, Hkv, G, Nq, T, D, vb, pads):
    """Few heads with long caches: each head's tiles spread over many split
    blocks, so a row has many partial records and the combine merges them in
    several chunks whose sums the last chunk to finish adds up (on a 152-SM
    GB300: 3, 2, 2 and 4 chunks per row tile for these cases), with row tiles
    spanning two heads, two query-row tiles and left pads."""
    got, want, vmax, _, _ = run_case(B, Hkv, G, Nq, T, D, 8, True, vb, left_pad=pads, seed=T + D)
    compare_attention(got.cpu().numpy(), want, vmax, G, "B%d Hkv%d G%d Nq%d T%d D%d" % (B, Hkv, G, Nq, T, D))


@pytest.mark.parametrize("pads", [[0, 5, 17, 63], [16, 1, 40, 0], [89, 0, 3, 90]])
def test_left_pad(pads):
    """Left-padded batch rows; a pad that covers every key gives a zero row."""
    got, want, vmax, _, _ = run_case(4, 2, 4, 2, 90, 128, 8, True, 3, left_pad=pads, seed=sum(pads))
    compare_attention(got.cpu().numpy(), want, vmax, 4, "pads %s" % pads)


@pytest.mark.parametrize("T", [1, 2, 15, 16, 17, 64, 65, 1000])
def test_token_counts(T):
    got, want, vmax, _, _ = run_case(1, 2, 4, 1, T, 64, 4, False, 2, seed=T)
    compare_attention(got.cpu().numpy(), want, vmax, 4, "T%d" % T)


def test_capacity_larger_than_T():
    """Tokens past T inside the capacity are never read into the result, even
    when the bytes there are garbage."""
    B, Hkv, G, T, D, t_cap = 2, 2, 4, 37, 128, 80
    k = _rand((B, Hkv, T, D), torch.bfloat16, 5)
    v = _rand((B, Hkv, T, D), torch.bfloat16, 6)
    rc = oracle_encode(k, v, 8, True, 3, t_cap=t_cap)
    junk = {n: a.copy() for n, a in rc.items()}
    rng = np.random.default_rng(0)
    for n, a in junk.items():
        tail = a[:, :, T:]
        tail[...] = rng.integers(0, 256, size=tail.shape, dtype=np.uint8).view(a.dtype) if a.dtype == np.uint8 \
            else rng.integers(0, 65536, size=tail.shape, dtype=np.uint16)
    q = _rand((B, Hkv * G, 1, D), torch.bfloat16, 7)
    got = tq.tq_decode_attention(q.cuda(), cache_from_numpy(junk), T, 8, True, 3, out_dtype=torch.float32)
    want = oracle.decode_attention(_bits(q), rc, T, 8, True, 3)
    compare_attention(got.cpu().numpy(), want, _vrot_max(rc, T, 8, True, 3), G, "garbage tail")


def test_constant_key_group_nan_rows():
    """The page's constant key group decodes to NaN; exactly the rows that
    attend to it are NaN."""
    B, Hkv, G, Nq, T, D = 2, 2, 2, 2, 40, 64
    k = _rand((B, Hkv, T, D), torch.float32, 8)
    k[0, 1, 11, 32:] = 0.5
    got, want, vmax, _, _ = run_case(B, Hkv, G, Nq, T, D, 8, True, 3, k=k, seed=8, left_pad=[0, 0])
    assert np.isnan(want).any()
    compare_attention(got.cpu().numpy(), want, vmax, G, "constant group")
    got2, want2, vmax2, _, _ = run_case(B, Hkv, G, Nq, T, D, 8, True, 3, k=k, seed=8, left_pad=[12, 0])
    assert not np.isnan(want2).any()
    compare_attention(got2.cpu().numpy(), want2, vmax2, G, "constant group hidden by the pad")


def test_tiny_workload():
    """The tiny workload's cache (fp32 K, V [1,2,16,64], a constant key group,
    V 3-bit), attended by 4 query heads."""
    from turboquant_kv_cache_tq_gb300.workloads import WORKLOADS, make_kv

    w = WORKLOADS["tiny"]
    k, v = make_kv(w)
    rc = oracle_encode(k, v, w.k_bits, w.k_signed, w.v_bits[0], t_cap=16)
    q = _rand((1, 4, 1, 64), torch.bfloat16, 9)
    got = tq.tq_decode_attention(q.cuda(), cache_from_numpy(rc), 16, w.k_bits, w.k_signed, w.v_bits[0],
                                 out_dtype=torch.float32)
    want = oracle.decode_attention(_bits(q), rc, 16, w.k_bits, w.k_signed, w.v_bits[0])
    compare_attention(got.cpu().numpy(), want, _vrot_max(rc, 16, w.k_bits, w.k_signed, w.v_bits[0]), 2, "tiny")


def test_bf16_output_is_the_rounded_fp32_output():
    got32, want, vmax, rc, q = run_case(2, 2, 4, 1, 120, 128, 8, True, 4, seed=31)
    got16, _, _, _, _ = run_case(2, 2, 4, 1, 120, 128, 8, True, 4, seed=31, out_dtype=torch.bfloat16)
    r16 = oracle.f32_to_bf16_bits(got32.cpu().numpy())
    assert np.array_equal(_bits(got16), r16)


def test_large_scores_stay_finite():
    """Queries ~8x larger: sharply peaked softmax, still within tolerance."""
    got, want, vmax, _, _ = run_case(1, 2, 4, 1, 300, 128, 8, True, 3, seed=41, qscale=8.0)
    compare_attention(got.cpu().numpy(), want, vmax, 4, "peaked")


def test_matches_unfused_deferred_path():
    """The same quantity through the library's unfused calls: rotated decode
    (bf16), fp32 attention in torch, tq_unrotate."""
    B, Hkv, G, T, D = 2, 4, 4, 333, 128
    got, want, vmax, rc, q = run_case(B, Hkv, G, 1, T, D, 8, True, 3, seed=51)
    dev = cache_from_numpy(rc)
    kd, vd = tq.tq_decode_kv_rotated(dev, T, 8, True, 3, out_dtype=torch.bfloat16)
    qf = q.cuda().float()
    K = kd.float().repeat_interleave(G, dim=1)
    V = vd.float().repeat_interleave(G, dim=1)
    o_rot = torch.softmax((qf @ K.transpose(-1, -2)) * D ** -0.5, dim=-1) @ V
    o = tq.tq_unrotate(o_rot.contiguous())
    compare_attention(o.cpu().numpy(), want, vmax, G, "unfused path")
    d = (o - got.cuda()).abs().max().item()
    assert d <= 2 * ATTN_TOL * float(vmax.max())


def test_repeat_calls_are_identical_and_workspace_checked():
    B, Hkv, G, T, D = 2, 2, 4, 200, 128
    k = _rand((B, Hkv, T, D), torch.bfloat16, 61)
    v = _rand((B, Hkv, T, D), torch.bfloat16, 62)
    cache = tq.alloc_cache(B, Hkv, 208, D, 8, 3)
    tq.tq_encode_kv(k.cuda(), v.cuda(), 8, True, 3, cache)
    q = _rand((B, Hkv * G, 1, D), torch.bfloat16, 63).cuda()
    need = tq.tq_decode_attention_workspace_size(B, Hkv, T, D)
    ws = torch.full((need,), 0xAB, dtype=torch.uint8, device="cuda")
    a = tq.tq_decode_attention(q, cache, T, 8, True, 3, out_dtype=torch.float32, workspace=ws)
    b = tq.tq_decode_attention(q, cache, T, 8, True, 3, out_dtype=torch.float32, workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(a, b)
    with pytest.raises(tq.TQError):
        tq.tq_decode_attention(q, cache, T, 8, True, 3, workspace=ws[: need - 16])


def test_host_checks_on_device_tensors():
    cache = tq.alloc_cache(1, 2, 24, 128, 8, 3)  # t_cap not a multiple of 16
    q = torch.zeros((1, 8, 1, 128), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(tq.TQError) as e:
        tq.tq_decode_attention(q, cache, 20, 8, True, 3)
    assert e.value.status == 4
    cache = tq.alloc_cache(1, 2, 32, 128, 8, 3)
    with pytest.raises(tq.TQError):  # 8 heads per kv head x 3 tokens > 16 rows
        tq.tq_decode_attention(torch.zeros((1, 16, 3, 128), dtype=torch.bfloat16, device="cuda"), cache, 20,
                               8, True, 3)
    cache1k = tq.alloc_cache(1, 2, 32, 1024, 8, 3)
    with pytest.raises(tq.TQError) as e:  # head_dim 1024 is not a TurboQuant head dim
        tq.tq_decode_attention(torch.zeros((1, 2, 1, 1024), dtype=torch.bfloat16, device="cuda"), cache1k, 20,
                               8, True, 3)
    assert e.value.status == 2


def test_full_size_long_context_step_sampled_rows():
    """The bench's attention step at full size and in its launch configuration
    (cache [32, 8, 8256, 128], k8s, v3, 32 query heads, one query token),
    checked against the oracle on sampled batch rows (all their heads)."""
    B, H, T, D, G, vb = 32, 8, 8256, 128, 4, 3
    cache = tq.alloc_cache(B, H, T, D, 8, vb)
    g = torch.Generator(device="cuda").manual_seed(0)
    for b0 in range(0, B, 4):
        k = (0.5 * torch.randn((4, H, T, D), generator=g, device="cuda")).to(torch.bfloat16)
        v = (0.5 * torch.randn((4, H, T, D), generator=g, device="cuda")).to(torch.bfloat16)
        tq.tq_encode_kv(k, v, 8, True, vb, {n: t[b0:b0 + 4] for n, t in cache.items()})
        del k, v
    q = torch.randn((B, H * G, 1, D), generator=g, device="cuda").to(torch.bfloat16)
    got = tq.tq_decode_attention(q, cache, T, 8, True, vb, out_dtype=torch.float32)
    torch.cuda.synchronize()
    for b in (0, 13, 31):
        sub = cache_to_numpy({n: t[b:b + 1] for n, t in cache.items()})
        want = oracle.decode_attention(_bits(q[b:b + 1]), sub, T, 8, True, vb)
        compare_attention(got[b:b + 1].cpu().numpy(), want, _vrot_max(sub, T, 8, True, vb), G, "batch row %d" % b)
