"""GPU parity of the deferred-V read path: tq_decode_kv_rotated (values left in
the rotated domain, centroid * scale) and tq_unrotate (the inverse rotation
applied once to an attention output), against the oracle's
decode_kv(rotated_v=True) and unrotate, on the same seeded inputs.

Page "@mlx-bun/inference 0.0.0-stage -> 1.0.0", file
package/src/kernels/turboquant/ops.ts: decodeValuesRotated, unrotateValues and
the deferV branch of tryDecodePackedKv.
"""
import numpy as np
import pytest
import torch

import oracle
import turboquant_kv_cache_tq_gb300 as tq
from turboquant_kv_cache_tq_gb300.workloads import WORKLOADS, make_kv
from tests.gpu_common import cache_from_numpy, compare_decoded, oracle_encode, require_gpu

pytestmark = pytest.mark.gpu

KEY_MODES = [(2, False), (4, False), (5, False), (8, False), (8, True)]


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def _rand(shape, dtype, seed, scale=1.0):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(shape, generator=g) * scale).to(dtype).contiguous()


def _bits(t):
    return t.cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


@pytest.mark.parametrize("D", [64, 128, 256, 512])
@pytest.mark.parametrize("v_bits", [2, 3, 4, 5, 8])
def test_rotated_decode_matches_oracle(D, v_bits):
    """V: one fp32 product per element, so fp32 and bf16 results are
    bit-exact; K: the same decode as tq_decode_kv."""
    T = {64: 37, 128: 29, 256: 13, 512: 7}[D]
    for i, (kb, ks) in enumerate(KEY_MODES):
        dt = torch.bfloat16 if i % 2 else torch.float32
        k = _rand((2, 3, T, D), dt, 300 + i + D + v_bits)
        v = _rand((2, 3, T, D), dt, 400 + i + D + v_bits, scale=2.0)
        rc = oracle_encode(k, v, kb, ks, v_bits)
        dev = cache_from_numpy(rc)
        kg, vg = tq.tq_decode_kv_rotated(dev, T, kb, ks, v_bits, out_dtype=torch.float32)
        kr, vr = oracle.decode_kv(rc, T, kb, ks, v_bits, out_dtype=oracle.F32, rotated_v=True)
        assert np.array_equal(vg.cpu().numpy(), vr)
        compare_decoded(kg.cpu().numpy(), kr, "K decode (rotated call)")
        kb16, vb16 = tq.tq_decode_kv_rotated(dev, T, kb, ks, v_bits, out_dtype=torch.bfloat16)
        _, vr16 = oracle.decode_kv(rc, T, kb, ks, v_bits, out_dtype=oracle.BF16, rotated_v=True)
        assert np.array_equal(_bits(vb16), vr16)
        # the K half equals the eager call's K half, bit for bit
        ke, _ = tq.tq_decode_kv(dev, T, kb, ks, v_bits, out_dtype=torch.bfloat16)
        assert torch.equal(ke.view(torch.int16), kb16.view(torch.int16))


@pytest.mark.parametrize("D", [64, 128, 256, 512])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_unrotate_matches_oracle(D, dtype):
    # ragged row counts: a partial last warp step and a partial last block
    for n, seed in ((1, 1), (5, 2), (1001, 3)):
        x = _rand((n, D), dtype, 500 + seed + D, scale=3.0)
        y = tq.tq_unrotate(x.cuda())
        torch.cuda.synchronize()
        assert y.dtype == dtype and y.shape == x.shape
        xf = x.float().numpy()
        ref = oracle.unrotate(xf)
        if dtype == torch.float32:
            compare_decoded(y.cpu().numpy(), ref, "unrotate f32")
        else:
            rb = oracle.f32_to_bf16_bits(ref)
            gb = _bits(y)
            if not np.array_equal(gb, rb):
                d = np.abs(oracle.bf16_bits_to_f32(gb).astype(np.float64) - oracle.bf16_bits_to_f32(rb))
                assert np.all(d <= 2.0 ** -7 * np.abs(ref) + 1e-30)


@pytest.mark.parametrize("D", [64, 128, 256, 512])
@pytest.mark.parametrize("v_bits", [3, 8])
def test_unrotate_of_rotated_decode_is_the_eager_decode(D, v_bits):
    """fwht(centroid * scale) is the eager V decode by definition: the two
    calls reproduce it exactly in fp32."""
    T = 33
    k = _rand((1, 2, T, D), torch.bfloat16, 600 + D)
    v = _rand((1, 2, T, D), torch.bfloat16, 700 + D)
    cache = tq.alloc_cache(1, 2, T, D, 8, v_bits)
    tq.tq_encode_kv(k.cuda(), v.cuda(), 8, True, v_bits, cache)
    _, ve = tq.tq_decode_kv(cache, T, 8, True, v_bits, out_dtype=torch.float32)
    _, vr = tq.tq_decode_kv_rotated(cache, T, 8, True, v_bits, out_dtype=torch.float32)
    vu = tq.tq_unrotate(vr)
    torch.cuda.synchronize()
    assert torch.equal(vu, ve)


def test_attention_over_rotated_values_then_unrotate():
    """Attention is linear in V, so unrotate(P @ V_rot) = P @ V_eager up to
    the summation order (the deferred-V identity the page relies on)."""
    w = WORKLOADS["llama3_8b_layer"]
    k, v = make_kv(w, B=1, T=256)
    B, H, T, D = k.shape
    cache = tq.alloc_cache(B, H, T, D, w.k_bits, 3)
    tq.tq_encode_kv(k.cuda(), v.cuda(), w.k_bits, w.k_signed, 3, cache)
    kd, ve = tq.tq_decode_kv(cache, T, w.k_bits, w.k_signed, 3, out_dtype=torch.float32)
    _, vr = tq.tq_decode_kv_rotated(cache, T, w.k_bits, w.k_signed, 3, out_dtype=torch.float32)
    g = torch.Generator(device="cuda").manual_seed(11)
    q = torch.randn((B, H, 4, D), generator=g, device="cuda")
    p = torch.softmax(q @ kd.transpose(-1, -2) / D ** 0.5, dim=-1).double()
    eager = p @ ve.double()
    deferred = tq.tq_unrotate((p @ vr.double()).float().contiguous())
    torch.cuda.synchronize()
    err = (deferred.double() - eager).abs().max().item()
    assert err <= 1e-5 * eager.abs().max().item()


def test_rotated_edge_cases():
    cache = tq.alloc_cache(1, 1, 4, 128, 8, 3)
    ko, vo = tq.tq_decode_kv_rotated(cache, 0, 8, True, 3)
    assert ko.numel() == 0 and vo.numel() == 0
    assert tq.tq_unrotate(torch.empty((0, 128), device="cuda")).numel() == 0
    with pytest.raises(tq.TQError):
        tq.tq_unrotate(torch.zeros((4, 96), device="cuda"))
    with pytest.raises(ValueError):
        tq.tq_unrotate(torch.zeros((4, 128), dtype=torch.float16, device="cuda"))
    # rows past n_rows stay untouched
    x = torch.randn((8, 128), device="cuda")
    out = torch.full((9, 128), 7.0, device="cuda")
    st = tq.lib().tq_unrotate(x.data_ptr(), 0, 8, 128, out.data_ptr(), None)
    torch.cuda.synchronize()
    assert st == 0 and torch.all(out[8] == 7.0)
    assert torch.equal(out[:8], tq.tq_unrotate(x))
