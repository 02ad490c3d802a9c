"""The library's calls inside CUDA graphs, the way the benchmark runs them:
encode + decode and the fused decode attention are captured once (after a
first eager call, which sets each kernel's attributes and occupancy), then
replayed on new input contents; every replay must equal the eager calls on
the same inputs, byte for byte.
"""
import pytest
import torch

import turboquant_kv_cache_tq_gb300 as tq
from tests.gpu_common import require_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def _fill(t, seed):
    g = torch.Generator(device="cuda").manual_seed(seed)
    t.copy_(torch.randn(t.shape, generator=g, device="cuda").to(t.dtype))


def test_codec_in_a_graph():
    B, H, T, D, kb, ks, vb = 2, 4, 300, 128, 8, True, 3
    k = torch.empty((B, H, T, D), dtype=torch.bfloat16, device="cuda")
    v = torch.empty_like(k)
    cache = tq.alloc_cache(B, H, T, D, kb, vb)
    ko, vo = torch.empty_like(k), torch.empty_like(v)
    s = torch.cuda.Stream()
    _fill(k, 1), _fill(v, 2)
    with torch.cuda.stream(s):
        tq.tq_encode_kv(k, v, kb, ks, vb, cache, stream=s)
        tq.tq_decode_kv(cache, T, kb, ks, vb, k_out=ko, v_out=vo, stream=s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        tq.tq_encode_kv(k, v, kb, ks, vb, cache, stream=s)
        tq.tq_decode_kv(cache, T, kb, ks, vb, k_out=ko, v_out=vo, stream=s)
    for seed in (3, 4):
        _fill(k, seed), _fill(v, seed + 10)
        g.replay()
        torch.cuda.synchronize()
        c2 = tq.alloc_cache(B, H, T, D, kb, vb)
        tq.tq_encode_kv(k, v, kb, ks, vb, c2)
        k2, v2 = tq.tq_decode_kv(c2, T, kb, ks, vb)
        torch.cuda.synchronize()
        for n in c2:
            assert torch.equal(cache[n].view(torch.uint8), c2[n].view(torch.uint8)), n
        assert torch.equal(ko.view(torch.int16), k2.view(torch.int16))
        assert torch.equal(vo.view(torch.int16), v2.view(torch.int16))


def test_attention_in_a_graph():
    B, Hkv, G, T, D, kb, ks, vb = 3, 2, 4, 500, 128, 8, True, 4
    t_cap = 512
    k = torch.empty((B, Hkv, T, D), dtype=torch.bfloat16, device="cuda")
    v = torch.empty_like(k)
    cache = tq.alloc_cache(B, Hkv, t_cap, D, kb, vb)
    q = torch.empty((B, Hkv * G, 1, D), dtype=torch.bfloat16, device="cuda")
    lp = torch.tensor([0, 7, 100], dtype=torch.int32, device="cuda")
    out = torch.empty((B, Hkv * G, 1, D), dtype=torch.float32, device="cuda")
    work = torch.empty(tq.tq_decode_attention_workspace_size(B, Hkv, T, D), dtype=torch.uint8, device="cuda")
    s = torch.cuda.Stream()
    _fill(k, 5), _fill(v, 6), _fill(q, 7)
    with torch.cuda.stream(s):
        tq.tq_encode_kv(k, v, kb, ks, vb, cache, stream=s)
        tq.tq_decode_attention(q, cache, T, kb, ks, vb, left_pad=lp, out_dtype=torch.float32, out=out,
                               workspace=work, stream=s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        tq.tq_encode_kv(k, v, kb, ks, vb, cache, stream=s)
        tq.tq_decode_attention(q, cache, T, kb, ks, vb, left_pad=lp, out_dtype=torch.float32, out=out,
                               workspace=work, stream=s)
    for seed in (8, 9):
        _fill(k, seed), _fill(v, seed + 10), _fill(q, seed + 20)
        g.replay()
        torch.cuda.synchronize()
        got = out.clone()
        tq.tq_encode_kv(k, v, kb, ks, vb, cache)
        want = tq.tq_decode_attention(q, cache, T, kb, ks, vb, left_pad=lp, out_dtype=torch.float32)
        torch.cuda.synchronize()
        assert torch.equal(got, want)
