"""The allocation-free attention entry point, tq_decode_attention_noalloc.

Some callers cannot allocate device memory (a plugin inside a serving runtime
that owns the whole device memory budget, or a latency-bound path where an
allocation could synchronize the device), so they cannot hand
tq_decode_attention the scratch workspace it needs. The no-allocation entry
point takes that scratch from a fixed array inside the library. This test
calls it through the C ABI (ctypes, no Python wrapper in between) twice in a
row, with different inputs each time so that whatever the first call left in
the shared array would show, and checks each result against the existing
entry point's within the attention parity tolerance. It also checks that a
size needing more scratch than the array holds is refused on the host.

The file name makes pytest collect it last, so a run that stops at the first
failure has run every other test first; it also passes on its own in a fresh
process.
"""
import ctypes

import numpy as np
import pytest
import torch

import turboquant_kv_cache_tq_gb300 as tq

pytestmark = pytest.mark.gpu

ATTN_TOL = 5e-6  # the attention parity tolerance (x max|Vrot|), as in test_gpu_attention.py
SCRATCH_BYTES = 64 << 20  # TQ_ATTENTION_NOALLOC_SCRATCH_BYTES in include/tq.h


@pytest.fixture(scope="module")
def L():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from turboquant_kv_cache_tq_gb300 import build

    build.build()
    return tq.lib()


def _case(B, Hkv, G, T, D, kb, ks, vb, seed):
    g = torch.Generator().manual_seed(seed)
    t_cap = (T + 15) // 16 * 16
    k = torch.randn((B, Hkv, T, D), generator=g).to(torch.bfloat16).cuda()
    v = (1.5 * torch.randn((B, Hkv, T, D), generator=g)).to(torch.bfloat16).cuda()
    q = torch.randn((B, Hkv * G, 1, D), generator=g).to(torch.bfloat16).cuda()
    cache = tq.alloc_cache(B, Hkv, t_cap, D, kb, vb)
    tq.tq_encode_kv(k, v, kb, ks, vb, cache)
    lp = torch.tensor([(3 * b) % max(T // 2, 1) for b in range(B)], dtype=torch.int32, device="cuda")
    return q, cache, lp, t_cap


def _noalloc(L, q, cache, lp, T, kb, ks, vb, t_cap, out):
    B, Hq, Nq, D = q.shape
    Hkv = cache["k_codes"].shape[1]
    ptrs = [cache[n].data_ptr() for n in ("k_codes", "k_scales", "k_zeros", "v_codes", "v_scales")]
    return L.tq_decode_attention_noalloc(q.data_ptr(), B, Hq, Nq, *ptrs, Hkv, T, D, t_cap, kb, int(ks), vb,
                                         lp.data_ptr(), ctypes.c_float(D ** -0.5), out.data_ptr(), 0,
                                         torch.cuda.current_stream().cuda_stream)


def _vrot_max(cache, T, kb, ks, vb):
    _, vr = tq.tq_decode_kv_rotated(cache, T, kb, ks, vb, out_dtype=torch.float32)
    return vr.abs().nan_to_num(0.0).amax(dim=(2, 3))  # [B, Hkv]


def test_noalloc_matches_workspace_entry_point_twice(L):
    cases = [(4, 8, 4, 1000, 128, 8, True, 3, 1), (2, 4, 2, 333, 64, 4, False, 5, 2),
             (3, 8, 2, 517, 256, 8, True, 4, 3), (2, 4, 4, 211, 512, 8, True, 5, 4)]
    for (B, Hkv, G, T, D, kb, ks, vb, seed) in cases:
        q, cache, lp, t_cap = _case(B, Hkv, G, T, D, kb, ks, vb, seed)
        assert tq.tq_decode_attention_workspace_size(B, Hkv, T, D) <= SCRATCH_BYTES
        want = tq.tq_decode_attention(q, cache, T, kb, ks, vb, left_pad=lp, out_dtype=torch.float32)
        got = torch.full_like(want, float("nan"))
        st = _noalloc(L, q, cache, lp, T, kb, ks, vb, t_cap, got)
        assert st == 0, tq.tq_status_string(st)
        torch.cuda.synchronize()
        vmax = _vrot_max(cache, T, kb, ks, vb).repeat_interleave(G, dim=1)[:, :, None, None]
        err = ((got - want).abs() / vmax).max().item()
        assert not torch.isnan(got).any()
        assert err <= ATTN_TOL, err


def test_noalloc_refuses_sizes_beyond_the_scratch(L):
    # 128 x 64 (batch, kv head) pairs need more partial records than the fixed
    # array holds at head_dim 128 (6849 pairs on a 152-SM part); the call is
    # refused on the host, before any launch
    need = tq.tq_decode_attention_workspace_size(128, 64, 1 << 20, 128)
    assert need > SCRATCH_BYTES
    q = torch.zeros((128, 64, 1, 128), dtype=torch.bfloat16, device="cuda")
    one = torch.zeros(16, dtype=torch.uint8, device="cuda")
    p = one.data_ptr()
    st = L.tq_decode_attention_noalloc(q.data_ptr(), 128, 64, 1, p, p, p, p, p, 64, 1 << 20, 128, 1 << 20, 8, 1,
                                       3, None, ctypes.c_float(0.1), p, 0, None)
    assert st == 1  # TQ_ERR_INVALID_ARG


def test_noalloc_empty_batch_is_a_no_op(L):
    """B == 0 returns TQ_OK like the workspace entry point, whatever the head_dim."""
    for D in (64, 128, 256, 512):
        q = torch.zeros((1, 8, 1, D), dtype=torch.bfloat16, device="cuda")
        one = torch.zeros(16, dtype=torch.uint8, device="cuda")
        p = one.data_ptr()
        st = L.tq_decode_attention_noalloc(q.data_ptr(), 0, 8, 1, p, p, p, p, p, 8, 64, D, 64, 8, 1, 3, None,
                                           ctypes.c_float(0.1), p, 0, None)
        assert st == 0, tq.tq_status_string(st)
