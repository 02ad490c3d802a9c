"""The debug build of the library on the small parity cases.

The debug build (libtq_debug.so, compiled with -DTQ_DEBUG_CHECKS) checks
the row, tile and record indices of its kernels' global accesses against the
buffers' extents; an index outside them sets the library's device error word
(read by tq_device_status as TQ_ERR_DEVICE_CHECK) and skips the access,
without a trap. These tests run the encode, both decode paths (per-lane and
bulk copy), the rotated decode, the unrotate and the fused attention through
the debug build on small cases, check every output equals the release
build's byte for byte, and check that no index check failed.
"""
import numpy as np
import pytest
import torch

import turboquant_kv_cache_tq_gb300 as tq
from tests.gpu_common import cache_to_numpy

pytestmark = pytest.mark.gpu

KEY_MODES = [(2, False), (4, False), (5, False), (8, False), (8, True)]


@pytest.fixture(scope="module")
def libs():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from turboquant_kv_cache_tq_gb300 import build

    build.build()
    release = tq.lib()
    debug = tq.load_library(build.build(debug=True))
    yield release, debug
    tq._lib = release


def _with(lib, fn):
    """Run fn() with the binding routed to `lib`."""
    saved = tq._lib
    tq._lib = lib
    try:
        out = fn()
        torch.cuda.synchronize()
        return out
    finally:
        tq._lib = saved


def _bytes(t):
    return t.detach().cpu().contiguous().view(torch.uint8).numpy()


def test_flags(libs):
    release, debug = libs
    assert release.tq_debug_checks() == 0 and debug.tq_debug_checks() == 1


@pytest.mark.parametrize("D", [64, 128, 256, 512])
def test_codec_matches_release(libs, D):
    release, debug = libs
    rpw = 32 // (D // 32)
    g = torch.Generator().manual_seed(D)
    for T, t_cap in ((3 * rpw, 3 * rpw + 2 * rpw), (3 * rpw + 1, 3 * rpw + 5)):  # bulk decode, per-lane decode
        for i, (kb, ks) in enumerate(KEY_MODES):
            vb = (2, 3, 4, 5, 8)[i]
            k = torch.randn((2, 2, T, D), generator=g).to(torch.bfloat16).cuda()
            v = torch.randn((2, 2, T, D), generator=g).to(torch.bfloat16).cuda()
            outs = []
            for L in (release, debug):
                def run():
                    cache = tq.alloc_cache(2, 2, t_cap, D, kb, vb)
                    tq.tq_encode_kv(k, v, kb, ks, vb, cache, t_off=t_cap - T)
                    dec = [tq.tq_decode_kv(cache, t_cap, kb, ks, vb, out_dtype=dt) for dt in (torch.bfloat16,
                                                                                           torch.float32)]
                    rot = tq.tq_decode_kv_rotated(cache, t_cap, kb, ks, vb, out_dtype=torch.bfloat16)
                    un = tq.tq_unrotate(rot[1])
                    return cache, dec, rot, un
                outs.append(_with(L, run))
            (c0, d0, r0, u0), (c1, d1, r1, u1) = outs
            g0, g1 = cache_to_numpy(c0), cache_to_numpy(c1)
            for name in g0:
                assert np.array_equal(g0[name], g1[name]), name
            for a, b in zip(d0 + [r0] + [u0], d1 + [r1] + [u1]):
                for x, y in zip(a if isinstance(a, tuple) else (a,), b if isinstance(b, tuple) else (b,)):
                    assert np.array_equal(_bytes(x), _bytes(y))
    assert debug.tq_device_status(None) == 0
    assert release.tq_device_status(None) == 0


@pytest.mark.parametrize("D", [128, 512])
def test_attention_matches_release(libs, D):
    release, debug = libs
    g = torch.Generator().manual_seed(7 + D)
    B, Hkv, G, T = 3, 2, 4, 100
    t_cap = 112
    k = torch.randn((B, Hkv, T, D), generator=g).to(torch.bfloat16).cuda()
    v = torch.randn((B, Hkv, T, D), generator=g).to(torch.bfloat16).cuda()
    q = torch.randn((B, Hkv * G, 1, D), generator=g).to(torch.bfloat16).cuda()
    lp = torch.tensor([0, 7, 40], dtype=torch.int32, device="cuda")
    cache = tq.alloc_cache(B, Hkv, t_cap, D, 8, 3)
    tq.tq_encode_kv(k, v, 8, True, 3, cache)
    outs = [_with(L, lambda: tq.tq_decode_attention(q, cache, T, 8, True, 3, left_pad=lp,
                                                    out_dtype=torch.float32)) for L in (release, debug)]
    assert np.array_equal(_bytes(outs[0]), _bytes(outs[1]))
    assert debug.tq_device_status(None) == 0
