"""Randomised GPU parity over the configuration space, against the oracle,
with fixed seeds (so a failure reproduces): the codec (every head_dim, key
mode, value width and input dtype, ragged token counts, cache offsets and
capacities), the fused decode attention (head maps, query tokens, left pads,
capacities) and the batched row assembly. The acceptance rules are those of
the dedicated parity tests.
"""
import numpy as np
import pytest
import torch

import oracle
import turboquant_kv_cache_tq_gb300 as tq
from tests.gpu_common import cache_from_numpy, cache_to_numpy, check_roundtrip, require_gpu
from tests.test_gpu_attention import _bits, _vrot_max, compare_attention

pytestmark = pytest.mark.gpu

KEY_MODES = [(2, False), (4, False), (5, False), (8, False), (8, True)]


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def _rand(shape, dtype, gen, scale):
    return (torch.randn(shape, generator=gen) * scale).to(dtype).contiguous()


@pytest.mark.parametrize("seed", range(40))
def test_codec_random_configs(seed):
    rng = np.random.default_rng(1000 + seed)
    gen = torch.Generator().manual_seed(2000 + seed)
    D = int(rng.choice([64, 128, 256, 512]))
    kb, ks = KEY_MODES[rng.integers(len(KEY_MODES))]
    vb = int(rng.choice([2, 3, 4, 5, 8]))
    dtype = torch.bfloat16 if rng.random() < 0.7 else torch.float32
    B, H = int(rng.integers(1, 4)), int(rng.integers(1, 5))
    T = int(rng.integers(1, {64: 90, 128: 60, 256: 30, 512: 16}[D]))
    t_off = int(rng.integers(0, 5))
    t_cap = T + t_off + int(rng.integers(0, 4))
    scale = float(rng.choice([0.01, 1.0, 30.0]))
    k = _rand((B, H, T, D), dtype, gen, scale)
    v = _rand((B, H, T, D), dtype, gen, scale)
    check_roundtrip(k, v, kb, ks, vb, t_cap=t_cap, t_off=t_off)


@pytest.mark.parametrize("seed", range(30))
def test_attention_random_configs(seed):
    rng = np.random.default_rng(3000 + seed)
    gen = torch.Generator().manual_seed(4000 + seed)
    D = int(rng.choice([64, 128, 256]))
    kb, ks = KEY_MODES[rng.integers(len(KEY_MODES))]
    vb = int(rng.choice([2, 3, 4, 5, 8]))
    B, Hkv = int(rng.integers(1, 4)), int(rng.integers(1, 4))
    while True:
        G, Nq = int(rng.integers(1, 9)), int(rng.integers(1, 4))
        if G * Nq <= 16:
            break
    T = int(rng.integers(1, 400))
    t_cap = (T + 15) // 16 * 16 + 16 * int(rng.integers(0, 3))
    pads = [int(rng.integers(0, T + 1)) if rng.random() < 0.6 else 0 for _ in range(B)]
    k = _rand((B, Hkv, T, D), torch.bfloat16, gen, 1.0)
    v = _rand((B, Hkv, T, D), torch.bfloat16, gen, 1.0)
    rc = oracle.encode_kv(_bits(k), _bits(v), kb, ks, vb, t_cap=t_cap)
    q = _rand((B, Hkv * G, Nq, D), torch.bfloat16, gen, float(rng.choice([0.5, 1.0, 3.0])))
    lp = torch.tensor(pads, dtype=torch.int32, device="cuda")
    out_dtype = torch.float32 if rng.random() < 0.7 else torch.bfloat16
    got = tq.tq_decode_attention(q.cuda(), cache_from_numpy(rc), T, kb, ks, vb, left_pad=lp, out_dtype=out_dtype)
    torch.cuda.synchronize()
    want = oracle.decode_attention(_bits(q), rc, T, kb, ks, vb, left_pad=pads)
    vmax = _vrot_max(rc, T, kb, ks, vb)
    g = got.float().cpu().numpy()
    if out_dtype == torch.float32:
        compare_attention(g, want, vmax, G, "seed %d" % seed)
    else:  # bf16 output: the fp32 tolerance plus half a bf16 step of the value
        err = np.abs(g.astype(np.float64) - want)
        lim = 5e-6 * np.repeat(vmax, G, axis=1)[:, :, None, None] + np.abs(want) * 2.0 ** -8
        ok = np.isnan(want) | (err <= lim)
        assert np.all(ok), "seed %d: bf16 attention output off by more than rounding" % seed


@pytest.mark.parametrize("seed", range(12))
def test_assemble_random_plans(seed):
    rng = np.random.default_rng(5000 + seed)
    D = int(rng.choice([64, 128, 256, 512]))
    kb, _ = KEY_MODES[rng.integers(len(KEY_MODES))]
    vb = int(rng.choice([2, 3, 4, 5, 8]))
    H = int(rng.integers(1, 4))
    sources = []
    for i in range(int(rng.integers(1, 4))):
        Bs, tc = int(rng.integers(1, 4)), int(rng.integers(1, 40))
        c = {n: rng.integers(0, 256, size=a.shape, dtype=np.uint8).view(a.dtype) if a.dtype == np.uint8
             else rng.integers(0, 65536, size=a.shape, dtype=np.uint16)
             for n, a in oracle.alloc_cache(Bs, H, tc, D, kb, vb).items()}
        sources.append(c)
    width = int(rng.integers(1, 40))
    t_cap = width + int(rng.integers(0, 5))
    n_rows = int(rng.integers(1, 70))
    dev_src = [cache_from_numpy(c) for c in sources]
    plan, want_rows = [], []
    for _ in range(n_rows):
        if rng.random() < 0.1:
            plan.append(None)
            want_rows.append(None)
            continue
        si = int(rng.integers(len(sources)))
        c = sources[si]
        Bs, _, tc, _ = c["k_codes"].shape
        length = int(rng.integers(0, min(width, tc) + 1))
        t0 = int(rng.integers(0, tc - length + 1))
        b = int(rng.integers(Bs))
        plan.append((dev_src[si], b, t0, length))
        want_rows.append((si, b, t0, length))
    dst = tq.alloc_cache(n_rows, H, t_cap, D, kb, vb)
    for t in dst.values():
        t.view(torch.uint8).fill_(0x5A)
    tq.tq_cache_assemble(plan, dst, width)
    torch.cuda.synchronize()
    got = cache_to_numpy(dst)
    for name in got:
        for r, wr in enumerate(want_rows):
            row = got[name][r]
            length = 0 if wr is None else wr[3]
            assert np.all(row[:, :width - length].view(np.uint8) == 0), (seed, name, r)
            if length:
                si, b, t0, _ = wr
                assert np.array_equal(row[:, width - length:width], sources[si][name][b, :, t0:t0 + length])
            assert np.all(row[:, width:].view(np.uint8) == 0x5A), (seed, name, r)
