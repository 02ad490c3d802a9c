"""The C ABI library without a GPU: it builds, loads, exports every function
include/tq.h declares, and rejects bad arguments on the host before any CUDA
call (so these checks run anywhere). Every call below is invalid by
construction; none can reach a kernel launch.
"""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "tq.h")

OK, INVALID, HEAD_DIM, BITS, ALIGN, DTYPE, CUDA, TIMEOUT = range(8)


@pytest.fixture(scope="module")
def L():
    from turboquant_kv_cache_tq_gb300 import build

    build.build()
    import turboquant_kv_cache_tq_gb300 as tq

    return tq.lib()


def _declared():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"\b(tq_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_abi():
    names = _declared()
    for n in ("tq_packed_dim", "tq_encode_kv", "tq_decode_kv", "tq_decode_kv_rotated", "tq_unrotate",
              "tq_lloyd_max_index", "tq_decode_attention", "tq_decode_attention_workspace_size",
              "tq_decode_attention_noalloc", "tq_cache_assemble", "tq_status_string"):
        assert n in names


def test_library_exports_every_declared_symbol(L):
    lib = ctypes.CDLL(L._name)
    for name in _declared():
        assert hasattr(lib, name), name


def test_packed_dim(L):
    for d in (64, 128, 256, 512):
        for b in (2, 3, 4, 5, 8):
            assert L.tq_packed_dim(d, b) == d * b // 8
    assert L.tq_packed_dim(512, 5) == 320 and L.tq_packed_dim(128, 3) == 48
    assert L.tq_packed_dim(3, 3) == -ALIGN and L.tq_packed_dim(5, 5) == -ALIGN
    assert L.tq_packed_dim(-1, 3) == -INVALID and L.tq_packed_dim(64, 0) == -INVALID


def test_status_strings(L):
    for s in range(8):
        assert L.tq_status_string(s).startswith(b"TQ_")
    assert b"unknown" in L.tq_status_string(99)


def _enc(L, D=128, T=4, kb=8, ks=1, vb=3, dtype=1, t_cap=None, t_off=0, ptrs=None, B=1, H=2):
    t_cap = T if t_cap is None else t_cap
    ptrs = ptrs if ptrs is not None else [0] * 7
    return L.tq_encode_kv(ptrs[0], ptrs[1], dtype, B, H, T, D, kb, ks, vb, *ptrs[2:], t_cap, t_off, None)


def _dec(L, D=128, T=4, kb=8, ks=1, vb=3, dtype=1, t_cap=None, ptrs=None, B=1, H=2):
    t_cap = T if t_cap is None else t_cap
    ptrs = ptrs if ptrs is not None else [0] * 7
    return L.tq_decode_kv(*ptrs[:5], B, H, T, D, t_cap, kb, ks, vb, ptrs[5], ptrs[6], dtype, None)


def _dec_rot(L, D=128, T=4, kb=8, ks=1, vb=3, dtype=1, t_cap=None, ptrs=None, B=1, H=2):
    t_cap = T if t_cap is None else t_cap
    ptrs = ptrs if ptrs is not None else [0] * 7
    return L.tq_decode_kv_rotated(*ptrs[:5], B, H, T, D, t_cap, kb, ks, vb, ptrs[5], ptrs[6], dtype, None)


@pytest.mark.parametrize("fn", [_enc, _dec, _dec_rot])
def test_argument_checks(L, fn):
    assert fn(L, D=96) == HEAD_DIM and fn(L, D=32) == HEAD_DIM and fn(L, D=1024) == HEAD_DIM
    assert fn(L, vb=6) == BITS and fn(L, vb=1) == BITS
    assert fn(L, kb=3, ks=0) == BITS and fn(L, kb=4, ks=1) == BITS and fn(L, kb=16, ks=0) == BITS
    assert fn(L, dtype=7) == DTYPE
    assert fn(L, T=-1) == INVALID and fn(L, B=-2) == INVALID
    assert fn(L, T=8, t_cap=4) == INVALID
    # null buffers with work to do
    assert fn(L) == INVALID
    # empty work is a no-op, even with null buffers
    assert fn(L, T=0) == OK and fn(L, B=0) == OK and fn(L, H=0) == OK


def test_encode_offset_checks(L):
    assert _enc(L, T=4, t_cap=5, t_off=2) == INVALID
    assert _enc(L, T=4, t_cap=8, t_off=-1) == INVALID
    assert _enc(L, T=0, t_cap=8, t_off=8) == OK


def test_misaligned_buffers_rejected(L):
    # one misaligned pointer among non-null ones: the check fires before launch
    base = 1 << 20
    ptrs = [base + 256 * i for i in range(7)]
    for i in range(7):
        bad = list(ptrs)
        bad[i] += 8
        assert _enc(L, ptrs=bad) == ALIGN
        assert _dec(L, ptrs=bad) == ALIGN
        assert _dec_rot(L, ptrs=bad) == ALIGN


def test_size_overflow_rejected(L):
    assert _enc(L, B=1 << 20, H=1 << 20, T=1 << 12) == INVALID
    assert _dec(L, T=1 << 31, t_cap=1 << 31) == INVALID
    # rows just past 2^31 - 1 - 2^24 (kernel item indices keep 2^24 of headroom)
    over = (1 << 31) - (1 << 24)
    assert _enc(L, H=1, T=over, t_cap=over) == INVALID
    assert _dec(L, H=1, T=over, t_cap=over) == INVALID
    assert L.tq_unrotate(1 << 20, 0, over, 128, 1 << 21, None) == INVALID


def test_unrotate_checks(L):
    assert L.tq_unrotate(None, 1, 0, 128, None, None) == OK
    assert L.tq_unrotate(None, 1, -1, 128, None, None) == INVALID
    assert L.tq_unrotate(None, 1, 4, 96, None, None) == HEAD_DIM
    assert L.tq_unrotate(None, 3, 4, 128, None, None) == DTYPE
    assert L.tq_unrotate(None, 0, 4, 128, None, None) == INVALID
    assert L.tq_unrotate(1 << 20, 0, 4, 128, None, None) == INVALID
    assert L.tq_unrotate(1 << 20 | 8, 0, 4, 128, 1 << 21, None) == ALIGN
    assert L.tq_unrotate(1 << 20, 0, 4, 128, (1 << 21) + 4, None) == ALIGN
    assert L.tq_unrotate(1 << 20, 0, 1 << 31, 128, 1 << 21, None) == INVALID


def test_lloyd_max_index_checks(L):
    assert L.tq_lloyd_max_index(None, 0, 3, None, None) == OK
    assert L.tq_lloyd_max_index(None, 5, 6, None, None) == BITS
    assert L.tq_lloyd_max_index(None, -1, 3, None, None) == INVALID
    assert L.tq_lloyd_max_index(None, 5, 3, None, None) == INVALID
    assert L.tq_lloyd_max_index(1 << 20 | 2, 5, 3, 1 << 21, None) == ALIGN


def test_binding_fails_loudly_without_library(tmp_path, monkeypatch):
    import turboquant_kv_cache_tq_gb300 as tq

    monkeypatch.setattr(tq, "_lib", None)
    monkeypatch.setattr(tq, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="not built"):
        tq.lib()


def _attn(L, D=128, B=2, Hq=8, Hkv=2, Nq=1, T=20, t_cap=32, kb=8, ks=1, vb=3, dtype=1, ptrs=None,
          left_pad=None, ws_bytes=1 << 30):
    ptrs = ptrs if ptrs is not None else [0] * 8
    return L.tq_decode_attention(ptrs[0], B, Hq, Nq, *ptrs[1:6], Hkv, T, D, t_cap, kb, ks, vb, left_pad, 0.1,
                                 ptrs[6], dtype, ptrs[7], ws_bytes, None)


def test_attention_argument_checks(L):
    assert _attn(L, D=1024) == HEAD_DIM and _attn(L, D=96) == HEAD_DIM
    assert _attn(L, vb=6) == BITS and _attn(L, kb=4, ks=1) == BITS
    assert _attn(L, dtype=5) == DTYPE
    assert _attn(L, Hq=6, Hkv=4) == INVALID            # Hq not a multiple of Hkv
    assert _attn(L, Hq=16, Hkv=2, Nq=3) == INVALID      # 24 query rows per kv head
    assert _attn(L, Nq=0) == INVALID and _attn(L, T=-1) == INVALID
    assert _attn(L, T=40, t_cap=32) == INVALID
    assert _attn(L, t_cap=24) == ALIGN
    assert _attn(L) == INVALID                          # null buffers
    assert _attn(L, B=0) == OK
    base = 1 << 20
    ptrs = [base + 4096 * i for i in range(8)]
    for i in range(8):
        bad = list(ptrs)
        bad[i] += 8
        assert _attn(L, ptrs=bad) == ALIGN
    assert _attn(L, ptrs=ptrs, left_pad=base + 2) == ALIGN
    assert _attn(L, ptrs=ptrs, ws_bytes=16) == INVALID  # workspace too small


def test_attention_workspace_size(L):
    assert L.tq_decode_attention_workspace_size(2, 2, 100, 1024) == -HEAD_DIM
    assert L.tq_decode_attention_workspace_size(-1, 2, 100, 128) == -INVALID
    assert L.tq_decode_attention_workspace_size(2, 0, 100, 128) == -INVALID
    rec = 16 * (128 + 2) * 4
    # many heads: one record per split block (at most 8 per SM) and per
    # (batch, kv head), nothing else (a head has few records: one combine
    # block per row tile)
    big = L.tq_decode_attention_workspace_size(64, 64, 100, 128)
    sms8 = big // rec - 64 * 64  # 8 x SMs
    assert big % rec == 0 and sms8 > 0 and sms8 % 8 == 0
    assert L.tq_decode_attention_workspace_size(64, 65, 100, 128) == big + 64 * rec
    # few heads: the records, then the combine's partial sums (row tiles of
    # 1024 / D rows for up to 16 query rows per kv head, 32 x 34 floats per
    # chunk of 32 records, at most 8 chunks) and one ticket counter per tile
    for B, H, D in [(2, 2, 128), (1, 1, 512), (4, 4, 256), (2, 2, 64), (3, 5, 128)]:
        bhkv = B * H
        recs = (sms8 + bhkv) * 16 * (D + 2) * 4
        chunks = min(8, max(1, -(-(sms8 // bhkv + 2) // 32)))
        tiles = -(-16 * bhkv * D // 1024)
        extra = tiles * chunks * 32 * 34 * 4 + -(-tiles * 4 // 16) * 16 if chunks > 1 else 0
        assert L.tq_decode_attention_workspace_size(B, H, 100, D) == recs + extra, (B, H, D)


def test_cache_assemble_checks(L):
    import turboquant_kv_cache_tq_gb300 as tq

    base = 1 << 20
    d = [base + 4096 * i for i in range(5)]

    def call(rows, n=1, H=2, D=128, kb=8, vb=3, t_cap=16, width=8, dst=d):
        arr = (tq.TQRowSource * max(len(rows), 1))(*rows)
        return L.tq_cache_assemble(ctypes.cast(arr, ctypes.c_void_p), n, H, D, kb, vb, *dst, t_cap, width, None)

    src = [base + 8192 * i for i in range(5)]
    ok_row = tq.TQRowSource(*src, 1, 0, 16, 0, 8)
    assert call([ok_row], D=96) == HEAD_DIM
    assert call([ok_row], kb=3) == BITS and call([ok_row], vb=6) == BITS
    assert call([ok_row], width=20) == INVALID                                   # window past capacity
    assert call([tq.TQRowSource(*src, 1, 0, 16, 10, 8)]) == INVALID             # source range past t_cap
    assert call([tq.TQRowSource(*src, 1, 1, 16, 0, 8)]) == INVALID              # b >= B
    assert call([tq.TQRowSource(*src, 1, 0, 16, 0, 9)]) == INVALID              # len > width
    assert call([tq.TQRowSource(None, *src[1:], 1, 0, 16, 0, 8)]) == INVALID    # null source
    assert call([tq.TQRowSource(src[0] + 4, *src[1:], 1, 0, 16, 0, 8)]) == ALIGN
    assert call([ok_row], dst=[d[0] + 8] + d[1:]) == ALIGN
    assert call([ok_row], n=0) == OK and call([ok_row], width=0) == OK


def test_lloyd_fit_checks(L):
    """Host checks of the Lloyd fit entry points (no device work is reached)."""
    base = 1 << 20
    x, init, c, b, ws = base, base + 4096, base + 8192, base + 12288, base + 16384
    need = L.tq_lloyd_max_fit_workspace_size(16)
    assert need == 64 + 48 * 16
    assert L.tq_lloyd_max_fit_workspace_size(3) == -INVALID
    assert L.tq_lloyd_max_fit(x, 100, 3, 1, init, c, b, ws, need, None) == INVALID      # not a power of two
    assert L.tq_lloyd_max_fit(x, 100, 16, 1, init, c, b, ws, need - 1, None) == INVALID  # workspace too small
    assert L.tq_lloyd_max_fit(x + 2, 100, 16, 1, init, c, b, ws, need, None) == ALIGN
    assert L.tq_lloyd_max_fit(x, 100, 16, 1, init, c, b, ws + 4, need, None) == ALIGN
    assert L.tq_lloyd_max_fit_bounded(x, 100, 16, 1, init, c, b, ws, need, -1, -1, None) == INVALID
    assert L.tq_lloyd_max_fit_bounded(x, 100, 16, 1, init, c, b, ws, need, 1 << 32, -1, None) == INVALID
    assert L.tq_lloyd_max_fit_bounded(x, 100, 16, 1, init, c, b, ws, need, 100, -2, None) == INVALID
    assert L.tq_lloyd_max_fit_status(None, None) == INVALID
    assert L.tq_lloyd_max_fit_status(ws + 8, None) == ALIGN
