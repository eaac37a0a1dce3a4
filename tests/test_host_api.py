"""CPU-only checks of the C ABI: the library loads, exports every symbol the
header declares, and rejects bad arguments before launching anything.

Every call here fails host validation (or launches nothing), so no GPU and no
device pointer is needed; the fake pointers are never dereferenced.
"""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "kvattn.h")


@pytest.fixture(scope="module")
def kv():
    import kv_cache_attention_rope_gb300 as kv

    return kv


def header_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(kvattn_[a-z0-9_]+)\s*\(", text)))


def test_library_exports_every_declared_function(kv):
    names = header_functions()
    assert len(names) >= 18
    for n in names:
        assert hasattr(kv.lib, n), f"{n} declared in kvattn.h but not exported"
    assert sorted(kv.EXPORTED) == names


def test_version_and_status_strings(kv):
    assert kv.version() == 1
    for code in range(8):
        assert kv.status_string(code) and kv.status_string(code) != "unknown status"
    assert kv.status_string(99) == "unknown status"


FAKE = ctypes.c_void_p(0x7F0000001000)  # never dereferenced: every call below fails validation


def _cache(kv, nb=8, bs=16, k=FAKE, v=FAKE):
    return kv.CacheDesc(k, v, nb, bs)


def _rope(kv, cfg, cache, T=1, nseq=1, maxb=1, q=FAKE):
    return kv.lib.kvattn_rope_append(ctypes.byref(cfg) if cfg is not None else None,
                                     ctypes.byref(cache) if cache is not None else None,
                                     q, FAKE, FAKE, FAKE, FAKE, FAKE, nseq, maxb, T, None)


def test_rope_append_validation(kv):
    E = kv.STATUS_CODE
    good = kv.make_config(8, 2, 128, kv.BF16)
    assert _rope(kv, None, _cache(kv)) == E["KVATTN_ERR_INVALID_ARG"]
    assert _rope(kv, good, None) == E["KVATTN_ERR_INVALID_ARG"]
    assert _rope(kv, good, _cache(kv), T=-1) == E["KVATTN_ERR_INVALID_ARG"]
    assert _rope(kv, good, _cache(kv), nseq=0) == E["KVATTN_ERR_INVALID_ARG"]
    assert _rope(kv, kv.make_config(8, 2, 96, kv.BF16), _cache(kv)) == E["KVATTN_ERR_UNSUPPORTED"]
    assert _rope(kv, kv.make_config(9, 3, 128, kv.BF16), _cache(kv)) == E["KVATTN_ERR_UNSUPPORTED"]  # G=3
    assert _rope(kv, kv.make_config(32, 2, 128, kv.BF16), _cache(kv)) == E["KVATTN_ERR_UNSUPPORTED"]  # G=16
    assert _rope(kv, kv.make_config(8, 3, 128, kv.BF16), _cache(kv)) == E["KVATTN_ERR_UNSUPPORTED"]  # 8 % 3
    assert _rope(kv, kv.make_config(8, 2, 128, 7), _cache(kv)) == E["KVATTN_ERR_INVALID_ARG"]  # dtype
    assert _rope(kv, kv.make_config(8, 2, 128, kv.BF16, rope_base=-1.0), _cache(kv)) == E["KVATTN_ERR_INVALID_ARG"]
    assert _rope(kv, good, _cache(kv, nb=0)) == E["KVATTN_ERR_INVALID_ARG"]
    assert _rope(kv, good, _cache(kv, k=None)) == E["KVATTN_ERR_INVALID_ARG"]
    assert _rope(kv, good, _cache(kv, k=ctypes.c_void_p(0x7F0000001004))) == E["KVATTN_ERR_INVALID_ARG"]
    # a paged cache needs 16-token multiples for its blocks
    assert _rope(kv, good, _cache(kv, bs=24), maxb=2) == E["KVATTN_ERR_INVALID_ARG"]
    assert _rope(kv, good, _cache(kv), maxb=0) == E["KVATTN_ERR_INVALID_ARG"]
    # no tokens: nothing to do, nothing launched
    assert _rope(kv, good, _cache(kv), T=0) == E["KVATTN_OK"]
    # null q with work to do
    assert _rope(kv, good, _cache(kv), q=None) == E["KVATTN_ERR_INVALID_ARG"]


def _rope_strided(kv, cfg, cache, qs, ks, vs, T=4, q=FAKE, q_out=None):
    return kv.lib.kvattn_rope_append_strided(ctypes.byref(cfg), ctypes.byref(cache), q, qs, FAKE, ks, FAKE, vs,
                                             q_out, FAKE, FAKE, FAKE, 1, 1, T, None)


def test_rope_append_strided_validation(kv):
    E = kv.STATUS_CODE
    cfg = kv.make_config(8, 2, 128, kv.BF16)
    fused = (8 + 2 * 2) * 128
    c = _cache(kv)
    # the fused-QKV strides and the dense strides pass host validation (T = 0 launches nothing)
    assert _rope_strided(kv, cfg, c, fused, fused, fused, T=0) == E["KVATTN_OK"]
    assert _rope_strided(kv, cfg, c, 8 * 128, 2 * 128, 2 * 128, T=0) == E["KVATTN_OK"]
    # a stride below its row length would overlap rows
    assert _rope_strided(kv, cfg, c, 8 * 128 - 8, fused, fused, T=0) == E["KVATTN_ERR_INVALID_ARG"]
    assert _rope_strided(kv, cfg, c, fused, 2 * 128 - 8, fused, T=0) == E["KVATTN_ERR_INVALID_ARG"]
    assert _rope_strided(kv, cfg, c, fused, fused, 1, T=0) == E["KVATTN_ERR_INVALID_ARG"]
    # rows must start on 16-byte boundaries: bf16 strides in multiples of 8, f32 in multiples of 4
    assert _rope_strided(kv, cfg, c, fused + 4, fused, fused, T=0) == E["KVATTN_ERR_INVALID_ARG"]
    assert _rope_strided(kv, cfg, c, fused, fused, fused + 8, T=0) == E["KVATTN_OK"]
    f32 = kv.make_config(8, 2, 128, kv.F32)
    assert _rope_strided(kv, f32, c, fused + 4, fused, fused, T=0) == E["KVATTN_OK"]
    assert _rope_strided(kv, f32, c, fused + 2, fused, fused, T=0) == E["KVATTN_ERR_INVALID_ARG"]
    # strides whose byte offsets would overflow
    assert _rope_strided(kv, cfg, c, 2 ** 62, fused, fused) == E["KVATTN_ERR_INVALID_ARG"]
    # misaligned base pointer, null q
    assert _rope_strided(kv, cfg, c, fused, fused, fused, q=ctypes.c_void_p(0x7F0000001008)) == \
        E["KVATTN_ERR_INVALID_ARG"]
    assert _rope_strided(kv, cfg, c, fused, fused, fused, q=None) == E["KVATTN_ERR_INVALID_ARG"]
    assert _rope_strided(kv, cfg, c, fused, fused, fused, q_out=ctypes.c_void_p(0x7F0000002004)) == \
        E["KVATTN_ERR_INVALID_ARG"]


def test_split_qkv_views(kv):
    import torch

    T, hq, hkv, d = 5, 8, 2, 64
    qkv = torch.arange(T * (hq + 2 * hkv) * d, dtype=torch.float32).view(T, -1)
    q, k, v = kv.split_qkv(qkv, hq, hkv, d)
    assert q.shape == (T, hq, d) and k.shape == (T, hkv, d) and v.shape == (T, hkv, d)
    row = (hq + 2 * hkv) * d
    assert q.stride() == k.stride() == v.stride() == (row, d, 1)
    assert k.data_ptr() - q.data_ptr() == hq * d * 4
    assert v.data_ptr() - k.data_ptr() == hkv * d * 4
    # the views alias the fused buffer (no copy)
    assert torch.equal(torch.cat([q.reshape(T, -1), k.reshape(T, -1), v.reshape(T, -1)], 1), qkv)
    with pytest.raises(ValueError):
        kv.split_qkv(qkv[:, :-d], hq, hkv, d)


def test_layered_cache_placement(kv):
    """One block id names 2 * L regions: layer l's K area is region 2l, its V area 2l + 1."""
    E = kv.STATUS_CODE
    cfg = kv.make_config(32, 8, 128, kv.BF16)
    L, nb, bs = 4, 1000, 16
    region = nb * 8 * bs * 128 * 2
    assert kv.lib.kvattn_layered_cache_bytes(ctypes.byref(cfg), L, nb, bs) == 2 * L * region
    f32 = kv.make_config(12, 12, 64, kv.F32)
    assert kv.lib.kvattn_layered_cache_bytes(ctypes.byref(f32), 24, 3, 1025) == 2 * 24 * 3 * 12 * 1025 * 64 * 4
    base = 0x7F0000000000
    for layer in range(L):
        out = kv.CacheDesc()
        assert kv.lib.kvattn_layer_cache(ctypes.byref(cfg), ctypes.c_void_p(base), L, nb, bs, layer,
                                         ctypes.byref(out)) == E["KVATTN_OK"]
        assert out.k_pool == base + 2 * layer * region
        assert out.v_pool == base + (2 * layer + 1) * region
        assert (out.num_blocks, out.block_size) == (nb, bs)

    def call(layer=0, b=base, n=nb, L_=L, c=cfg, out=True):
        o = kv.CacheDesc()
        return kv.lib.kvattn_layer_cache(ctypes.byref(c), ctypes.c_void_p(b), L_, n, bs, layer,
                                         ctypes.byref(o) if out else None)

    assert call(layer=-1) == E["KVATTN_ERR_INVALID_ARG"]
    assert call(layer=L) == E["KVATTN_ERR_INVALID_ARG"]
    assert call(b=base + 8) == E["KVATTN_ERR_INVALID_ARG"]
    assert call(b=0) == E["KVATTN_ERR_INVALID_ARG"]
    assert call(n=0) == E["KVATTN_ERR_INVALID_ARG"]
    assert call(L_=0) == E["KVATTN_ERR_INVALID_ARG"]
    assert call(out=False) == E["KVATTN_ERR_INVALID_ARG"]
    assert call(c=kv.make_config(32, 8, 96, kv.BF16)) == E["KVATTN_ERR_UNSUPPORTED"]
    # sizes past int64 are refused, not wrapped
    assert kv.lib.kvattn_layered_cache_bytes(ctypes.byref(cfg), 1 << 20, 1 << 40, bs) == 0
    assert call(n=1 << 40, L_=1 << 20) == E["KVATTN_ERR_INVALID_ARG"]


def test_copy_blocks_validation(kv):
    E = kv.STATUS_CODE
    cfg = kv.make_config(8, 2, 128, kv.BF16)
    c = _cache(kv)
    cp = kv.lib.kvattn_copy_blocks
    assert cp(ctypes.byref(cfg), ctypes.byref(c), FAKE, FAKE, 0, None) == E["KVATTN_OK"]      # nothing launched
    assert cp(ctypes.byref(cfg), ctypes.byref(c), FAKE, FAKE, -1, None) == E["KVATTN_ERR_INVALID_ARG"]
    assert cp(ctypes.byref(cfg), ctypes.byref(c), None, FAKE, 2, None) == E["KVATTN_ERR_INVALID_ARG"]
    assert cp(ctypes.byref(cfg), None, FAKE, FAKE, 2, None) == E["KVATTN_ERR_INVALID_ARG"]
    assert cp(ctypes.byref(kv.make_config(8, 2, 80, kv.BF16)), ctypes.byref(c), FAKE, FAKE, 2, None) == \
        E["KVATTN_ERR_UNSUPPORTED"]
    lay = kv.lib.kvattn_copy_blocks_layered
    assert lay(ctypes.byref(cfg), FAKE, 4, 100, 16, FAKE, FAKE, 0, None) == E["KVATTN_OK"]
    assert lay(ctypes.byref(cfg), FAKE, 0, 100, 16, FAKE, FAKE, 1, None) == E["KVATTN_ERR_INVALID_ARG"]
    assert lay(ctypes.byref(cfg), ctypes.c_void_p(0x7F0000001008), 4, 100, 16, FAKE, FAKE, 1, None) == \
        E["KVATTN_ERR_INVALID_ARG"]
    assert lay(ctypes.byref(cfg), FAKE, 4, 100, 16, FAKE, None, 1, None) == E["KVATTN_ERR_INVALID_ARG"]


def test_fp8_cache_validation(kv):
    E = kv.STATUS_CODE
    cfg = kv.make_config(32, 8, 128, kv.BF16)

    def c8(bs=16, pool=FAKE):
        return kv.CacheFP8Desc(pool, 8, bs)

    def dec(c, config=cfg, B=2, out=FAKE):
        return kv.lib.kvattn_decode_fp8(ctypes.byref(config), ctypes.byref(c) if c is not None else None, FAKE,
                                        FAKE, 4, FAKE, B, 64, 0, out, FAKE, 1 << 20, None)

    def rope(c, config=cfg, T=1):
        return kv.lib.kvattn_rope_append_fp8(ctypes.byref(config), ctypes.byref(c) if c is not None else None,
                                             FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1, 4, T, None)

    assert dec(None) == E["KVATTN_ERR_INVALID_ARG"]
    assert dec(c8(pool=None)) == E["KVATTN_ERR_INVALID_ARG"]
    assert dec(c8(pool=ctypes.c_void_p(0x7F0000001004))) == E["KVATTN_ERR_INVALID_ARG"]
    assert dec(c8(bs=24)) == E["KVATTN_ERR_INVALID_ARG"]                      # pages of 16 rows
    assert dec(c8(), config=kv.make_config(32, 8, 64, kv.BF16)) == E["KVATTN_ERR_UNSUPPORTED"]
    assert dec(c8(), config=kv.make_config(16, 8, 128, kv.BF16)) == E["KVATTN_ERR_UNSUPPORTED"]  # group 2
    assert dec(c8(), config=kv.make_config(32, 8, 128, kv.F32)) == E["KVATTN_ERR_UNSUPPORTED"]
    assert dec(c8(), B=0) == E["KVATTN_OK"]
    assert dec(c8(), out=None) == E["KVATTN_ERR_INVALID_ARG"]
    assert rope(None) == E["KVATTN_ERR_INVALID_ARG"]
    assert rope(c8(pool=None)) == E["KVATTN_ERR_INVALID_ARG"]
    assert rope(c8(bs=24)) == E["KVATTN_ERR_INVALID_ARG"]
    assert rope(c8(), config=kv.make_config(12, 12, 64, kv.BF16)) == E["KVATTN_ERR_UNSUPPORTED"]
    assert rope(c8(), config=kv.make_config(32, 8, 128, kv.F32)) == E["KVATTN_ERR_UNSUPPORTED"]
    assert rope(c8(), T=0) == E["KVATTN_OK"]


def _decode(kv, cfg, cache, B=2, maxlen=64, splits=0, ws=None, ws_bytes=0, out=FAKE, maxb=4):
    return kv.lib.kvattn_decode(ctypes.byref(cfg), ctypes.byref(cache), FAKE, FAKE, maxb, FAKE, B, maxlen,
                                splits, out, ws, ws_bytes, None)


def test_decode_validation_and_workspace(kv):
    E = kv.STATUS_CODE
    cfg = kv.make_config(32, 8, 128, kv.BF16)
    c = _cache(kv)
    assert _decode(kv, cfg, c, B=-1) == E["KVATTN_ERR_INVALID_ARG"]
    assert _decode(kv, cfg, c, splits=-1) == E["KVATTN_ERR_INVALID_ARG"]
    assert _decode(kv, cfg, c, B=0) == E["KVATTN_OK"]
    assert _decode(kv, cfg, c, out=None) == E["KVATTN_ERR_INVALID_ARG"]
    assert _decode(kv, kv.make_config(32, 8, 80, kv.BF16), c) == E["KVATTN_ERR_UNSUPPORTED"]
    assert _decode(kv, cfg, c, B=10000) == E["KVATTN_ERR_UNSUPPORTED"]
    # more than one split needs a workspace of the advertised size
    need = kv.decode_workspace_size(cfg, 2, 4096, 4)
    assert need >= 2 * 32 * 4 * (128 + 2) * 4
    assert kv.decode_num_splits(cfg, 2, 4096, 4) == 4
    assert _decode(kv, cfg, c, maxlen=4096, splits=4, ws=None) == E["KVATTN_ERR_WORKSPACE_TOO_SMALL"]
    assert _decode(kv, cfg, c, maxlen=4096, splits=4, ws=FAKE, ws_bytes=need - 1) == \
        E["KVATTN_ERR_WORKSPACE_TOO_SMALL"]
    # misaligned workspace
    assert _decode(kv, cfg, c, maxlen=4096, splits=4, ws=ctypes.c_void_p(0x7F0000001010), ws_bytes=need) == \
        E["KVATTN_ERR_INVALID_ARG"]


def test_decode_plan_properties(kv):
    cfg = kv.make_config(32, 8, 128, kv.BF16)
    # explicit split requests are honoured (at most that many chunks)
    for maxlen in (1, 15, 16, 17, 1000, 8193):
        for s in (1, 2, 3, 7):
            n = kv.decode_num_splits(cfg, 4, maxlen, s)
            assert 1 <= n <= s
    # a segment cut where two CTA ranges meet has at most (tiles + 1) pieces
    assert kv.decode_num_splits(cfg, 4, 16, 8) == 2
    assert kv.decode_num_splits(cfg, 4, 16, 1) == 1     # 1 = whole segments, no workspace
    assert kv.decode_workspace_size(cfg, -1, 10, 0) == 0
    # workspace grows with the batch
    assert kv.decode_workspace_size(cfg, 64, 4096, 4) > kv.decode_workspace_size(cfg, 8, 4096, 4)


def test_prefill_validation(kv):
    E = kv.STATUS_CODE

    def call(cfg, cache, n=2, maxq=512, tq=1024, out=FAKE):
        return kv.lib.kvattn_prefill_chunk(ctypes.byref(cfg), ctypes.byref(cache), FAKE, FAKE, FAKE, FAKE, 4,
                                           n, maxq, tq, out, None)

    cfg = kv.make_config(32, 8, 128, kv.BF16)
    assert call(kv.make_config(32, 8, 128, kv.F32), _cache(kv)) == E["KVATTN_ERR_UNSUPPORTED"]
    assert call(kv.make_config(32, 8, 80, kv.BF16), _cache(kv)) == E["KVATTN_ERR_UNSUPPORTED"]
    assert call(kv.make_config(12, 12, 64, kv.BF16), _cache(kv), n=0) == E["KVATTN_OK"]   # GPT-2 shape accepted
    assert call(cfg, _cache(kv), n=-1) == E["KVATTN_ERR_INVALID_ARG"]
    assert call(cfg, _cache(kv), n=0) == E["KVATTN_OK"]
    assert call(cfg, _cache(kv), out=None) == E["KVATTN_ERR_INVALID_ARG"]


def test_prefill_fp8_validation_and_workspace(kv):
    """kvattn_prefill_chunk_fp8's host checks and its workspace formula: a bf16
    copy of ceil(max_kv_tokens / block_size) + num_chunks blocks (K and V),
    the copy's block table, owners and first blocks, each part 1 KB aligned,
    plus 1 KB of slack for the base alignment."""
    E = kv.STATUS_CODE
    cfg = kv.make_config(32, 8, 128, kv.BF16)

    def size(config=cfg, bs=16, maxb=64, n=4, kvt=4096):
        return kv.lib.kvattn_prefill_fp8_workspace_size(ctypes.byref(config), bs, maxb, n, kvt)

    def call(c, config=cfg, n=2, kvt=1000, ws=FAKE, ws_bytes=1 << 40, out=FAKE):
        return kv.lib.kvattn_prefill_chunk_fp8(ctypes.byref(config), ctypes.byref(c) if c is not None else None,
                                               FAKE, FAKE, FAKE, FAKE, 64, n, 512, 1024, kvt, out, ws, ws_bytes,
                                               None)

    def up(x):
        return -(-x // 1024) * 1024

    nb = -(-4096 // 16) + 4
    want = up(5 * 8) + up(nb * 4) + up(4 * 64 * 4) + 2 * up(nb * 8 * 16 * 128 * 2) + 1024
    assert size() == want
    assert size(config=kv.make_config(32, 8, 128, kv.F32)) == 0
    assert size(config=kv.make_config(12, 12, 64, kv.BF16)) == 0
    assert size(bs=24) == 0 and size(maxb=0) == 0 and size(n=-1) == 0 and size(kvt=-1) == 0
    c8 = kv.CacheFP8Desc(FAKE, 8, 16)
    assert call(None) == E["KVATTN_ERR_INVALID_ARG"]
    assert call(kv.CacheFP8Desc(None, 8, 16)) == E["KVATTN_ERR_INVALID_ARG"]
    assert call(kv.CacheFP8Desc(FAKE, 8, 24)) == E["KVATTN_ERR_INVALID_ARG"]
    assert call(c8, config=kv.make_config(32, 8, 128, kv.F32)) == E["KVATTN_ERR_UNSUPPORTED"]
    assert call(c8, config=kv.make_config(12, 12, 64, kv.BF16)) == E["KVATTN_ERR_UNSUPPORTED"]
    assert call(c8, n=0) == E["KVATTN_OK"]
    assert call(c8, n=-1) == E["KVATTN_ERR_INVALID_ARG"]
    assert call(c8, kvt=-1) == E["KVATTN_ERR_INVALID_ARG"]
    assert call(c8, ws=None) == E["KVATTN_ERR_INVALID_ARG"]
    assert call(c8, out=None) == E["KVATTN_ERR_INVALID_ARG"]
    need = kv.lib.kvattn_prefill_fp8_workspace_size(ctypes.byref(cfg), 16, 64, 2, 1000)
    assert call(c8, ws_bytes=need - 1) == E["KVATTN_ERR_WORKSPACE_TOO_SMALL"]


def test_get_device_status_needs_out(kv):
    assert kv.lib.kvattn_get_device_status(None, None) == kv.STATUS_CODE["KVATTN_ERR_INVALID_ARG"]


def test_binding_rejects_cpu_tensors(kv):
    import torch

    cfg = kv.make_config(4, 4, 64, kv.F32)
    t = torch.zeros(4, 4, 1, 64)
    with pytest.raises(ValueError):
        kv.Cache(t, t)
