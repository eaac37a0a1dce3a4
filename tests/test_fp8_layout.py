"""The fp8 page packer and unpacker the GPU tests use, checked element by
element against the byte layout kvattn.h states for kvattn_cache_fp8 (CPU
only), so that a mistake in the test helpers cannot hide one in the kernels."""
import numpy as np

from test_gpu_fp8 import pack_pages, unpack_rows


def _swz(r):
    return (r & 1) | ((r >> 1) & 6)


def test_pages_follow_the_documented_byte_layout():
    g = np.random.default_rng(11)
    nb, hkv, bs, D = 3, 2, 32, 128
    ck = g.integers(0, 256, (nb, hkv, bs, D)).astype(np.uint8)
    cv = g.integers(0, 256, (nb, hkv, bs, D)).astype(np.uint8)
    sk = g.random((nb, hkv, bs)).astype(np.float32)
    sv = g.random((nb, hkv, bs)).astype(np.float32)
    pages = pack_pages(ck, sk, cv, sv)
    assert pages.shape == (nb, hkv, bs // 16, 4224)
    for b in range(nb):
        for h in range(hkv):
            for t in range(bs):
                pg, r = pages[b, h, t // 16], t % 16
                for c in range(8):                     # K: chunk c of token r at r*128 + 16*(c ^ s(r))
                    o = r * 128 + 16 * (c ^ _swz(r))
                    assert np.array_equal(pg[o:o + 16], ck[b, h, t, 16 * c:16 * c + 16])
                for d in (0, 1, 63, 127):              # V transposed: dim d of token r at 2048 + 16*d + r
                    assert pg[2048 + 16 * d + r] == cv[b, h, t, d]
                assert pg[4096 + 4 * r:4100 + 4 * r].view(np.float32)[0] == sk[b, h, t]
                assert pg[4160 + 4 * r:4164 + 4 * r].view(np.float32)[0] == sv[b, h, t]
    blk = np.repeat(np.arange(nb), bs)
    off = np.tile(np.arange(bs), nb)
    k2, s2, v2, t2 = unpack_rows(pages, blk, off)
    assert np.array_equal(k2, ck.transpose(0, 2, 1, 3).reshape(-1, hkv, D))
    assert np.array_equal(v2, cv.transpose(0, 2, 1, 3).reshape(-1, hkv, D))
    assert np.array_equal(s2, sk.transpose(0, 2, 1).reshape(-1, hkv))
    assert np.array_equal(t2, sv.transpose(0, 2, 1).reshape(-1, hkv))


def test_row_rotation_is_conflict_free_for_the_decode_loads():
    """The rotation s(r) puts the K words read together by one MMA (rows
    {0,1,4,5,8,9,12,13} or {2,3,6,7,10,11,14,15}, the same chunk, lanes q4
    0..3) in 32 distinct banks."""
    for rows in ([0, 1, 4, 5, 8, 9, 12, 13], [2, 3, 6, 7, 10, 11, 14, 15]):
        for kk in range(8):
            banks = {((r * 128 + 16 * (kk ^ _swz(r)) + 4 * q4) // 4) % 32 for r in rows for q4 in range(4)}
            assert len(banks) == 32
    # and the transposed V words (dim 8 nd + g4, tokens 4 q4 ..) likewise
    for nd in range(16):
        banks = {((2048 + 16 * (8 * nd + g4) + 4 * q4) // 4) % 32 for g4 in range(8) for q4 in range(4)}
        assert len(banks) == 32
