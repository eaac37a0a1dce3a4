"""GPU parity of the fp8 (e4m3) KV cache against the oracle.

Bar: rope_append_fp8 stores codes and scales bit-identical to
oracle.fp8.quantize_rows of the correctly rounded bf16 rotation of k (and of
the bf16 v), and leaves every other slot untouched; q is rotated in place as
in rope_append (within 1 bf16 ulp).  decode_fp8 output is within the bf16
attention tolerance (max abs <= 1e-2, rel L2 <= 5e-3) of the exact fp64
attention over the dequantised cache (code * scale), for ragged lengths,
several split counts, groups of 4 and 8 query heads, and rows whose scales
span powers of two (K 2^-4 .. 2^2, V 2^-8 .. 2^0: the kernel's lazy V-scale
reference has to rescale).  Stored codes are compared with +0 and -0 taken
as one value.  prefill_chunk_fp8 attends over the dequantised values rounded
to fp32 and then to bf16 (its bf16 tensor-core path; kvattn.h states this),
and is compared at the same bf16 tolerance with exact attention over those
values.
"""
import numpy as np
import pytest
import torch

import oracle
from oracle import fp8
from _gpu_support import check_rotation, compare, f64

pytestmark = pytest.mark.gpu

BS = 16


def _bf16(a) -> np.ndarray:
    return torch.from_numpy(np.asarray(a, dtype=np.float32)).to(torch.bfloat16).double().numpy()


def _swz(r):
    return (r & 1) | ((r >> 1) & 6)


def pack_pages(ck, sk, cv, sv):
    """The library's fp8 page layout (kvattn.h, kvattn_cache_fp8) of codes [nb, hkv, BS, 128]
    and scales [nb, hkv, BS]: [nb, hkv, BS // 16, 4224] bytes."""
    nb, hkv, bs, D = ck.shape
    P = bs // 16
    r = np.arange(16)
    slot = (r[:, None] * 8 + (np.arange(8)[None, :] ^ _swz(r)[:, None])).reshape(-1)   # (token, chunk) -> slot
    kpart = np.zeros((nb, hkv, P, 128, 16), np.uint8)
    kpart[:, :, :, slot, :] = ck.reshape(nb, hkv, P, 128, 16)
    pages = np.zeros((nb, hkv, P, 4224), np.uint8)
    pages[..., :2048] = kpart.reshape(nb, hkv, P, 2048)
    pages[..., 2048:4096] = cv.reshape(nb, hkv, P, 16, D).transpose(0, 1, 2, 4, 3).reshape(nb, hkv, P, 2048)
    pages[..., 4096:4160] = np.ascontiguousarray(sk.reshape(nb, hkv, P, 16).astype(np.float32)).view(np.uint8)
    pages[..., 4160:4224] = np.ascontiguousarray(sv.reshape(nb, hkv, P, 16).astype(np.float32)).view(np.uint8)
    return pages


def unpack_rows(pages, blk, off):
    """Codes [T, hkv, 128] and scales [T, hkv] of K and V at (block, offset) pairs."""
    T = len(blk)
    pg = pages[blk, :, off // 16]                       # [T, hkv, 4224]
    hkv = pg.shape[1]
    r = off % 16
    slot = r[:, None] * 8 + (np.arange(8)[None, :] ^ _swz(r)[:, None])
    ck = np.take_along_axis(pg[..., :2048].reshape(T, hkv, 128, 16), slot[:, None, :, None], axis=2).reshape(T, hkv, 128)
    cv = np.take_along_axis(pg[..., 2048:4096].reshape(T, hkv, 128, 16), r[:, None, None, None], axis=3)[..., 0]
    sk = np.ascontiguousarray(pg[..., 4096:4160]).view(np.float32)[np.arange(T), :, r]
    sv = np.ascontiguousarray(pg[..., 4160:4224]).view(np.float32)[np.arange(T), :, r]
    return ck, sk, cv, sv


def _random_cache(kv, g, nb, hkv, D, bs=BS, k_exp=(-4, 2)):
    """Oracle-quantised random rows uploaded as an fp8 cache; dequantised K, V [nb, hkv, bs, D].
    Row magnitudes vary by powers of two (exact in bf16): K over 2^k_exp, V over
    2^-8 .. 2^0, so that outputs stay of unit scale, where the absolute bound applies."""
    deq = []
    parts = []
    for lo, hi in (k_exp, (-8, 0)):
        r = _bf16(g.standard_normal((nb, hkv, bs, D)))
        r *= 2.0 ** g.integers(lo, hi + 1, size=(nb, hkv, bs, 1))
        codes, scale = fp8.quantize_rows(r)
        parts += [codes, scale]
        deq.append(fp8.dequantize_rows(codes, scale))
    cache = kv.CacheFP8(torch.from_numpy(pack_pages(*parts)).cuda(), bs)
    return cache, deq[0], deq[1]


def _oracle_cache(deq_k, deq_v):
    nb, hkv, bs, D = deq_k.shape
    oc = oracle.Cache(nb, bs, hkv, D)
    oc.K[:] = deq_k.transpose(0, 2, 1, 3).reshape(nb * bs, hkv, D)
    oc.V[:] = deq_v.transpose(0, 2, 1, 3).reshape(nb * bs, hkv, D)
    return oc


@pytest.mark.parametrize("hq,hkv,splits", [(32, 8, 0), (32, 8, 1), (32, 8, 5), (32, 4, 0), (16, 4, 3)])
def test_decode_fp8_matches_oracle(kvattn_lib, hq, hkv, splits):
    kv = kvattn_lib
    D = 128
    lens = np.array([0, 1, 15, 16, 17, 700, 2100, 3001], dtype=np.int32)
    B = len(lens)
    maxb = (int(lens.max()) + BS - 1) // BS
    g = np.random.default_rng(100 + hq + hkv + splits)
    nb = B * maxb + 3
    table = g.permutation(nb)[: B * maxb].astype(np.int32).reshape(B, maxb)
    cache, dk, dv = _random_cache(kv, g, nb, hkv, D)
    q = torch.from_numpy(g.standard_normal((B, hq, D)).astype(np.float32)).to(torch.bfloat16)
    cfg = kv.make_config(hq, hkv, D, kv.BF16)
    out = kv.decode_fp8(cfg, cache, q.cuda(), torch.from_numpy(table).cuda(), torch.from_numpy(lens).cuda(),
                        int(lens.max()), num_splits=splits)
    assert kv.get_device_status() == 0
    got = f64(out)
    assert np.all(got[lens == 0] == 0.0)
    rows = np.nonzero(lens > 0)[0]
    ref = oracle.attend(_oracle_cache(dk, dv), q.double().numpy()[rows], rows, lens[rows] - 1, table, hq)
    compare(got[rows], ref, "bf16", f"fp8 decode {hq}/{hkv} splits {splits}")


def _check_append_fp8(kv, g, hq, hkv, D, nb, table, seq, pos):
    """rope_append_fp8 of tokens (seq, pos) against the oracle: codes and scales
    bit-identical, q within 1 ulp, every other slot keeps its sentinel bytes."""
    T = len(pos)
    scale_in = 2.0 ** g.integers(-6, 7, size=(T, 1, 1))
    q = _bf16(g.standard_normal((T, hq, D)) * 3)
    k = _bf16(g.standard_normal((T, hkv, D)) * scale_in)
    v = _bf16(g.standard_normal((T, hkv, D)) * scale_in)
    k[0, 0] = 0.0                                         # an all-zero row: scale 1
    v[-1, -1] = 0.0
    cfg = kv.make_config(hq, hkv, D, kv.BF16)
    cache = kv.CacheFP8.empty(nb, hkv, BS)
    cache.pool.fill_(0x7F)
    bf = lambda a: torch.from_numpy(a.astype(np.float32)).to(torch.bfloat16).cuda()   # noqa: E731
    qd = bf(q)
    kv.rope_append_fp8(cfg, cache, qd, bf(k), bf(v), torch.from_numpy(pos).cuda(), torch.from_numpy(seq).cuda(),
                       torch.from_numpy(table).cuda())
    assert kv.get_device_status() == 0
    assert check_rotation(f64(qd), oracle.rope(q, pos), "bf16", "q") <= 2
    kr = oracle.round_to(oracle.rope(k, pos), oracle.BF16)
    ck, sk = fp8.quantize_rows(kr)
    cv, sv = fp8.quantize_rows(v)
    blk = table[seq, pos // BS].astype(np.int64)
    off = (pos % BS).astype(np.int64)
    pages = cache.pool.cpu().numpy()
    gk, gsk, gv, gsv = unpack_rows(pages, blk, off)
    # codes compared with +0 and -0 identified (0x00 / 0x80): the sign of an exact zero
    # from the rotation is not fixed by its definition
    z = lambda c: np.where(c == 0x80, 0, c)   # noqa: E731
    assert np.array_equal(z(gk), z(ck))
    assert np.array_equal(z(gv), z(cv))
    assert np.array_equal(gsk.view(np.uint32), sk.view(np.uint32))
    assert np.array_equal(gsv.view(np.uint32), sv.view(np.uint32))
    assert gsk[0, 0] == 1.0 and gsv[-1, -1] == 1.0
    # every other slot keeps its sentinel bytes
    written = np.zeros((nb, BS), dtype=bool)
    written[blk, off] = True
    ub, uo = np.nonzero(~written)
    rk, rks, rv, rvs = unpack_rows(pages, ub, uo)
    assert np.all(rk == 0x7F) and np.all(rv == 0x7F)
    assert np.all(rks.view(np.uint32) == 0x7F7F7F7F) and np.all(rvs.view(np.uint32) == 0x7F7F7F7F)


@pytest.mark.parametrize("hq,hkv,D", [(32, 8, 128), (12, 12, 128), (32, 4, 128)])
def test_rope_append_fp8_codes_and_scales_bit_exact(kvattn_lib, hq, hkv, D):
    """Tokens at random distinct positions of six sequences (mostly alone in their page)."""
    kv = kvattn_lib
    g = np.random.default_rng(7 + hq + hkv + D)
    rows, maxb, T = 6, 250, 300
    nb = rows * maxb + 5
    table = g.permutation(nb)[: rows * maxb].astype(np.int32).reshape(rows, maxb)
    seq = g.integers(0, rows, size=T).astype(np.int32)
    pos = np.empty(T, dtype=np.int32)
    used = set()
    for t in range(T):
        while True:
            p = int(g.integers(0, maxb * BS))
            if (seq[t], p) not in used:
                used.add((seq[t], p))
                pos[t] = p
                break
    _check_append_fp8(kv, g, hq, hkv, D, nb, table, seq, pos)


@pytest.mark.parametrize("hq,hkv", [(32, 8), (8, 1)])
def test_rope_append_fp8_page_runs_bit_exact(kvattn_lib, hq, hkv):
    """Runs of consecutive tokens sharing a page, as prefill chunks give:
    whole pages, ragged starts and ends, a run in descending positions, a page
    written by two runs cut by another sequence's token (their bytes share
    words), 40 consecutive tokens over three pages, and single tokens.  V of a
    run is written in 16-byte rows, 4-byte words and bytes."""
    kv = kvattn_lib
    g = np.random.default_rng(11 + hq + hkv)
    maxb = 8
    rows = 6
    nb = rows * maxb + 3
    table = g.permutation(nb)[: rows * maxb].astype(np.int32).reshape(rows, maxb)
    parts = [
        (0, np.arange(5, 41)),            # ragged start and end, two whole pages in between
        (1, np.arange(0, 64)),            # four whole pages
        (2, np.arange(47, 31, -1)),       # one page, descending
        (3, np.arange(16, 22)),           # 16..21, cut below by another token
        (4, np.array([3])),
        (3, np.arange(22, 30)),           # the same page again after the cut
        (5, np.arange(8, 48)),            # 40 tokens: half of page 0, pages 1 and 2
        (4, np.array([100, 17, 18])),
    ]
    seq = np.concatenate([np.full(len(p), s) for s, p in parts]).astype(np.int32)
    pos = np.concatenate([p for _, p in parts]).astype(np.int32)
    _check_append_fp8(kv, g, hq, hkv, 128, nb, table, seq, pos)


def test_fp8_history_through_rope_append_then_decode(kvattn_lib):
    """Every token of three sequences through rope_append_fp8, then decode_fp8 of the last one."""
    kv = kvattn_lib
    hq, hkv, D = 32, 8, 128
    lens = [5, 40, 129]
    g = np.random.default_rng(77)
    maxb = (max(lens) + BS - 1) // BS
    nb = len(lens) * maxb + 2
    table = g.permutation(nb)[: len(lens) * maxb].astype(np.int32).reshape(len(lens), maxb)
    pos = np.concatenate([np.arange(n) for n in lens]).astype(np.int32)
    seq = np.concatenate([np.full(n, r) for r, n in enumerate(lens)]).astype(np.int32)
    T = len(pos)
    q = _bf16(g.standard_normal((T, hq, D)))
    k = _bf16(g.standard_normal((T, hkv, D)))
    v = _bf16(g.standard_normal((T, hkv, D)))
    cfg = kv.make_config(hq, hkv, D, kv.BF16)
    cache = kv.CacheFP8.empty(nb, hkv, BS)
    bf = lambda a: torch.from_numpy(a.astype(np.float32)).to(torch.bfloat16).cuda()   # noqa: E731
    qd = bf(q)
    d_table = torch.from_numpy(table).cuda()
    kv.rope_append_fp8(cfg, cache, qd, bf(k), bf(v), torch.from_numpy(pos).cuda(), torch.from_numpy(seq).cuda(),
                       d_table)
    last = np.cumsum(lens) - 1
    out = kv.decode_fp8(cfg, cache, qd[torch.from_numpy(last).cuda()].contiguous(), d_table,
                        torch.tensor(lens, dtype=torch.int32).cuda(), max(lens))
    assert kv.get_device_status() == 0
    ck, sk = fp8.quantize_rows(oracle.round_to(oracle.rope(k, pos), oracle.BF16))
    cv, sv = fp8.quantize_rows(v)
    oc = oracle.Cache(nb, BS, hkv, D)
    oracle.append(oc, fp8.dequantize_rows(ck, sk), fp8.dequantize_rows(cv, sv), pos, seq, table)
    qr = oracle.round_to(oracle.rope(q[last], pos[last]), oracle.BF16)
    ref = oracle.attend(oc, qr, np.arange(len(lens)), pos[last], table, hq)
    compare(f64(out), ref, "bf16", "fp8 end to end")


def _copy_values(deq):
    """The values kvattn_prefill_chunk_fp8 attends over: each dequantised
    element code * scale rounded to fp32, then to bf16 (the header's rule)."""
    return oracle.round_to(oracle.round_to(deq, oracle.F32), oracle.BF16)


def _chunk_table(g, prefixes, qlens, bs, extra=3):
    total = np.asarray(prefixes) + np.asarray(qlens)
    need = (total + bs - 1) // bs
    nb = int(need.sum()) + extra
    perm = g.permutation(nb).astype(np.int32)
    table = np.full((len(total), int(need.max())), -1, dtype=np.int32)
    o = 0
    for r, k in enumerate(need):
        table[r, :k] = perm[o:o + k]
        o += k
    return nb, table


def _chunk_rows(prefixes, qlens):
    seq = np.concatenate([np.full(q, c) for c, q in enumerate(qlens)]).astype(np.int64)
    pos = np.concatenate([np.arange(p, p + q) for p, q in zip(prefixes, qlens)]).astype(np.int64)
    cu = np.zeros(len(qlens) + 1, dtype=np.int32)
    cu[1:] = np.cumsum(qlens)
    return seq, pos, cu


@pytest.mark.parametrize("hq,hkv,bs", [(32, 8, 16), (16, 16, 16), (8, 2, 32)])
def test_prefill_fp8_matches_oracle(kvattn_lib, hq, hkv, bs):
    """Chunked prefill over an fp8 cache against exact attention over the
    dequantised cache values as the library defines them for prefill (each
    rounded to fp32, then bf16): ragged chunks (one row, an empty chunk, prefixes off the
    16-token grid, a chunk of two query tiles), K row scales 2^-4 .. 2^0 (scores
    of unit scale, as the bf16 prefill tests) and V row scales 2^-8 .. 2^0."""
    kv = kvattn_lib
    D = 128
    prefixes = [0, 17, 300, 1000, 5]
    qlens = [200, 1, 129, 64, 0]
    g = np.random.default_rng(200 + hq + hkv + bs)
    nb, table = _chunk_table(g, prefixes, qlens, bs)
    cache, dk, dv = _random_cache(kv, g, nb, hkv, D, bs=bs, k_exp=(-4, 0))
    seq, pos, cu = _chunk_rows(prefixes, qlens)
    q = torch.from_numpy(g.standard_normal((len(seq), hq, D)).astype(np.float32)).to(torch.bfloat16)
    cfg = kv.make_config(hq, hkv, D, kv.BF16)
    kvt = int(np.sum(np.asarray(prefixes) + np.asarray(qlens)))
    out = kv.prefill_chunk_fp8(cfg, cache, q.cuda(), torch.from_numpy(cu).cuda(),
                               torch.tensor(prefixes, dtype=torch.int32).cuda(), torch.from_numpy(table).cuda(),
                               max(qlens), kvt)
    assert kv.get_device_status() == 0
    ref = oracle.attend(_oracle_cache(_copy_values(dk), _copy_values(dv)), q.double().numpy(), seq, pos, table, hq)
    compare(f64(out), ref, "bf16", f"fp8 prefill {hq}/{hkv} BS {bs}")


def test_prefill_fp8_after_rope_append_fp8(kvattn_lib):
    """History and chunk tokens of three sequences through rope_append_fp8 (one
    call), then the chunks' causal attention from the fp8 cache: the oracle
    quantises the correctly rounded rotated k (and v) itself."""
    kv = kvattn_lib
    hq, hkv, D = 32, 8, 128
    prefixes, qlens = [0, 40, 333], [50, 16, 130]
    g = np.random.default_rng(78)
    nb, table = _chunk_table(g, prefixes, qlens, BS)
    lens = np.asarray(prefixes) + np.asarray(qlens)
    pos = np.concatenate([np.arange(n) for n in lens]).astype(np.int32)
    seq = np.concatenate([np.full(n, r) for r, n in enumerate(lens)]).astype(np.int32)
    T = len(pos)
    q = _bf16(g.standard_normal((T, hq, D)))
    k = _bf16(g.standard_normal((T, hkv, D)))
    v = _bf16(g.standard_normal((T, hkv, D)))
    cfg = kv.make_config(hq, hkv, D, kv.BF16)
    cache = kv.CacheFP8.empty(nb, hkv, BS)
    cache.pool.fill_(0x7F)                            # unwritten slots decode to NaN codes
    bf = lambda a: torch.from_numpy(a.astype(np.float32)).to(torch.bfloat16).cuda()   # noqa: E731
    qd = bf(q)
    d_table = torch.from_numpy(table).cuda()
    kv.rope_append_fp8(cfg, cache, qd, bf(k), bf(v), torch.from_numpy(pos).cuda(), torch.from_numpy(seq).cuda(),
                       d_table)
    rows = np.nonzero(pos >= np.asarray(prefixes)[seq])[0]     # the chunk tokens, in chunk order
    _, cpos, cu = _chunk_rows(prefixes, qlens)
    assert np.array_equal(pos[rows], cpos)
    out = kv.prefill_chunk_fp8(cfg, cache, qd[torch.from_numpy(rows).cuda()].contiguous(),
                               torch.from_numpy(cu).cuda(), torch.tensor(prefixes, dtype=torch.int32).cuda(),
                               d_table, max(qlens), int(lens.sum()))
    assert kv.get_device_status() == 0
    ck, sk = fp8.quantize_rows(oracle.round_to(oracle.rope(k, pos), oracle.BF16))
    cv, sv = fp8.quantize_rows(v)
    oc = oracle.Cache(nb, BS, hkv, D)
    oracle.append(oc, _copy_values(fp8.dequantize_rows(ck, sk)), _copy_values(fp8.dequantize_rows(cv, sv)), pos,
                  seq, table)
    qr = oracle.round_to(oracle.rope(q[rows], pos[rows]), oracle.BF16)
    ref = oracle.attend(oc, qr, seq[rows], pos[rows], table, hq)
    compare(f64(out), ref, "bf16", "fp8 prefill end to end")


def test_prefill_fp8_copy_too_small_reports_bad_index(kvattn_lib):
    """max_kv_tokens below what the chunks need: the bf16 copy holds fewer
    blocks than the chunks' keys occupy, which the library reports as
    BAD_INDEX (the blocks past the copy are never written or read)."""
    kv = kvattn_lib
    hq, hkv, D = 32, 8, 128
    prefixes, qlens = [600, 900], [64, 64]
    g = np.random.default_rng(79)
    nb, table = _chunk_table(g, prefixes, qlens, BS)
    cache, _, _ = _random_cache(kv, g, nb, hkv, D, k_exp=(-4, 0))
    _, _, cu = _chunk_rows(prefixes, qlens)
    q = torch.from_numpy(g.standard_normal((sum(qlens), hq, D)).astype(np.float32)).to(torch.bfloat16).cuda()
    cfg = kv.make_config(hq, hkv, D, kv.BF16)
    kv.prefill_chunk_fp8(cfg, cache, q, torch.from_numpy(cu).cuda(), torch.tensor(prefixes, dtype=torch.int32).cuda(),
                         torch.from_numpy(table).cuda(), max(qlens), 700)
    assert kv.get_device_status() == kv.STATUS_CODE["KVATTN_ERR_BAD_INDEX"]
