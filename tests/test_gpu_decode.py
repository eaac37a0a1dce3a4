"""GPU parity of rope_append + split-KV decode against the fp64 oracle.

Tolerance (attention output): bf16 max abs <= 1e-2 and rel L2 <= 5e-3; fp32
<= 1e-5 for both.  Covers the five workloads (full size where the oracle is
quick, else a seeded subset of rows; the largest also at full size with
sampled rows), the split counts, GQA group sizes 1/2/4/8, empty and ragged
sequences, paged vs contiguous layouts, and device-side index errors.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from _gpu_support import OR_DT, TORCH_DT, DecodeCase, check_rotation, compare, f64, put_rows

pytestmark = pytest.mark.gpu


def _check(case, out, what):
    _, ref = case.expected()
    got = f64(out)[case.rows]
    return compare(got, ref, case.wl.dtype, what)


def test_c1_tiny_fp32_full_history_through_rope_append(kvattn_lib):
    """Config 1 end to end: all 128 tokens go through rope_append, then decode."""
    kv = kvattn_lib
    wl = workloads.WORKLOADS["c1"]
    dev = torch.device("cuda")
    L = 128
    g = workloads.rng(workloads.DATA_SEED)
    q = g.standard_normal((L, 12, 64), dtype=np.float32)
    k = g.standard_normal((L, 12, 64), dtype=np.float32)
    v = g.standard_normal((L, 12, 64), dtype=np.float32)
    cfg = kv.make_config(12, 12, 64, kv.F32)
    cache = kv.Cache.empty(1, 12, 128, 64, torch.float32, dev)
    table = np.zeros((1, 1), dtype=np.int32)
    pos = np.arange(L, dtype=np.int32)
    qd = torch.from_numpy(q).to(dev)
    kv.rope_append(cfg, cache, qd, torch.from_numpy(k).to(dev), torch.from_numpy(v).to(dev),
                   torch.from_numpy(pos).to(dev), torch.zeros(L, dtype=torch.int32, device=dev),
                   torch.from_numpy(table).to(dev))
    out = kv.decode(cfg, cache, qd[-1:].contiguous(), torch.from_numpy(table).to(dev),
                    torch.tensor([L], dtype=torch.int32, device=dev), L)
    assert kv.get_device_status() == 0
    oc = oracle.Cache(1, 128, 12, 64)
    kh = oracle.round_to(oracle.rope(k.astype(np.float64), pos), oracle.F32)
    oracle.append(oc, kh, v.astype(np.float64), pos, np.zeros(L, np.int32), table)
    qh = oracle.round_to(oracle.rope(q[-1:].astype(np.float64), [L - 1]), oracle.F32)
    ref = oracle.attend(oc, qh, [0], [L - 1], table, 12)
    compare(f64(out), ref, "f32", "c1")
    check_rotation(f64(qd), oracle.rope(q.astype(np.float64), pos), "f32", "c1 q")


def test_c2_gpt2_bf16_contiguous_full(kvattn_lib):
    wl = workloads.WORKLOADS["c2"]
    b = workloads.make_batch(wl)
    case = DecodeCase(wl, b, range(b.rows))
    q, out = case.run()
    assert kvattn_lib.get_device_status() == 0
    _check(case, out, "c2")
    qh, _ = case.expected()
    assert np.array_equal(f64(q), qh), "rotated q differs from the correctly rounded value"


@pytest.mark.parametrize("key,rows", [("c3", range(0, 64, 8)), ("c4", range(0, 256, 32)),
                                      ("c5", list(range(16, 144, 16)))])
def test_paged_workloads_subset(kvattn_lib, key, rows):
    """Rows of configs 3-5 (their lengths, head layouts and block tables) on a compact pool."""
    wl = workloads.WORKLOADS[key]
    # c5: rows 16.. are the decode rows of the mixed workload (new token at position past)
    b = workloads.make_batch(wl, num_blocks=1 << 20, rows_subset=list(rows))
    case = DecodeCase(wl, b, range(b.rows))
    _, out = case.run()
    assert kvattn_lib.get_device_status() == 0
    _check(case, out, key)


@pytest.mark.parametrize("splits", [1, 2, 7, 0])
def test_split_counts_agree(kvattn_lib, splits):
    wl = workloads.WORKLOADS["c4"]
    b = workloads.make_batch(wl, num_blocks=1 << 19, rows_subset=[3, 50, 77, 200])
    case = DecodeCase(wl, b, range(b.rows))
    _, out = case.run(num_splits=splits)
    assert kvattn_lib.get_device_status() == 0
    _check(case, out, f"splits={splits}")


@pytest.mark.parametrize("hq,hkv,d", [(8, 8, 128), (16, 8, 128), (32, 8, 64), (32, 4, 128), (64, 8, 128),
                                      (8, 1, 64)])
def test_group_sizes_and_head_dims(kvattn_lib, hq, hkv, d):
    wl = workloads.Workload("g", "group sweep", "bf16", hq, hkv, d, "paged", 16, 5, (0, 700))
    b = workloads.make_batch(wl)
    case = DecodeCase(wl, b, range(b.rows))
    _, out = case.run()
    assert kvattn_lib.get_device_status() == 0
    _check(case, out, f"{hq}/{hkv}x{d}")


def test_ragged_lengths_and_empty_sequences(kvattn_lib):
    """Lengths 0 (no keys: output zeros), 1, 15, 16, 17, 31, 33 and a long one."""
    kv = kvattn_lib
    wl = workloads.Workload("r", "ragged", "bf16", 8, 2, 128, "paged", 16, 8, (0, 0))
    total = np.array([0, 1, 15, 16, 17, 31, 33, 1500], dtype=np.int64)
    BS = 16
    need = (total + BS - 1) // BS
    nb = int(need.sum()) + 4
    perm = np.random.default_rng(7).permutation(nb).astype(np.int32)
    table = np.full((8, int(need.max())), -1, dtype=np.int32)
    o = 0
    for r, n in enumerate(need):
        table[r, :n] = perm[o:o + n]
        o += n
    past = np.maximum(total - 1, 0)
    new = (total > 0).astype(np.int64)
    b = workloads.Batch(wl, past, new, ["decode"] * 8, nb, table)
    case = DecodeCase(wl, b, range(8))
    # the row with no tokens gets no new token: decode it with seq_len 0
    case.seq_lens = torch.from_numpy(total.astype(np.int32)).cuda()
    dev = case.device
    keep = np.nonzero(total > 0)[0]
    qk = case.q_raw[keep].to(dev).contiguous()
    kv.rope_append(case.cfg, case.cache, qk, case.k_raw[keep].to(dev).contiguous(),
                   case.v_raw[keep].to(dev).contiguous(), case.positions[keep].contiguous(),
                   case.seq_ids[keep].contiguous(), case.d_table)
    qrot = torch.zeros_like(case.q_raw, device=dev)
    qrot[keep] = qk
    out = kv.decode(case.cfg, case.cache, qrot, case.d_table, case.seq_lens, int(total.max()), num_splits=3)
    assert kv.get_device_status() == 0
    got = f64(out)
    assert np.all(got[0] == 0.0)
    # oracle over the rows that have keys
    od = OR_DT["bf16"]
    qh, outs = [], []
    for r in keep:
        p = int(past[r])
        kh = oracle.round_to(oracle.rope(case.k_raw[r:r + 1].double().numpy(), [p]), od)
        oracle.append(case.ocache, kh, case.v_raw[r:r + 1].double().numpy(), [p], [case.rows.index(r)],
                      case.o_table)
        qh.append(oracle.round_to(oracle.rope(case.q_raw[r:r + 1].double().numpy(), [p]), od)[0])
    ref = oracle.attend(case.ocache, np.stack(qh), [case.rows.index(r) for r in keep], [int(past[r]) for r in keep],
                        case.o_table, 8)
    compare(got[keep], ref, "bf16", "ragged")


def test_paged_and_contiguous_layouts_agree(kvattn_lib):
    """The same logical cache in 16-token pages and in contiguous rows gives the same output."""
    kv = kvattn_lib
    dev = torch.device("cuda")
    g = np.random.default_rng(11)
    B, Hq, Hkv, D, maxlen = 4, 16, 4, 128, 700
    lens = g.integers(1, maxlen + 1, size=B)
    cfg = kv.make_config(Hq, Hkv, D, kv.BF16)
    paged = kv.Cache.empty(B * 44 + 3, Hkv, 16, D, torch.bfloat16, dev)
    contig = kv.Cache.empty(B, Hkv, maxlen, D, torch.bfloat16, dev)
    ptab = g.permutation(B * 44 + 3)[: B * 44].astype(np.int32).reshape(B, 44)
    ctab = g.permutation(B).astype(np.int32).reshape(B, 1)
    for r in range(B):
        kk = torch.randn(int(lens[r]), Hkv, D, device=dev).to(torch.bfloat16)
        vv = torch.randn(int(lens[r]), Hkv, D, device=dev).to(torch.bfloat16)
        pos = np.arange(lens[r])
        put_rows(paged.k_pool, ptab[r], pos, kk); put_rows(paged.v_pool, ptab[r], pos, vv)
        put_rows(contig.k_pool, ctab[r], pos, kk); put_rows(contig.v_pool, ctab[r], pos, vv)
    q = torch.randn(B, Hq, D, device=dev).to(torch.bfloat16)
    sl = torch.from_numpy(lens.astype(np.int32)).to(dev)
    a = kv.decode(cfg, paged, q, torch.from_numpy(ptab).to(dev), sl, maxlen, num_splits=3)
    c = kv.decode(cfg, contig, q, torch.from_numpy(ctab).to(dev), sl, maxlen, num_splits=3)
    assert kv.get_device_status() == 0
    assert torch.equal(a, c)


def test_bad_block_id_is_reported(kvattn_lib):
    kv = kvattn_lib
    dev = torch.device("cuda")
    cfg = kv.make_config(8, 2, 128, kv.BF16)
    cache = kv.Cache.empty(8, 2, 16, 128, torch.bfloat16, dev)
    cache.k_pool.normal_(); cache.v_pool.normal_()
    table = torch.tensor([[0, 1, 2], [3, 99, 4]], dtype=torch.int32, device=dev)
    q = torch.randn(2, 8, 128, device=dev).to(torch.bfloat16)
    kv.decode(cfg, cache, q, table, torch.tensor([40, 40], dtype=torch.int32, device=dev), 48)
    assert kv.STATUS[kv.get_device_status()] == "KVATTN_ERR_BAD_INDEX"
    # a sequence longer than max_seq_len is an index error too
    kv.decode(cfg, cache, q, table, torch.tensor([40, 47], dtype=torch.int32, device=dev), 45)
    assert kv.STATUS[kv.get_device_status()] == "KVATTN_ERR_BAD_INDEX"


@pytest.mark.slow
def test_c4_full_size_sampled_rows(kvattn_lib):
    """Config 4 as bench.py runs it: 256 sequences over a 180e9-byte pool (halved until it
    fits), auto split count; 16 sampled rows recomputed by the oracle."""
    wl = workloads.WORKLOADS["c4"]
    per_block = 2 * wl.block_size * wl.num_kv_heads * wl.head_dim * wl.elem_bytes
    nb = wl.pool_bytes // per_block
    free = torch.cuda.mem_get_info()[0]
    while nb * per_block > free * 0.85:
        nb //= 2
    b = workloads.make_batch(wl, num_blocks=nb)
    rows = list(range(0, 256, 16))
    case = DecodeCase(wl, b, rows, fill_nan=False)
    _, out = case.run()
    assert kvattn_lib.get_device_status() == 0
    _check(case, out, "c4 full")
    del case
    torch.cuda.empty_cache()


def test_c3_full_size_sampled_rows(kvattn_lib):
    wl = workloads.WORKLOADS["c3"]
    b = workloads.make_batch(wl)
    case = DecodeCase(wl, b, list(range(0, 64, 9)))
    _, out = case.run()
    assert kvattn_lib.get_device_status() == 0
    _check(case, out, "c3 full")


def test_large_batch_short_sequences(kvattn_lib):
    """6000 sequences: the per-batch prefix array takes ~24 KB of shared memory,
    so the kernel runs with a shallower ring (a multiple of the consumer warps);
    checked on a sample of rows."""
    wl = workloads.Workload("lb", "large batch", "bf16", 32, 8, 128, "paged", 16, 6000, (0, 60))
    b = workloads.make_batch(wl)
    rows = list(range(0, 6000, 397))
    case = DecodeCase(wl, b, rows)
    _, out = case.run()
    assert kvattn_lib.get_device_status() == 0
    _check(case, out, "large batch")


def test_c4_gqa8_full_size_sampled_rows(kvattn_lib):
    """c4's lengths and block tables with 64 query heads over its 8 KV heads (groups of
    8, one tensor-core segment per KV head) on a compact pool; 12 sampled rows."""
    wl = workloads.WORKLOADS["c4g8"]
    b = workloads.make_batch(wl, num_blocks=1 << 20)
    case = DecodeCase(wl, b, list(range(0, 256, 22)), fill_nan=False)
    _, out = case.run()
    assert kvattn_lib.get_device_status() == 0
    _check(case, out, "c4 GQA-8")
    del case
    torch.cuda.empty_cache()


def test_c4_gqa2_full_size_sampled_rows(kvattn_lib):
    """c4's lengths and block tables with 16 query heads over its 8 KV heads (groups of
    2, the CUDA-core path) on a compact pool; 12 sampled rows."""
    wl = workloads.WORKLOADS["c4g2"]
    b = workloads.make_batch(wl, num_blocks=1 << 20)
    case = DecodeCase(wl, b, list(range(0, 256, 22)), fill_nan=False)
    _, out = case.run()
    assert kvattn_lib.get_device_status() == 0
    _check(case, out, "c4 GQA-2")
    del case
    torch.cuda.empty_cache()
