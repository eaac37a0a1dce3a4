"""GPU checks of prefix sharing with copy on write.

kvattn_copy_blocks must make bit copies of whole blocks in every K and V
region (one-layer and multi-layer caches) and leave every other block as it
was; a pair naming a block outside the pool is skipped and reported.  End to
end, a sequence forked from another's 37-token prefix shares its two full
blocks, copies the partial third block before appending, and both sequences'
decode results match the fp64 oracle of their own token histories (bf16: max
abs <= 1e-2, rel L2 <= 5e-3).
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from _gpu_support import compare, f64

pytestmark = pytest.mark.gpu


def _bits(t):
    return t.view(torch.int16) if t.dtype == torch.bfloat16 else t.view(torch.int32)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_copy_blocks_one_layer(kvattn_lib, dtype):
    kv = kvattn_lib
    cfg = kv.make_config(8, 2, 128, kv.BF16 if dtype == torch.bfloat16 else kv.F32)
    cache = kv.Cache.empty(40, 2, 16, 128, dtype, "cuda")
    cache.k_pool.copy_(torch.randn(cache.k_pool.shape, device="cuda").to(dtype))
    cache.v_pool.copy_(torch.randn(cache.v_pool.shape, device="cuda").to(dtype))
    k0, v0 = cache.k_pool.clone(), cache.v_pool.clone()
    src, dst = [3, 7, 7, 39, 0], [10, 11, 12, 0 + 20, 38]
    kv.copy_blocks(cfg, cache, src, dst)
    assert kv.get_device_status() == 0
    k1, v1 = k0.clone(), v0.clone()
    for s, d in zip(src, dst):
        k1[d], v1[d] = k0[s], v0[s]
    assert torch.equal(_bits(cache.k_pool), _bits(k1)) and torch.equal(_bits(cache.v_pool), _bits(v1))


def test_copy_blocks_layered_and_bad_ids(kvattn_lib):
    kv = kvattn_lib
    cfg = kv.make_config(16, 4, 64, kv.BF16)
    lc = kv.LayeredCache.empty(cfg, 3, 25, 16, torch.bfloat16, "cuda")
    lc.pool.copy_(torch.randn(lc.pool.shape, device="cuda").to(torch.bfloat16))
    before = lc.pool.clone()
    src, dst = [1, 2, 24, 5], [20, 21, 99, 22]      # the third pair names a block outside the pool
    kv.copy_blocks(cfg, lc, src, dst)
    assert kv.STATUS[kv.get_device_status()] == "KVATTN_ERR_BAD_INDEX"
    want = before.clone()
    for s, d in zip(src, dst):
        if d < 25:
            want[:, :, d] = before[:, :, s]
    assert torch.equal(_bits(lc.pool), _bits(want))
    # nothing to copy launches nothing
    kv.copy_blocks(cfg, lc, [], [])
    assert kv.get_device_status() == 0


def test_fork_copy_on_write_then_decode_matches_oracle(kvattn_lib):
    kv = kvattn_lib
    dev = torch.device("cuda")
    Hq, Hkv, D, BS = 8, 2, 128, 16
    P = 37                                   # prefix: blocks 0, 1 full, block 2 holds positions 32..36
    nb, maxb = 12, 4
    cfg = kv.make_config(Hq, Hkv, D, kv.BF16)
    cache = kv.Cache.empty(nb, Hkv, BS, D, torch.bfloat16, dev)
    cache.k_pool.fill_(float("nan"))
    cache.v_pool.fill_(float("nan"))
    alloc = kv.BlockAllocator(nb)
    table = np.full((2, maxb), -1, dtype=np.int32)
    alloc.grow(table[0], BS, 0, P)
    g = workloads.rng(workloads.DATA_SEED, 31)
    q = g.standard_normal((P + 2, Hq, D), dtype=np.float32)
    k = g.standard_normal((P + 2, Hkv, D), dtype=np.float32)
    v = g.standard_normal((P + 2, Hkv, D), dtype=np.float32)
    bf = lambda x: torch.from_numpy(x).to(torch.bfloat16)   # noqa: E731
    # parent history, positions 0..P-1 (row 0)
    pos_h = np.arange(P, dtype=np.int32)
    kv.rope_append(cfg, cache, bf(q[:P]).to(dev), bf(k[:P]).to(dev), bf(v[:P]).to(dev),
                   torch.from_numpy(pos_h).to(dev), torch.zeros(P, dtype=torch.int32, device=dev),
                   torch.from_numpy(table).to(dev))
    # the child (row 1) starts as the parent's 37-token prefix
    alloc.fork(table[0], table[1], BS, P)
    assert list(table[1, :3]) == list(table[0, :3])
    # both append one token at position P: the child copies the shared partial block first
    cow = alloc.prepare_append(table[1], BS, P, P + 1)
    assert cow is not None and cow[0] == table[0, 2] and table[1, 2] == cow[1]
    assert alloc.prepare_append(table[0], BS, P, P + 1) is None
    kv.copy_blocks(cfg, cache, [cow[0]], [cow[1]])
    d_table = torch.from_numpy(table).to(dev)
    q_new = bf(q[P:P + 2]).to(dev)                          # parent's new token, child's new token
    kv.rope_append(cfg, cache, q_new, bf(k[P:P + 2]).to(dev), bf(v[P:P + 2]).to(dev),
                   torch.tensor([P, P], dtype=torch.int32, device=dev),
                   torch.tensor([0, 1], dtype=torch.int32, device=dev), d_table)
    lens = torch.tensor([P + 1, P + 1], dtype=torch.int32, device=dev)
    out = kv.decode(cfg, cache, q_new, d_table, lens, P + 1)
    assert kv.get_device_status() == 0
    # shared full blocks are one copy; the parent's block 2 never saw the child's token
    assert alloc.refcount(int(table[0, 0])) == 2 and alloc.refcount(int(table[0, 2])) == 1

    # oracle: each row's own history (prefix, then its own token at position P)
    x = lambda a: bf(a).double().numpy()   # noqa: E731
    oc = oracle.Cache(nb, BS, Hkv, D)
    for row in (0, 1):
        kk = np.concatenate([x(k[:P]), x(k[P + row:P + row + 1])])
        vv = np.concatenate([x(v[:P]), x(v[P + row:P + row + 1])])
        pos = np.arange(P + 1, dtype=np.int32)
        oracle.append(oc, oracle.round_to(oracle.rope(kk, pos), oracle.BF16), vv, pos,
                      np.full(P + 1, row, np.int32), table)
    qr = oracle.round_to(oracle.rope(x(q[P:P + 2]), [P, P]), oracle.BF16)
    ref = oracle.attend(oc, qr, [0, 1], [P, P], table, Hq)
    compare(f64(out), ref, "bf16", "forked decode")
    # the two rows really differ (the child did not read the parent's token or the reverse)
    assert not np.allclose(ref[0], ref[1])
