"""GPU check of continuous-batching block reuse.

A finished sequence hands its blocks back to the host allocator, and a new
sequence that starts again at position 0 gets those same blocks
("From-scratch AI inference engine" page, sections 4.1 and 4.4: freed cache
blocks are reused by new requests, whose positions restart).  The reused
blocks still hold the old sequence's rotated keys and values, finite and
plausible, in every slot the new sequence has not written yet.  Decode of the
new sequence must see only its own tokens: its output is compared with the
fp64 oracle of the new sequence's history alone (bf16: max abs <= 1e-2, rel
L2 <= 5e-3), for a length that ends inside a block so that stale slots sit
right after the last valid one.
"""
import numpy as np
import pytest
import torch

import oracle
from _gpu_support import compare, f64

pytestmark = pytest.mark.gpu


def _tokens(g, n, hq, hkv, d):
    q = torch.from_numpy(g.standard_normal((n, hq, d), dtype=np.float32)).to(torch.bfloat16)
    k = torch.from_numpy(g.standard_normal((n, hkv, d), dtype=np.float32)).to(torch.bfloat16)
    v = torch.from_numpy(g.standard_normal((n, hkv, d), dtype=np.float32)).to(torch.bfloat16)
    return q, k, v


@pytest.mark.parametrize("old_len,new_len", [(300, 37), (64, 64), (130, 129)])
def test_released_blocks_reused_from_position_zero(kvattn_lib, old_len, new_len):
    kv = kvattn_lib
    dev = torch.device("cuda")
    Hq, Hkv, D, BS = 32, 8, 128, 16
    num_blocks = 64
    cfg = kv.make_config(Hq, Hkv, D, kv.BF16)
    cache = kv.Cache.empty(num_blocks, Hkv, BS, D, torch.bfloat16, dev)
    cache.k_pool.fill_(float("nan"))
    cache.v_pool.fill_(float("nan"))
    alloc = kv.BlockAllocator(num_blocks)
    maxb = 32
    g = np.random.default_rng(old_len * 1000 + new_len)

    def run_sequence(length):
        """Allocate a row for `length` tokens, append them all, decode the last one."""
        row = np.full(maxb, -1, dtype=np.int32)
        alloc.grow(row, BS, 0, length)
        q, k, v = _tokens(g, length, Hq, Hkv, D)
        pos = np.arange(length, dtype=np.int32)
        d_table = torch.from_numpy(row[None, :].copy()).to(dev)
        qd = q.to(dev)
        kv.rope_append(cfg, cache, qd, k.to(dev), v.to(dev), torch.from_numpy(pos).to(dev),
                       torch.zeros(length, dtype=torch.int32, device=dev), d_table)
        out = kv.decode(cfg, cache, qd[-1:].contiguous(), d_table,
                        torch.tensor([length], dtype=torch.int32, device=dev), length, num_splits=3)
        assert kv.get_device_status() == 0
        return row, q, k, v, pos, out

    old_row, *_ = run_sequence(old_len)
    old_blocks = set(int(b) for b in old_row[old_row >= 0])
    alloc.release(old_row, BS, old_len)
    assert alloc.num_free == num_blocks
    row, q, k, v, pos, out = run_sequence(new_len)
    new_blocks = [int(b) for b in row[row >= 0]]
    # LIFO free list: the new sequence gets blocks the old one held
    assert set(new_blocks) <= old_blocks
    # stale slots of the last block are finite (the old sequence's data), so a leak would show
    last = new_blocks[-1]
    if new_len % BS:
        assert torch.isfinite(cache.k_pool[last, :, new_len % BS:, :].float()).all()
    # oracle of the new sequence alone
    oc = oracle.Cache(num_blocks, BS, Hkv, D)
    table = row[None, :]
    kh = oracle.round_to(oracle.rope(k.double().numpy(), pos), oracle.BF16)
    oracle.append(oc, kh, v.double().numpy(), pos, np.zeros(new_len, np.int32), table)
    qh = oracle.round_to(oracle.rope(q[-1:].double().numpy(), [new_len - 1]), oracle.BF16)
    ref = oracle.attend(oc, qh, [0], [new_len - 1], table, Hq)
    compare(f64(out), ref, "bf16", f"reused blocks, old {old_len} new {new_len}")
    alloc.close()
