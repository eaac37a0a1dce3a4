"""GPU parity of a decode-step layer slice over a multi-layer cache.

Every layer's q, k, v come from one fused QKV projection output per layer
([T, (Hq + 2 Hkv) D], sliced with split_qkv, no copies); rope_append writes
that layer's K/V regions of one LayeredCache and a dense rotated q; decode and
a prefill chunk then run on the layer.  The oracle builds each layer's cache
on its own.  Checks: each layer matches the oracle (bf16: max abs <= 1e-2,
rel L2 <= 5e-3), writes to one layer leave the others' results bit-identical,
and blocks no token names stay NaN in every layer.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from _gpu_support import compare, f64

pytestmark = pytest.mark.gpu

HQ, HKV, D, BS = 16, 4, 128, 16


def _layer_qkv(layer: int, T: int) -> np.ndarray:
    g = workloads.rng(workloads.DATA_SEED, 100 + layer)
    return g.standard_normal((T, (HQ + 2 * HKV) * D), dtype=np.float32)


def test_layer_slice_fused_qkv_over_layered_cache(kvattn_lib):
    kv = kvattn_lib
    dev = torch.device("cuda")
    L = 3
    past = [40, 77, 130]                 # history of each row; the new token sits at position past[r]
    rows = len(past)
    maxb = (max(past) + 1 + BS - 1) // BS
    nb = rows * maxb + 7
    g = workloads.rng(workloads.PERM_SEED, 7)
    table = g.permutation(nb)[: rows * maxb].astype(np.int32).reshape(rows, maxb)
    pos = np.concatenate([np.arange(p + 1) for p in past]).astype(np.int32)
    sid = np.concatenate([np.full(p + 1, r) for r, p in enumerate(past)]).astype(np.int32)
    last = np.cumsum([p + 1 for p in past]) - 1           # each row's new token
    T = len(pos)
    cfg = kv.make_config(HQ, HKV, D, kv.BF16)
    lc = kv.LayeredCache.empty(cfg, L, nb, BS, torch.bfloat16, dev)
    lc.pool.fill_(float("nan"))
    d_pos, d_sid = torch.from_numpy(pos).to(dev), torch.from_numpy(sid).to(dev)
    d_table = torch.from_numpy(table).to(dev)
    d_lens = torch.tensor([p + 1 for p in past], dtype=torch.int32, device=dev)
    # prefill chunk on row 2: its last 24 tokens as queries over the prefix before them
    cq = 24
    p_prefix = past[2] + 1 - cq
    p_rows = np.arange(last[2] - cq + 1, last[2] + 1)
    d_cu = torch.tensor([0, cq], dtype=torch.int32, device=dev)
    d_prefix = torch.tensor([p_prefix], dtype=torch.int32, device=dev)

    host_qkv, dec_out, pre_out, q_last = [], [], [], []
    for layer in range(L):
        h = torch.from_numpy(_layer_qkv(layer, T)).to(torch.bfloat16)
        host_qkv.append(h)
        qkv = h.to(dev)
        q, k, v = kv.split_qkv(qkv, HQ, HKV, D)
        q_rot = torch.empty((T, HQ, D), dtype=torch.bfloat16, device=dev)
        cache = lc.layer(layer)
        kv.rope_append(cfg, cache, q, k, v, d_pos, d_sid, d_table, q_out=q_rot)
        q_last.append(q_rot[torch.from_numpy(last).to(dev)].contiguous())
        dec_out.append(kv.decode(cfg, cache, q_last[-1], d_table, d_lens, max(past) + 1))
        pre_out.append(kv.prefill_chunk(cfg, cache, q_rot[p_rows[0]: p_rows[-1] + 1].contiguous(), d_cu, d_prefix,
                                        d_table[2:3].contiguous(), cq))
        assert torch.equal(qkv.cpu().view(torch.int16), h.view(torch.int16))   # the QKV output is left as it was
    assert kv.get_device_status() == 0

    # layer 0 again, after layers 1 and 2 were written: bit-identical
    again = kv.decode(cfg, lc.layer(0), q_last[0], d_table, d_lens, max(past) + 1)
    assert torch.equal(again.view(torch.int16), dec_out[0].view(torch.int16))

    # every layer against the oracle, built from that layer's tokens only
    for layer in range(L):
        x = host_qkv[layer].double().numpy()
        qh = x[:, : HQ * D].reshape(T, HQ, D)
        kh = x[:, HQ * D: (HQ + HKV) * D].reshape(T, HKV, D)
        vh = x[:, (HQ + HKV) * D:].reshape(T, HKV, D)
        oc = oracle.Cache(nb, BS, HKV, D)
        oracle.append(oc, oracle.round_to(oracle.rope(kh, pos), oracle.BF16), vh, pos, sid, table)
        qr = oracle.round_to(oracle.rope(qh, pos), oracle.BF16)
        ref = oracle.attend(oc, qr[last], np.arange(rows), np.array(past), table, HQ)
        compare(f64(dec_out[layer]), ref, "bf16", f"layer {layer} decode")
        ref_p = oracle.attend(oc, qr[p_rows], np.zeros(cq, np.int32), p_prefix + np.arange(cq), table[2:3], HQ)
        compare(f64(pre_out[layer]), ref_p, "bf16", f"layer {layer} prefill")

    # blocks no token names keep their NaN fill in every layer's K and V region
    unused = np.setdiff1d(np.arange(nb), table[table >= 0])
    named = np.zeros((nb, BS), dtype=bool)
    for t in range(T):
        named[table[sid[t], pos[t] // BS], pos[t] % BS] = True
    nan_slots = lc.pool.float().isnan().all(dim=5).all(dim=3).cpu().numpy()   # [L, 2, nb, BS]
    assert np.array_equal(nan_slots, np.broadcast_to(~named, nan_slots.shape))
    assert nan_slots[:, :, unused].all()


def test_layered_cache_rejects_a_mismatched_pool(kvattn_lib):
    kv = kvattn_lib
    cfg = kv.make_config(HQ, HKV, D, kv.BF16)
    pool = torch.empty((2, 2, 4, HKV + 1, BS, D), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(ValueError):
        kv.LayeredCache(cfg, pool)
    lc = kv.LayeredCache.empty(cfg, 2, 4, BS, torch.bfloat16, "cuda")
    with pytest.raises(kv.KvattnError):
        lc.layer(2)
