"""GPU parity of the whole mixed step exactly as bench.py times it.

The mixed workload (16 prefill chunks of 512 causal queries over prefixes
U[0,8192] plus 128 decode sequences of past length U[256,8192], GQA 32/8 x 128,
bf16, paged 16) is built by bench.Step: its full pool, its block table handed
out through the host allocator, its history drawn on the device, and the
library's automatic split count.  One Step.launch() runs rope_append over all
8320 new tokens, prefill over the 16 chunks and decode over the 128 rows.

The history is input data: the rows the oracle recomputes are read back from
the device pools before the step.  The oracle then appends the correctly
rounded rotated keys of the new tokens and computes the attention of the
sampled queries: 16 decode rows spread over the length range (the shortest
and the longest included) and every 7th query row of three chunks (the
shortest, median and longest prefix).  Element by element against the
attention tolerance of every bf16 test (max abs 1e-2, relative L2 5e-3); the
rotated q of the sampled rows and the rotated k written into the cache must
equal the correctly rounded rotation, and the appended v rows must be bit
copies ("Hand-writing an LLM inference engine" series intro, section 4.2:
compare against an independent implementation step by step).
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from _gpu_support import compare, f64, get_rows

pytestmark = pytest.mark.gpu


def _pick(values, n):
    """Indices of n entries spread evenly over the sorted order of values (min and max included)."""
    order = np.argsort(values, kind="stable")
    return sorted({int(order[int(round(i * (len(order) - 1) / (n - 1)))]) for i in range(n)})


def test_c5_step_as_benched(kvattn_lib):
    import bench

    kv = kvattn_lib
    wl = workloads.WORKLOADS["c5"]
    dev = torch.device("cuda")
    st = bench.Step(wl, dev)
    b = st.batch
    nchunk, H, D, Hq, BS = st.nchunk, wl.num_kv_heads, wl.head_dim, wl.num_q_heads, wl.block_size
    assert nchunk == 16 and st.n_dec == 128 and st.n_tok == 16 * 512 + 128
    assert st.splits == kv.decode_num_splits(st.cfg, 128, st.max_len, 0) and st.splits > 1
    table = st.d_table.cpu().numpy()
    dec_rows = [nchunk + i for i in _pick(b.past[nchunk:], 16)]
    pre = b.past[:nchunk]
    order = np.argsort(pre, kind="stable")
    chunk_rows = sorted({int(order[0]), int(order[len(order) // 2]), int(order[-1])})
    rows = chunk_rows + dec_rows

    # ---- history of the sampled rows, read back from the device pools (input data)
    need = [(int(b.total[r]) + BS - 1) // BS for r in rows]
    o_table = np.full((len(rows), max(need)), -1, dtype=np.int32)
    nxt = 0
    for i, n in enumerate(need):
        o_table[i, :n] = np.arange(nxt, nxt + n, dtype=np.int32)
        nxt += n
    oc = oracle.Cache(nxt, BS, H, D)
    for i, r in enumerate(rows):
        P = int(b.past[r])
        if P == 0:
            continue
        pos = np.arange(P)
        k = f64(get_rows(st.cache.k_pool, table[r], pos))
        v = f64(get_rows(st.cache.v_pool, table[r], pos))
        oracle.append(oc, k, v, pos, np.full(P, i, np.int32), o_table)

    st.launch()
    torch.cuda.synchronize()
    assert kv.get_device_status() == 0

    # ---- the new tokens of the sampled rows through the oracle
    tok0 = np.concatenate([[0], np.cumsum(b.new)])
    q_raw, k_raw, v_raw = st.h_q.double().numpy(), st.h_k.double().numpy(), st.h_v.double().numpy()
    q_rot = f64(st.q)
    dec_q, dec_idx = [], []
    pre_q, pre_rows, pre_pos, pre_got = [], [], [], []
    out_pre, out_dec = f64(st.out_pre), f64(st.out_dec)
    for i, r in enumerate(rows):
        t0, n, P = int(tok0[r]), int(b.new[r]), int(b.past[r])
        pos = np.arange(P, P + n)
        kh = oracle.round_to(oracle.rope(k_raw[t0:t0 + n], pos), oracle.BF16)
        qh = oracle.round_to(oracle.rope(q_raw[t0:t0 + n], pos), oracle.BF16)
        oracle.append(oc, kh, v_raw[t0:t0 + n], pos, np.full(n, i, np.int32), o_table)
        # rope_append: correctly rounded q and k, v copied bit for bit
        assert np.array_equal(q_rot[t0:t0 + n], qh), f"row {r}: rotated q"
        assert np.array_equal(f64(get_rows(st.cache.k_pool, table[r], pos)), kh), f"row {r}: cached k"
        assert np.array_equal(f64(get_rows(st.cache.v_pool, table[r], pos)), v_raw[t0:t0 + n]), f"row {r}: v"
        if r < nchunk:
            sel = np.arange(0, n, 7)
            pre_q.append(qh[sel])
            pre_rows += [i] * len(sel)
            pre_pos.append(pos[sel])
            pre_got.append(out_pre[t0 + sel])
        else:
            dec_q.append(qh[0])
            dec_idx.append(i)
    ref_dec = oracle.attend(oc, np.stack(dec_q), dec_idx, [int(b.past[r]) for r in dec_rows], o_table, Hq)
    got_dec = out_dec[[r - nchunk for r in dec_rows]]
    compare(got_dec, ref_dec, "bf16", f"c5 step decode rows {dec_rows}")
    ref_pre = oracle.attend(oc, np.concatenate(pre_q), pre_rows, np.concatenate(pre_pos), o_table, Hq)
    compare(np.concatenate(pre_got), ref_pre, "bf16", f"c5 step prefill chunks {chunk_rows}")
    del st
    torch.cuda.empty_cache()
