"""GPU parity of kvattn_rope_append against the fp64 oracle.

Bar: cache slots and copied V rows bit-exact; rotated q and k within 1 ulp of
the exact rotation (the kernel rounds the exact value, so in practice every
element equals the oracle's round-to-nearest-even); slots not written keep
their sentinel.
"""
import numpy as np
import pytest
import torch

import oracle
from _gpu_support import OR_DT, TORCH_DT, check_rotation, f64, get_rows

pytestmark = pytest.mark.gpu


def _run_case(kv, dtype, Hq, Hkv, D, BS, rows, maxb, T, max_pos, seed, contiguous=False, fused_pad=None,
              separate_q_out=False):
    dev = torch.device("cuda")
    g = np.random.default_rng(seed)
    dt = TORCH_DT[dtype]
    if contiguous:
        nb = rows
        table = g.permutation(nb).astype(np.int32).reshape(rows, 1)
    else:
        nb = rows * maxb + 5
        table = g.permutation(nb)[: rows * maxb].astype(np.int32).reshape(rows, maxb)
    # distinct (row, position) pairs
    seq = g.integers(0, rows, size=T).astype(np.int32)
    pos = np.empty(T, dtype=np.int32)
    used = set()
    for t in range(T):
        while True:
            p = int(g.integers(0, max_pos))
            if (seq[t], p) not in used:
                used.add((seq[t], p))
                pos[t] = p
                break
    q = torch.from_numpy(g.standard_normal((T, Hq, D), dtype=np.float32) * 3).to(dt)
    k = torch.from_numpy(g.standard_normal((T, Hkv, D), dtype=np.float32) * 3).to(dt)
    v = torch.from_numpy(g.standard_normal((T, Hkv, D), dtype=np.float32)).to(dt)
    cfg = kv.make_config(Hq, Hkv, D, kv.BF16 if dtype == "bf16" else kv.F32)
    cache = kv.Cache.empty(nb, Hkv, BS, D, dt, dev)
    cache.k_pool.fill_(float("nan"))
    cache.v_pool.fill_(float("nan"))
    if fused_pad is None:
        qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    else:
        # one fused QKV projection output per token, [q | k | v | pad], taken as strided views
        width = (Hq + 2 * Hkv) * D
        buf = torch.full((T, width + fused_pad), -7.0, dtype=dt, device=dev)
        buf[:, :width] = torch.cat([q.reshape(T, -1), k.reshape(T, -1), v.reshape(T, -1)], 1).to(dev)
        qd, kd, vd = kv.split_qkv(buf[:, :width], Hq, Hkv, D)
        assert not qd.is_contiguous()
    q_out = torch.full((T, Hq, D), float("nan"), dtype=dt, device=dev) if separate_q_out else None
    kv.rope_append(cfg, cache, qd, kd, vd, torch.from_numpy(pos).to(dev),
                   torch.from_numpy(seq).to(dev), torch.from_numpy(table).to(dev), q_out=q_out)
    assert kv.get_device_status() == 0
    bits = torch.int16 if dtype == "bf16" else torch.int32
    if fused_pad is not None:
        # only the q slices were written (none of the buffer with a separate q_out)
        hb = buf.cpu()
        first = Hq * D if q_out is None else 0
        kept = torch.cat([q.reshape(T, -1), k.reshape(T, -1), v.reshape(T, -1)], 1)[:, first:]
        assert torch.equal(hb[:, first: width].view(bits), kept.view(bits))
        assert bool((hb[:, width:] == -7.0).all())
    if q_out is not None:
        assert torch.equal(qd.cpu().view(bits), q.view(bits))  # the input q is left as it was
        qd = q_out
    # q in place
    q_exact = oracle.rope(q.double().numpy(), pos)
    nq = check_rotation(f64(qd), q_exact, dtype, "q")
    # k and v at their slots
    k_exact = oracle.rope(k.double().numpy(), pos)
    k_got = np.stack([f64(get_rows(cache.k_pool, table[seq[t]], pos[t:t + 1]))[0] for t in range(T)])
    v_got = np.stack([f64(get_rows(cache.v_pool, table[seq[t]], pos[t:t + 1]))[0] for t in range(T)])
    nk = check_rotation(k_got, k_exact, dtype, "k")
    np.testing.assert_array_equal(v_got, v.double().numpy())
    # everything else untouched
    written = np.zeros((nb, BS), dtype=bool)
    for t in range(T):
        written[table[seq[t], pos[t] // BS], pos[t] % BS] = True
    kp = cache.k_pool.float().isnan().all(dim=3).all(dim=1).cpu().numpy()
    vp = cache.v_pool.float().isnan().all(dim=3).all(dim=1).cpu().numpy()
    assert np.array_equal(kp, ~written) and np.array_equal(vp, ~written)
    return nq, nk, q.numel() + k.numel()


def test_rope_append_bf16_gqa_paged_large_positions(kvattn_lib):
    nq, nk, n = _run_case(kvattn_lib, "bf16", 32, 8, 128, 16, rows=12, maxb=1100, T=400, max_pos=17600, seed=1)
    # the kernel returns the correctly rounded value; allow a handful of near-ties
    assert nq + nk <= max(2, n * 1e-6), (nq, nk)


def test_rope_append_bf16_mha_d64_contiguous(kvattn_lib):
    nq, nk, n = _run_case(kvattn_lib, "bf16", 12, 12, 64, 1025, rows=8, maxb=1, T=300, max_pos=1025, seed=2,
                          contiguous=True)
    assert nq + nk <= max(2, n * 1e-6), (nq, nk)


def test_rope_append_f32_gpt2_shape(kvattn_lib):
    nq, nk, n = _run_case(kvattn_lib, "f32", 12, 12, 64, 128, rows=1, maxb=1, T=128, max_pos=128, seed=3,
                          contiguous=True)
    assert nq + nk <= max(2, n * 1e-6)


def test_rope_append_gqa8_block32(kvattn_lib):
    _run_case(kvattn_lib, "bf16", 16, 2, 128, 32, rows=5, maxb=40, T=150, max_pos=1280, seed=4)


def test_rope_append_f32_gqa_d128_ring(kvattn_lib):
    """fp32 q/k/v of 32/8 heads x 128 (24.6 KB per token): two ring stages per CTA."""
    nq, nk, n = _run_case(kvattn_lib, "f32", 32, 8, 128, 16, rows=4, maxb=30, T=100, max_pos=480, seed=6)
    assert nq + nk <= max(2, n * 1e-6)


def test_rope_append_f32_many_heads_one_cta_per_token(kvattn_lib):
    """fp32, 64 q heads x 128: a token (42 KB) does not fit two ring stages and
    takes the one-CTA-per-token kernel."""
    nq, nk, n = _run_case(kvattn_lib, "f32", 64, 8, 128, 16, rows=3, maxb=20, T=60, max_pos=320, seed=5)
    assert nq + nk <= max(2, n * 1e-6)


def test_rope_append_fused_qkv_bf16_gqa(kvattn_lib):
    """q, k, v as slices of one fused [T, (32 + 2*8) * 128] projection output."""
    nq, nk, n = _run_case(kvattn_lib, "bf16", 32, 8, 128, 16, rows=6, maxb=200, T=300, max_pos=3200, seed=7,
                          fused_pad=0)
    assert nq + nk <= max(2, n * 1e-6), (nq, nk)


def test_rope_append_fused_qkv_padded_rows_f32_gpt2_shape(kvattn_lib):
    """GPT-2 12 x 64 heads in fp32, fused rows padded by 8 elements (row stride 2312)."""
    nq, nk, n = _run_case(kvattn_lib, "f32", 12, 12, 64, 128, rows=2, maxb=1, T=200, max_pos=128, seed=8,
                          contiguous=True, fused_pad=8)
    assert nq + nk <= max(2, n * 1e-6)


def test_rope_append_fused_qkv_separate_q_out(kvattn_lib):
    """Fused QKV rows left untouched, rotated q written to a dense q_out (ring kernel)."""
    nq, nk, n = _run_case(kvattn_lib, "bf16", 32, 8, 128, 16, rows=4, maxb=100, T=200, max_pos=1600, seed=10,
                          fused_pad=16, separate_q_out=True)
    assert nq + nk <= max(2, n * 1e-6), (nq, nk)


def test_rope_append_separate_q_out_one_cta_per_token(kvattn_lib):
    """Dense inputs with a separate q_out, fp32 64/8 x 128: the one-CTA-per-token kernel."""
    nq, nk, n = _run_case(kvattn_lib, "f32", 64, 8, 128, 16, rows=3, maxb=20, T=40, max_pos=320, seed=11,
                          separate_q_out=True)
    assert nq + nk <= max(2, n * 1e-6)


def test_rope_append_fused_qkv_one_cta_per_token(kvattn_lib):
    """fp32 64/8 x 128 (too large for two ring stages): the one-CTA-per-token kernel on strided rows."""
    nq, nk, n = _run_case(kvattn_lib, "f32", 64, 8, 128, 16, rows=3, maxb=20, T=60, max_pos=320, seed=9,
                          fused_pad=4)
    assert nq + nk <= max(2, n * 1e-6)


def test_rope_append_reports_bad_index_and_writes_the_rest(kvattn_lib):
    kv = kvattn_lib
    dev = torch.device("cuda")
    cfg = kv.make_config(4, 4, 64, kv.BF16)
    cache = kv.Cache.empty(4, 4, 16, 64, torch.bfloat16, dev)
    cache.k_pool.zero_()
    cache.v_pool.zero_()
    table = torch.tensor([[0, 1], [2, 9]], dtype=torch.int32, device=dev)   # block 9 does not exist
    T = 4
    q = torch.randn(T, 4, 64, device=dev).to(torch.bfloat16)
    k = torch.ones(T, 4, 64, device=dev).to(torch.bfloat16)
    pos = torch.tensor([0, 17, 40, 3], dtype=torch.int32, device=dev)       # 17 -> block 9; 40 -> past the table
    seq = torch.tensor([0, 1, 0, 1], dtype=torch.int32, device=dev)
    kv.rope_append(cfg, cache, q, k, k, pos, seq, table)
    assert kv.STATUS[kv.get_device_status()] == "KVATTN_ERR_BAD_INDEX"
    assert kv.get_device_status() == 0   # read clears it
    # valid tokens written: (seq 0, pos 0) -> block 0 slot 0; (seq 1, pos 3) -> block 2 slot 3
    assert (cache.v_pool[0, :, 0].float() == 1).all() and (cache.v_pool[2, :, 3].float() == 1).all()
    assert (cache.v_pool[1].float() == 0).all()


def test_rope_append_empty_call_launches_nothing(kvattn_lib):
    kv = kvattn_lib
    dev = torch.device("cuda")
    cfg = kv.make_config(4, 4, 64, kv.BF16)
    cache = kv.Cache.empty(2, 4, 16, 64, torch.bfloat16, dev)
    z = torch.empty(0, 4, 64, device=dev, dtype=torch.bfloat16)
    i = torch.empty(0, dtype=torch.int32, device=dev)
    kv.rope_append(cfg, cache, z, z, z, i, i, torch.zeros(1, 1, dtype=torch.int32, device=dev))
    assert kv.get_device_status() == 0
