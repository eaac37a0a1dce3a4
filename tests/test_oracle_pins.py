"""Pins of the fp64 oracle against what the pages and the mathematics fix.

None of these compares the oracle with itself: each expected value is a closed
form, a printed constant (tests/golden/, cited there), an invariant the pages
state, a library routine for a special case, or a second, independently
written statement (oracle/brute.py) on tiny inputs.  Each test names the
plausible mistake it catches.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import brute

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _gold(name):
    with open(os.path.join(GOLD, name)) as f:
        return json.load(f)


# --------------------------------------------------------------------------- rounding

def test_round_bf16_ties_and_double_rounding():
    r = oracle.round_bf16_scalar
    # tie between 1 and 1+2^-7 -> even mantissa (1.0)
    assert r(1 + 2**-8) == 1.0
    # tie between 1+2^-7 (odd) and 1+2^-6 (even) -> 1+2^-6
    assert r(1 + 3 * 2**-8) == 1 + 2**-6
    # just above the tie: must round up.  Rounding through float32 first would
    # drop the 2^-40 and turn it into a tie that goes down (double rounding).
    assert r(1 + 2**-8 + 2**-40) == 1 + 2**-7
    assert r(-(1 + 2**-8 + 2**-40)) == -(1 + 2**-7)
    # subnormals: spacing 2^-133
    assert r(2**-134) == 0.0
    assert r(3 * 2**-134) == 2**-132
    assert r(2**-133 * 5.4) == 5 * 2**-133
    # largest bf16 is 0x1.fe p127; the tie above it goes to infinity
    mx = float.fromhex("0x1.fep127")
    assert r(mx) == mx
    assert r(mx + 2.0**119) == math.inf
    assert r(mx + 2.0**118) == mx
    assert r(0.0) == 0.0 and math.isnan(r(math.nan))


def test_round_bf16_matches_torch_on_float32_values():
    # library cross-check: for values exactly representable in float32, torch's
    # float32 -> bfloat16 conversion is round-to-nearest-even too.
    g = np.random.default_rng(7)
    x = np.concatenate([g.standard_normal(20000), g.standard_normal(2000) * 1e-39,
                        g.standard_normal(2000) * 1e30]).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()
    got = oracle.round_to(x.astype(np.float64), oracle.BF16)
    np.testing.assert_array_equal(got, ref)


def test_round_f32():
    x = np.array([1 + 2**-24, 1 + 3 * 2**-24, 1 + 2**-24 + 2**-50])
    np.testing.assert_array_equal(oracle.round_to(x, oracle.F32), [1.0, 1 + 2**-22, 1 + 2**-23])


# --------------------------------------------------------------------------- RoPE

def test_rope_closed_forms_from_golden():
    for case in _gold("rope_closed_forms.json")["cases"]:
        D = case["D"]
        x = np.array(case["x"], dtype=np.float64).reshape(1, 1, D)
        got = oracle.rope(x, [case["pos"]])[0, 0]
        if "expect" in case:
            np.testing.assert_allclose(got, case["expect"], rtol=0, atol=1e-15, err_msg=case["what"])
        else:
            np.testing.assert_allclose(got[6:8], case["expect_pair3"], rtol=0, atol=1e-15,
                                       err_msg=case["what"])
            np.testing.assert_array_equal(got[:6], 0.0)


def test_rope_position_zero_is_identity():
    x = np.random.default_rng(1).standard_normal((3, 5, 64))
    np.testing.assert_array_equal(oracle.rope(x, [0, 0, 0]), x)


def test_rope_preserves_pair_norms():
    # "the rotation does not change the vector's length" (RoPE section of the
    # Tokenizer, KV Cache and RoPE page); a wrong sign in one entry breaks it.
    g = np.random.default_rng(2)
    x = g.standard_normal((50, 4, 128))
    pos = g.integers(0, 20000, size=50)
    y = oracle.rope(x, pos)
    n0 = x[..., 0::2] ** 2 + x[..., 1::2] ** 2
    n1 = y[..., 0::2] ** 2 + y[..., 1::2] ** 2
    np.testing.assert_allclose(n1, n0, rtol=1e-12, atol=0)


def test_rope_scores_depend_only_on_relative_position():
    # q_m . k_n after rotation depends on m - n only (angle linear in position).
    g = np.random.default_rng(3)
    q = g.standard_normal((1, 1, 128))
    k = g.standard_normal((1, 1, 128))
    for m, n, s in [(5, 3, 100), (0, 17, 4000), (1234, 1234, 77), (9000, 10, 3000)]:
        a = np.dot(oracle.rope(q, [m]).ravel(), oracle.rope(k, [n]).ravel())
        b = np.dot(oracle.rope(q, [m + s]).ravel(), oracle.rope(k, [n + s]).ravel())
        assert abs(a - b) <= 1e-9 * (abs(a) + 1)


def test_rope_composes_additively():
    g = np.random.default_rng(4)
    x = g.standard_normal((1, 2, 64))
    for a, b in [(3, 4), (100, 2000), (8191, 1)]:
        np.testing.assert_allclose(oracle.rope(oracle.rope(x, [a]), [b]), oracle.rope(x, [a + b]),
                                   rtol=0, atol=1e-11)


def test_rope_matches_complex_statement():
    g = np.random.default_rng(5)
    x = g.standard_normal((40, 3, 64))
    pos = g.integers(0, 16384, size=40)
    np.testing.assert_allclose(oracle.rope(x, pos), brute.rope_complex(x, pos), rtol=0, atol=1e-11)


def test_rope_base_parameter():
    # base 100, D=4: theta_1 = 100^(-1/2) = 0.1; position 10 -> 1 radian on pair 1
    x = np.array([0, 0, 1.0, 0]).reshape(1, 1, 4)
    got = oracle.rope(x, [10], base=100.0)[0, 0]
    np.testing.assert_allclose(got, [0, 0, math.cos(1), math.sin(1)], atol=1e-15)


# --------------------------------------------------------------------------- append

def test_append_slot_enumeration():
    # block table rows: seq 0 -> blocks [3, 1], seq 1 -> blocks [0, 2]; BS = 4.
    # slot = table[seq][p // 4] * 4 + p % 4, written out by hand:
    table = np.array([[3, 1], [0, 2]], dtype=np.int32)
    expect = {(0, 0): 12, (0, 3): 15, (0, 4): 4, (0, 5): 5, (0, 7): 7,
              (1, 0): 0, (1, 2): 2, (1, 4): 8, (1, 7): 11}
    c = oracle.Cache(4, 4, 2, 2, fill=np.nan)
    seqs = np.array([s for s, _ in expect], dtype=np.int32)
    pos = np.array([p for _, p in expect], dtype=np.int32)
    marks = np.arange(len(expect), dtype=np.float64)
    k = np.repeat(marks[:, None, None], 2, 1).repeat(2, 2)
    oracle.append(c, k, -k, pos, seqs, table)
    for i, ((s, p), slot) in enumerate(expect.items()):
        assert np.all(c.K[slot] == i) and np.all(c.V[slot] == -i)
    untouched = sorted(set(range(16)) - set(expect.values()))
    assert np.all(np.isnan(c.K[untouched])) and np.all(np.isnan(c.V[untouched]))


def test_append_rejects_out_of_range():
    c = oracle.Cache(2, 4, 1, 2)
    table = np.array([[1, -1]], dtype=np.int32)
    one = np.zeros((1, 1, 2))
    with pytest.raises(IndexError):
        oracle.append(c, one, one, [4], [0], table)      # block -1
    with pytest.raises(IndexError):
        oracle.append(c, one, one, [8], [0], table)      # past the table width
    with pytest.raises(IndexError):
        oracle.append(c, one, one, [0], [1], table)      # no such row


# --------------------------------------------------------------------------- attention

def _cache_from_seq(k, v, BS=4, perm_seed=0, extra_blocks=3):
    """Oracle cache holding one sequence's K/V rows at positions 0..N-1, blocks shuffled."""
    N, Hkv, D = k.shape
    nb = -(-N // BS)
    total = nb + extra_blocks
    blocks = np.random.default_rng(perm_seed).permutation(total)[:nb].astype(np.int32)
    table = blocks.reshape(1, -1)
    c = oracle.Cache(total, BS, Hkv, D)
    oracle.append(c, k, v, np.arange(N), np.zeros(N, dtype=np.int32), table)
    return c, table


def test_attention_closed_form_scale():
    case = _gold("attention_closed_forms.json")["cases"][0]
    k = np.array(case["k"]).reshape(2, 1, 4)
    v = np.array(case["v"]).reshape(2, 1, 4)
    c, table = _cache_from_seq(k, v)
    out = oracle.attend(c, np.array(case["q"]).reshape(1, 1, 4), [0], [1], table, 1)
    np.testing.assert_allclose(out[0, 0], case["expect"], rtol=0, atol=1e-15)
    # D=16: scale is 1/sqrt(16), not 1/16 and not 1/sqrt(hidden)
    case = _gold("attention_closed_forms.json")["cases"][1]
    D = 16
    k = np.zeros((2, 1, D)); k[0, 0, 0] = 1.0
    v = np.zeros((2, 1, D)); v[0, 0, 0] = 1.0; v[1, 0, 1] = 1.0
    q = np.zeros((1, 1, D)); q[0, 0, 0] = case["q_scale"]
    c, table = _cache_from_seq(k, v)
    out = oracle.attend(c, q, [0], [1], table, 1)
    np.testing.assert_allclose(out[0, 0, :2], case["expect_first_two"], rtol=0, atol=1e-15)


def test_single_cached_key_returns_v():
    g = np.random.default_rng(6)
    k, v = g.standard_normal((1, 2, 8)), g.standard_normal((1, 2, 8))
    c, table = _cache_from_seq(k, v)
    out = oracle.attend(c, g.standard_normal((1, 4, 8)) * 30, [0], [0], table, 4)
    for j in range(4):
        np.testing.assert_array_equal(out[0, j], v[0, j // 2])


def test_identical_keys_give_mean_of_v():
    g = np.random.default_rng(7)
    N = 37
    k = np.repeat(g.standard_normal((1, 1, 16)), N, 0)
    v = g.standard_normal((N, 1, 16))
    c, table = _cache_from_seq(k, v)
    out = oracle.attend(c, g.standard_normal((1, 1, 16)), [0], [N - 1], table, 1)
    np.testing.assert_allclose(out[0, 0], v[:, 0].mean(0), rtol=0, atol=1e-14)


def test_zero_query_gives_mean_of_v():
    g = np.random.default_rng(8)
    N = 29
    k, v = g.standard_normal((N, 2, 16)), g.standard_normal((N, 2, 16))
    c, table = _cache_from_seq(k, v)
    out = oracle.attend(c, np.zeros((1, 2, 16)), [0], [N - 1], table, 2)
    np.testing.assert_allclose(out[0, 1], v[:, 1].mean(0), rtol=0, atol=1e-14)


def test_dominant_key_with_huge_scores():
    # scores around 1e3 overflow exp() unless the max is subtracted first
    g = np.random.default_rng(9)
    N, D = 20, 8
    k = g.standard_normal((N, 1, D))
    q = np.zeros((1, 1, D)); q[0, 0, 0] = 1.0
    k[:, 0, 0] = 1000.0
    k[11, 0, 0] = 1300.0          # scores 500 vs 650 after 1/sqrt(8)... gap >= 100
    v = g.standard_normal((N, 1, D))
    c, table = _cache_from_seq(k, v)
    out = oracle.attend(c, q * math.sqrt(D) / 2, [0], [N - 1], table, 1)
    assert np.all(np.isfinite(out))
    np.testing.assert_allclose(out[0, 0], v[11, 0], rtol=0, atol=1e-12)


def test_causal_visibility_stops_at_own_position():
    # key p+1 carries an enormous score: a query at position p must not see it
    g = np.random.default_rng(10)
    N, D = 12, 8
    k, v = g.standard_normal((N, 1, D)), g.standard_normal((N, 1, D))
    k[7] = 0.0; k[7, 0, 0] = 1e4
    c, table = _cache_from_seq(k, v)
    q = np.zeros((1, 1, D)); q[0, 0, 0] = 1.0
    out6 = oracle.attend(c, q, [0], [6], table, 1)
    out7 = oracle.attend(c, q, [0], [7], table, 1)
    ref6 = brute.causal_attention_full(np.repeat(q, N, 0), k, v)[6]
    np.testing.assert_allclose(out6[0], ref6, atol=1e-13)
    np.testing.assert_allclose(out7[0, 0], v[7, 0], atol=1e-12)


def test_empty_sequence_gives_zero():
    c = oracle.Cache(2, 4, 1, 4, fill=np.nan)
    table = np.array([[1, 0]], dtype=np.int32)
    out = oracle.attend(c, np.ones((1, 1, 4)), [0], [-1], table, 1)
    np.testing.assert_array_equal(out, 0.0)


def test_gqa_equals_mha_with_repeated_kv_heads():
    g = np.random.default_rng(11)
    N, Hq, Hkv, D = 33, 8, 2, 16
    k, v = g.standard_normal((N, Hkv, D)), g.standard_normal((N, Hkv, D))
    q = g.standard_normal((1, Hq, D))
    c, table = _cache_from_seq(k, v)
    gqa = oracle.attend(c, q, [0], [N - 1], table, Hq)
    kr, vr = np.repeat(k, Hq // Hkv, axis=1), np.repeat(v, Hq // Hkv, axis=1)   # repeat_interleave
    c2, table2 = _cache_from_seq(kr, vr, perm_seed=5)
    mha = oracle.attend(c2, q, [0], [N - 1], table2, Hq)
    np.testing.assert_allclose(gqa, mha, rtol=0, atol=1e-14)


def test_block_table_permutation_invariance():
    g = np.random.default_rng(12)
    N = 45
    k, v = g.standard_normal((N, 2, 8)), g.standard_normal((N, 2, 8))
    q = g.standard_normal((1, 2, 8))
    outs = []
    for seed in range(4):
        c, table = _cache_from_seq(k, v, BS=4, perm_seed=seed, extra_blocks=7)
        outs.append(oracle.attend(c, q, [0], [N - 1], table, 2))
    for o in outs[1:]:
        np.testing.assert_array_equal(o, outs[0])


def test_threads_do_not_change_results():
    g = np.random.default_rng(13)
    N = 60
    k, v = g.standard_normal((N, 2, 16)), g.standard_normal((N, 2, 16))
    q = g.standard_normal((5, 4, 16))
    c, table = _cache_from_seq(k, v)
    pos = [59, 3, 0, 31, 44]
    a = oracle.attend(c, q, [0] * 5, pos, table, 4, nthreads=1)
    b = oracle.attend(c, q, [0] * 5, pos, table, 4, nthreads=7)
    np.testing.assert_array_equal(a, b)


@pytest.mark.parametrize("D,Hq,Hkv,N", [(4, 2, 1, 9), (8, 4, 4, 40), (64, 4, 2, 23)])
def test_cached_decode_equals_full_recomputation(D, Hq, Hkv, N):
    """Token-by-token: rope + round + append + attend over the cache equals the
    complex-number RoPE of the whole sequence with full causal attention."""
    g = np.random.default_rng(100 + D)
    raw_q = g.standard_normal((N, Hq, D))
    raw_k = g.standard_normal((N, Hkv, D))
    raw_v = g.standard_normal((N, Hkv, D))
    BS = 4
    nb = -(-N // BS)
    table = np.random.default_rng(1).permutation(nb + 2)[:nb].astype(np.int32).reshape(1, -1)
    c = oracle.Cache(nb + 2, BS, Hkv, D)
    outs = []
    for p in range(N):
        qh = oracle.rope(raw_q[p:p + 1], [p])
        kh = oracle.rope(raw_k[p:p + 1], [p])
        oracle.append(c, kh, raw_v[p:p + 1], [p], [0], table)
        outs.append(oracle.attend(c, qh, [0], [p], table, Hq)[0])
    pos = np.arange(N)
    ref = brute.causal_attention_full(brute.rope_complex(raw_q, pos), brute.rope_complex(raw_k, pos), raw_v)
    np.testing.assert_allclose(np.stack(outs), ref, rtol=0, atol=1e-12)


def test_chunk_equals_successive_decodes_and_two_sequences():
    g = np.random.default_rng(14)
    D, Hq, Hkv, BS = 8, 4, 2, 4
    lens = [19, 26]
    prefix = [7, 13]
    nb = [-(-n // BS) for n in lens]
    perm = np.random.default_rng(3).permutation(sum(nb) + 3).astype(np.int32)
    table = np.full((2, max(nb)), -1, dtype=np.int32)
    table[0, :nb[0]] = perm[:nb[0]]
    table[1, :nb[1]] = perm[nb[0]:nb[0] + nb[1]]
    c = oracle.Cache(sum(nb) + 3, BS, Hkv, D)
    raws = []
    for s, n in enumerate(lens):
        rq, rk, rv = g.standard_normal((n, Hq, D)), g.standard_normal((n, Hkv, D)), g.standard_normal((n, Hkv, D))
        raws.append((rq, rk, rv))
        pos = np.arange(n)
        oracle.append(c, oracle.rope(rk, pos), rv, pos, np.full(n, s, dtype=np.int32), table)
    # one call: both chunks' query rows (prefix..len-1) against the cache
    rows, qpos, qs = [], [], []
    for s, n in enumerate(lens):
        for p in range(prefix[s], n):
            rows.append(s); qpos.append(p)
            qs.append(oracle.rope(raws[s][0][p:p + 1], [p])[0])
    chunk = oracle.attend(c, np.stack(qs), rows, qpos, table, Hq)
    i = 0
    for s, n in enumerate(lens):
        pos = np.arange(n)
        ref = brute.causal_attention_full(brute.rope_complex(raws[s][0], pos),
                                          brute.rope_complex(raws[s][1], pos), raws[s][2])
        np.testing.assert_allclose(chunk[i:i + n - prefix[s]], ref[prefix[s]:], rtol=0, atol=1e-12)
        i += n - prefix[s]


def test_prefix_zero_chunk_matches_torch_softmax_with_explicit_mask():
    # library cross-check (not the oracle): textbook causal attention in torch fp64
    g = np.random.default_rng(15)
    N, H, D = 17, 2, 16
    q, k, v = g.standard_normal((N, H, D)), g.standard_normal((N, H, D)), g.standard_normal((N, H, D))
    c, table = _cache_from_seq(k, v, BS=4)
    got = oracle.attend(c, q, [0] * N, list(range(N)), table, H)
    tq, tk, tv = (torch.from_numpy(a).permute(1, 0, 2) for a in (q, k, v))
    s = tq @ tk.transpose(1, 2) / math.sqrt(D)
    mask = torch.ones(N, N, dtype=torch.bool).tril()
    s = s.masked_fill(~mask, float("-inf"))
    ref = (torch.softmax(s, dim=-1) @ tv).permute(1, 0, 2).numpy()
    np.testing.assert_allclose(got, ref, rtol=0, atol=1e-13)


# --------------------------------------------------------------------------- byte accounting

def test_kv_bytes_closed_form_from_page():
    import workloads

    gold = _gold("kv_bytes.json")
    wl = workloads.Workload("x", "x", "bf16", gold["kv_heads"], gold["kv_heads"], gold["head_dim"],
                            "paged", 16, 1, (0, 0))
    per_layer = workloads.kv_bytes_read(wl, [gold["tokens"]])
    assert per_layer * gold["layers"] == gold["expect_bytes"] == 2**30
    assert abs(gold["expect_bytes"] / 1e9 - gold["expect_gb_approx"]) < 0.01


# --------------------------------------------------------------------------- fp8 (e4m3) cache rows

def test_e4m3_decode_matches_the_format_definition():
    """Catches a wrong exponent bias, a missing implicit 1, or subnormals
    decoded as normals: spot codes from the bit layout, and every code against
    the library's float8_e4m3fn decoding."""
    from oracle import fp8

    d = fp8.e4m3_decode
    assert d(0x00) == 0.0 and d(0x01) == 2.0 ** -9 and d(0x07) == 7 * 2.0 ** -9
    assert d(0x08) == 2.0 ** -6 and d(0x38) == 1.0 and d(0x39) == 1.125
    assert d(0x7E) == 448.0 and d(0xFE) == -448.0 and np.isnan(d(0x7F)) and np.isnan(d(0xFF))
    codes = np.arange(256, dtype=np.uint8)
    lib = torch.from_numpy(codes).view(torch.float8_e4m3fn).double().numpy()
    ours = d(codes)
    assert np.array_equal(np.isnan(lib), np.isnan(ours))
    ok = ~np.isnan(ours)
    assert np.array_equal(ours[ok], lib[ok])


def test_e4m3_encode_rounding_and_saturation():
    """Catches round-half-up instead of ties-to-even, truncation, a wrong grid
    spacing at binade edges, and overflow to NaN instead of saturation."""
    from oracle import fp8

    e = fp8.e4m3_encode
    codes = np.arange(256, dtype=np.uint8)
    vals = fp8.e4m3_decode(codes)
    finite = ~np.isnan(vals)
    # every finite code round-trips (sign of zero included)
    assert np.array_equal(e(vals[finite]), codes[finite])
    # ties go to the even mantissa: 1 + 1/16 -> 1.0, 1 + 3/16 -> 1.25, 2^-6 + 2^-10 (subnormal spacing tie) -> 2^-6
    assert fp8.e4m3_decode(e(1.0625)) == 1.0
    assert fp8.e4m3_decode(e(1.1875)) == 1.25
    assert fp8.e4m3_decode(e(2.0 ** -10)) == 0.0 and fp8.e4m3_decode(e(3 * 2.0 ** -10)) == 2 * 2.0 ** -9
    # just past a tie rounds away from the even neighbour
    assert fp8.e4m3_decode(e(1.0625 + 2.0 ** -30)) == 1.125
    # saturation at 448 (no infinities), both signs
    assert e(500.0) == 0x7E and e(1e30) == 0x7E and e(-1e30) == 0xFE and e(464.0) == 0x7E
    # against the library's round-to-nearest-even conversion of in-range values
    g = np.random.default_rng(5)
    x = np.concatenate([g.standard_normal(20000) * 50, g.standard_normal(20000) * 0.01,
                        (vals[finite][:-1] + np.diff(vals[finite])[:] / 2)[np.abs(vals[finite][:-1]) < 400]])
    x = x[np.abs(x) < 448].astype(np.float32).astype(np.float64)
    lib = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(e(x), lib)


def test_fp8_row_quantisation_bounds():
    """Catches a scale computed from the wrong row, a missing inverse, or codes
    not saturating: the largest element of a row maps to +-448, and every
    dequantised value is within half an e4m3 step of the row value."""
    from oracle import fp8

    g = np.random.default_rng(6)
    r = torch.from_numpy(g.standard_normal((300, 8, 128)) * np.exp(g.standard_normal((300, 8, 1)))).to(
        torch.bfloat16).double().numpy()
    r[0, 0] = 0.0                       # an all-zero row: scale 1, codes 0
    codes, scale = fp8.quantize_rows(r)
    assert codes.dtype == np.uint8 and scale.dtype == np.float32 and scale.shape == (300, 8)
    assert scale[0, 0] == 1.0 and (codes[0, 0] & 0x7F).max() == 0
    amax = np.abs(r).max(-1)
    assert np.array_equal(scale[1:], (amax[1:].astype(np.float32) / np.float32(448)))
    arg = np.abs(r).argmax(-1)
    top = np.take_along_axis(codes, arg[..., None], -1)[..., 0]
    assert np.all((top[1:] & 0x7F) == 0x7E)
    deq = fp8.dequantize_rows(codes, scale)
    err = np.abs(deq - r)
    # normal range: half a step is 2^-4 of the magnitude; subnormal: 2^-10 * scale; plus fp32 rounding of r * inv
    bound = np.maximum(np.abs(r) * 2.0 ** -4, 2.0 ** -10 * scale[..., None].astype(np.float64)) * (1 + 2.0 ** -20)
    assert np.all(err <= bound + 1e-30)
