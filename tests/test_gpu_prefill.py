"""GPU parity of the tcgen05 chunked-prefill kernel against the fp64 oracle.

Tolerance: bf16 output, max abs <= 1e-2 and relative L2 <= 5e-3 against the
exact attention of the correctly rounded q/k/v.  Pools are NaN-filled, so a
stale cache slot that leaks into a result fails the test.
"""
import numpy as np
import pytest
import torch

import workloads
from _gpu_support import PrefillCase, compare, f64

pytestmark = pytest.mark.gpu


def _check(kv, case, rows=None, what="prefill"):
    _, out = case.run()
    assert kv.get_device_status() == 0
    rows, ref = case.expected(rows)
    return compare(f64(out)[rows], ref, "bf16", what)


def test_causal_no_prefix_two_query_tiles(kvattn_lib):
    _check(kvattn_lib, PrefillCase(4, 2, [0], [200]), what="prefix 0, 200 rows")


@pytest.mark.parametrize("prefixes,qlens", [
    ([300], [130]),                   # prefix not a multiple of 16 / 128
    ([0, 17, 128, 1000], [1, 128, 129, 64]),   # ragged chunks, one-row chunk
    ([5, 4096], [512, 3]),
])
def test_prefixes_and_ragged_chunks(kvattn_lib, prefixes, qlens):
    _check(kvattn_lib, PrefillCase(8, 2, prefixes, qlens, seed=len(prefixes)), what=f"{prefixes}/{qlens}")


def test_mha_and_block_size_32(kvattn_lib):
    _check(kvattn_lib, PrefillCase(4, 4, [50, 333], [77, 200], block_size=32, seed=3), what="MHA, BS 32")


def test_running_max_rescale(kvattn_lib):
    """Keys whose scale grows along the sequence push each row's max up by far
    more than 2^8 from tile to tile, so the accumulated output is rescaled.

    Scores here reach +-16, so a row's softmax is dominated by a few keys and
    the bf16 rounding of the probabilities fed to the tensor-core P.V product
    (P must share V's type) does not average out: each normalised weight is off
    by at most ~2^-8 relative, so |out - exact| <= 2^-8 (max|v| + |exact|).
    That derived bound replaces the 1e-2 absolute bar, which is stated for the
    N(0,1) workloads; the relative L2 bar is kept."""
    kv = kvattn_lib
    case = PrefillCase(4, 1, [0], [600], seed=4, k_scale=lambda t: 1.0 + t / 40.0)
    _, out = case.run()
    assert kv.get_device_status() == 0
    rows, ref = case.expected()
    got = f64(out)[rows]
    vmax = float(case.v_raw.abs().max())
    bound = 2.0 ** -8 * (vmax + np.abs(ref))
    assert np.all(np.abs(got - ref) <= bound), float(np.max(np.abs(got - ref) - bound))
    assert np.linalg.norm(got - ref) / np.linalg.norm(ref) <= 5e-3


def test_c5_chunks_sampled_rows(kvattn_lib):
    """Two chunks of the mixed workload (their prefixes, 512 queries, 32/8 x 128)."""
    wl = workloads.WORKLOADS["c5"]
    _, pre = workloads.lengths(wl)
    idx = [int(np.argmin(pre)), int(np.argmax(pre))]
    case = PrefillCase(32, 8, [int(pre[i]) for i in idx], [512, 512], seed=5)
    rows = np.arange(0, 1024, 13)
    _check(kvattn_lib, case, rows=rows, what="c5 chunks")


def test_persistent_schedule_many_items(kvattn_lib):
    """More work items (chunk x 256-row block x head: 384) than SMs, of mixed
    lengths and with empty blocks (chunks of 256 rows or fewer), so each
    persistent CTA runs several items back to back in length order."""
    prefixes = [3000, 0, 700, 1500, 64, 2222]
    qlens = [512, 300, 17, 512, 256, 1]
    case = PrefillCase(32, 8, prefixes, qlens, seed=6)
    rows = np.arange(0, int(sum(qlens)), 7)
    _check(kvattn_lib, case, rows=rows, what="persistent schedule")


def test_unsorted_schedule_many_chunks(kvattn_lib):
    """1100 one-token chunks: more (chunk, 256-row block) pairs than the
    kernel ranks in shared memory, so items run in launch order."""
    g = np.random.default_rng(7)
    n = 1100
    prefixes = [int(p) for p in g.integers(0, 200, n)]
    case = PrefillCase(4, 1, prefixes, [1] * n, seed=7)
    rows = np.arange(0, n, 11)
    _check(kvattn_lib, case, rows=rows, what="unsorted schedule")


@pytest.mark.parametrize("hq,hkv,block_size", [(12, 12, 16), (16, 4, 16), (12, 12, 1040)])
def test_head_dim_64_gpt2_shape(kvattn_lib, hq, hkv, block_size):
    """Head dim 64 (GPT-2: 12 heads x 64, and a grouped variant): chunks over
    prefixes drawn like the GPT-2-shape decode workload (past U[1, 1024]), on a
    paged cache of 16-token blocks and on one of 1040-token blocks (the
    contiguous layout's row size rounded to a multiple of 16)."""
    g = np.random.default_rng(64 + hkv)
    prefixes = [int(p) for p in g.integers(1, 1025, 6)]
    qlens = [130, 1, 64, 257, 17, 16]
    case = PrefillCase(hq, hkv, prefixes, qlens, block_size=block_size, seed=64, head_dim=64,
                       extra_blocks=5 if block_size == 16 else 1)
    rows = np.arange(0, int(sum(qlens)), 3)
    _check(kvattn_lib, case, rows=rows, what=f"D=64 {hq}/{hkv} BS {block_size}")


def test_head_dim_64_full_chunk_no_prefix(kvattn_lib):
    """A whole 512-token GPT-2 prompt as one chunk (prefix 0), every row checked."""
    _check(kvattn_lib, PrefillCase(12, 12, [0], [512], seed=65, head_dim=64), what="D=64 prompt")
