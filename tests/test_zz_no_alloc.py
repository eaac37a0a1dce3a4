"""kvattn_decode_static_scratch: the decode entry point that allocates nothing.

It exists for callers that cannot allocate device memory when they run a
decode step (an engine whose HBM is already committed to its own KV pool and
arenas, or an operator inside a host framework with no device allocator that
must not call cudaMalloc/cudaFree mid-step).  Its partial results live in a
fixed 32 MiB array inside the library.  This test calls it through the C ABI
twice in a row, on two different batches, and checks each result against
kvattn_decode with a caller workspace on the same inputs, within the
attention tolerance of the other decode tests.  The file is named to be
collected last.
"""
import ctypes

import numpy as np
import pytest
import torch

import workloads
from _gpu_support import DecodeCase, compare, f64

pytestmark = pytest.mark.gpu


def _static_decode(kv, case, q):
    out = torch.empty_like(q)
    code = kv.lib.kvattn_decode_static_scratch(
        ctypes.byref(case.cfg), ctypes.byref(case.cache.desc), ctypes.c_void_p(q.data_ptr()),
        ctypes.c_void_p(case.d_table.data_ptr()), case.d_table.shape[1],
        ctypes.c_void_p(case.seq_lens.data_ptr()), q.shape[0], case.max_len, 0,
        ctypes.c_void_p(out.data_ptr()), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    kv.check(code, "kvattn_decode_static_scratch")
    return out


def test_static_scratch_decode_matches_workspace_decode_twice(kvattn_lib):
    kv = kvattn_lib
    wl = workloads.WORKLOADS["c4"]
    cases = [DecodeCase(wl, workloads.make_batch(wl, num_blocks=1 << 18, rows_subset=rows), [])
             for rows in ([0, 5, 9, 40, 77, 120, 200, 255], [1, 2, 3, 100])]
    for case in cases:
        q, ref = case.run()                     # rope_append, then kvattn_decode with a workspace
        assert kv.get_device_status() == 0
        got = _static_decode(kv, case, q)       # same rotated q, same cache
        assert kv.get_device_status() == 0
        compare(f64(got), f64(ref).astype(np.float64), "bf16", "static-scratch decode")


def test_static_scratch_rejects_requests_beyond_its_size(kvattn_lib):
    kv = kvattn_lib
    cfg = kv.make_config(32, 8, 128, kv.BF16)
    big = kv.decode_workspace_size(cfg, 8192, 65536, 64)
    assert big > 32 << 20
    desc = kv.CacheDesc(ctypes.c_void_p(0x7F0000001000), ctypes.c_void_p(0x7F0000001000), 16, 16)
    fake = ctypes.c_void_p(0x7F0000001000)     # never dereferenced: refused on the host
    code = kv.lib.kvattn_decode_static_scratch(ctypes.byref(cfg), ctypes.byref(desc), fake, fake, 4096, fake,
                                               8192, 65536, 64, fake, None)
    assert kv.STATUS[code] == "KVATTN_ERR_WORKSPACE_TOO_SMALL"
