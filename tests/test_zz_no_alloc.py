"""kvattn_decode_static_scratch: the decode entry point that allocates nothing.

It exists for callers that cannot allocate device memory when they run a
decode step (an engine whose HBM is already committed to its own KV pool and
arenas, or an operator inside a host framework with no device allocator that
must not call cudaMalloc/cudaFree mid-step).  Its partial results live in a
fixed 32 MiB array inside the library, placed on the device by the first call.

The GPU test calls it through the C ABI twice in a row, on two different
batches (the second with an explicit split count of 16, so that more of the
array is in use), and checks each result bit for bit against kvattn_decode
with a caller workspace on the same inputs (both run the same plan and
kernels, so a stale or overlapping scratch slot would show), and against the
fp64 oracle within the attention tolerance of the other decode tests.  It also
checks that calls after the set-up take no device memory.  The file is named
to be collected last.
"""
import ctypes

import numpy as np
import pytest
import torch

import workloads
from _gpu_support import DecodeCase, compare, f64

FAKE = ctypes.c_void_p(0x7F0000001000)  # never dereferenced: the host checks refuse these calls


def _static_decode(kv, case, q, num_splits, out=None):
    out = torch.empty_like(q) if out is None else out
    code = kv.lib.kvattn_decode_static_scratch(
        ctypes.byref(case.cfg), ctypes.byref(case.cache.desc), ctypes.c_void_p(q.data_ptr()),
        ctypes.c_void_p(case.d_table.data_ptr()), case.d_table.shape[1],
        ctypes.c_void_p(case.seq_lens.data_ptr()), q.shape[0], case.max_len, num_splits,
        ctypes.c_void_p(out.data_ptr()), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    kv.check(code, "kvattn_decode_static_scratch")
    return out


@pytest.mark.gpu
def test_static_scratch_decode_twice_matches_workspace_decode_and_oracle(kvattn_lib):
    kv = kvattn_lib
    # the set-up form places the array and resolves its address, nothing else
    setup = kv.lib.kvattn_decode_static_scratch(None, None, None, None, 0, None, 0, 0, 0, None, None)
    assert kv.STATUS[setup] == "KVATTN_OK"
    wl = workloads.WORKLOADS["c4"]
    runs = [([0, 5, 9, 40, 77, 120, 200, 255], 0), ([1, 2, 3, 100], 16)]
    for rows, splits in runs:
        case = DecodeCase(wl, workloads.make_batch(wl, num_blocks=1 << 18, rows_subset=rows), range(len(rows)))
        q, ref_gpu = case.run(num_splits=splits)   # rope_append, then kvattn_decode with a workspace
        assert kv.get_device_status() == 0
        out = torch.empty_like(q)
        torch.cuda.synchronize()
        free0 = torch.cuda.mem_get_info()[0]
        got = _static_decode(kv, case, q, splits, out)      # same rotated q, same cache
        torch.cuda.synchronize()
        assert torch.cuda.mem_get_info()[0] == free0, "the call took device memory"
        assert kv.get_device_status() == 0
        assert torch.equal(got, ref_gpu), f"rows {rows}: differs from kvattn_decode with a workspace"
        _, ref = case.expected()
        compare(f64(got), ref, "bf16", f"static-scratch decode, rows {rows}, splits {splits}")
        del case
        torch.cuda.empty_cache()


def test_static_scratch_host_checks():
    """Refusals made on the host, before any device work (no GPU needed):
    the codes of kvattn_decode, then the 32 MiB limit of the array."""
    import kv_cache_attention_rope_gb300 as kv

    E = kv.STATUS_CODE
    desc = kv.CacheDesc(FAKE, FAKE, 16, 16)

    def call(cfg, B, maxlen=64, splits=0, cache=desc, out=FAKE):
        return kv.lib.kvattn_decode_static_scratch(ctypes.byref(cfg) if cfg is not None else None,
                                                   ctypes.byref(cache) if cache is not None else None,
                                                   FAKE, FAKE, 4096, FAKE, B, maxlen, splits, out, None)

    good = kv.make_config(32, 8, 128, kv.BF16)
    assert call(kv.make_config(32, 8, 80, kv.BF16), 4) == E["KVATTN_ERR_UNSUPPORTED"]
    assert call(kv.make_config(32, 5, 128, kv.BF16), 4) == E["KVATTN_ERR_UNSUPPORTED"]
    assert call(good, 8193) == E["KVATTN_ERR_UNSUPPORTED"]
    assert call(None, 4) == E["KVATTN_ERR_INVALID_ARG"]
    assert call(good, -1) == E["KVATTN_ERR_INVALID_ARG"]
    assert call(good, 4, out=None) == E["KVATTN_ERR_INVALID_ARG"]
    assert call(good, 4, cache=kv.CacheDesc(FAKE, None, 16, 16)) == E["KVATTN_ERR_INVALID_ARG"]
    assert call(good, 0) == E["KVATTN_OK"]
    big = kv.decode_workspace_size(good, 8192, 65536, 64)
    assert big > 32 << 20
    assert call(good, 8192, 65536, 64) == E["KVATTN_ERR_WORKSPACE_TOO_SMALL"]
