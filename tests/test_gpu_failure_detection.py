"""Failure detection on the GPU without a GPU fault: a wait that runs out is
reported through the device status word, and the context stays usable."""
import pytest
import torch

pytestmark = pytest.mark.gpu


def test_bounded_wait_reports_timeout_and_context_survives(kvattn_lib):
    kv = kvattn_lib
    assert kv.get_device_status() == 0
    kv.selftest_wait_timeout(2000)          # 2 ms on a barrier nothing completes
    assert kv.STATUS[kv.get_device_status()] == "KVATTN_ERR_TIMEOUT"
    assert kv.get_device_status() == 0      # read clears it
    # the context still runs work: a small decode afterwards succeeds
    dev = torch.device("cuda")
    cfg = kv.make_config(4, 4, 64, kv.BF16)
    cache = kv.Cache.empty(4, 4, 16, 64, torch.bfloat16, dev)
    cache.k_pool.normal_(); cache.v_pool.normal_()
    table = torch.tensor([[0, 1]], dtype=torch.int32, device=dev)
    out = kv.decode(cfg, cache, torch.randn(1, 4, 64, device=dev).to(torch.bfloat16), table,
                    torch.tensor([20], dtype=torch.int32, device=dev), 32)
    assert kv.get_device_status() == 0 and torch.isfinite(out.float()).all()


def test_selftest_limit_validated(kvattn_lib):
    kv = kvattn_lib
    with pytest.raises(kv.KvattnError):
        kv.selftest_wait_timeout(0)
    with pytest.raises(kv.KvattnError):
        kv.selftest_wait_timeout(2_000_000)
