"""Failure detection on the GPU without a fault: a bounded on-device wait that runs out reports
KVE_ETIMEOUT through the device error word, and the context stays usable afterwards."""
import pytest
import torch

from kv_cache_eviction_02_gb300 import api

pytestmark = pytest.mark.gpu


def test_bounded_wait_timeout_is_reported_and_context_survives():
    api.kve_check_device()                      # clean start
    api.kve_selftest_wait_timeout(50)           # a barrier nothing signals, 50 ms limit
    with pytest.raises(api.KveError) as e:
        api.kve_check_device()
    assert e.value.status == api.KVE_ETIMEOUT
    api.kve_check_device()                      # the word was cleared
    x = torch.arange(1024, device="cuda", dtype=torch.float32)
    assert float(x.sum()) == 1023 * 1024 / 2    # the context is still usable


def test_selftest_rejects_bad_limits():
    with pytest.raises(api.KveError) as e:
        api.kve_selftest_wait_timeout(0)
    assert e.value.status == api.KVE_EINVAL


def test_injected_failure_reaches_python_on_a_gpu_call():
    api.kve_inject_failure(api.KVE_ECUDA, 1)
    with pytest.raises(api.KveError) as e:
        api.kve_selftest_wait_timeout(5)
    assert e.value.status == api.KVE_ECUDA
    api.kve_check_device()
