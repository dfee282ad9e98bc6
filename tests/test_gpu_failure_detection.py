"""Failure detection on the GPU without a fault: a kernel whose bounded wait
runs out (an mbarrier nothing arrives on) records a timeout that the host
reads through gdn_device_status; the context stays usable and the next
prefill is correct."""
import pytest
import torch

from gated_deltanet_mixer_gb300 import gdn
from gated_deltanet_mixer_gb300 import inputs as I

from gpu_harness import compare_prefill, gpu_prefill

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from gated_deltanet_mixer_gb300 import build
    build.build()
    gdn.lib()
    assert torch.cuda.is_available()


def test_wait_timeout_is_reported_and_context_survives():
    assert gdn.gdn_device_status(reset=True) == gdn.GDN_OK
    gdn.gdn_selftest_wait_timeout(20000)  # 20 ms
    assert gdn.gdn_device_status() == gdn.GDN_ERR_TIMEOUT
    # the record stays until reset
    assert gdn.gdn_device_status(reset=True) == gdn.GDN_ERR_TIMEOUT
    assert gdn.gdn_device_status() == gdn.GDN_OK
    # the context still runs kernels: a small prefill against the oracle
    p = I.prefill_problem(1, 70, 1, 2, io="bf16", case=90)
    compare_prefill(p, gpu_prefill(p))
    assert gdn.gdn_device_status() == gdn.GDN_OK


def test_selftest_rejects_bad_limits():
    for us in (0, -5, 1000001):
        with pytest.raises(gdn.GdnError) as e:
            gdn.gdn_selftest_wait_timeout(us)
        assert e.value.status == gdn.GDN_ERR_INVALID_ARG
