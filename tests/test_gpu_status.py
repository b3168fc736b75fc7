"""Failure reporting without faulting the GPU: a bounded device-side wait on
an mbarrier that nothing arrives on gives up, records a timeout in the
library's device error word and the kernel returns normally; the context
stays usable."""
import pytest
import torch

pytestmark = pytest.mark.gpu


def test_bounded_wait_reports_timeout_and_context_survives():
    import int8_convrot_w8a8_gb300 as cr
    assert cr.convrot_get_device_status() == 0
    cr.convrot_selftest_wait_timeout(2000)
    assert cr.convrot_get_device_status() == 5   # CONVROT_ERR_TIMEOUT
    assert cr.convrot_get_device_status() == 0   # read clears the word
    x = torch.ones(1024, device="cuda")
    assert float(x.sum()) == 1024.0


def test_library_errors_raise():
    import int8_convrot_w8a8_gb300 as cr
    X = torch.zeros((4, 2688), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(cr.ConvRotError) as e:
        cr.convrot_quantize_act(X, 256, "h4")
    assert e.value.status == 2
