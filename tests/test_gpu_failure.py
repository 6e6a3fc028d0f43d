"""Failure detection on the GPU without a fault: a bounded device-side wait
that nothing satisfies gives up, records TPS_ERR_TIMEOUT in the device error
word and returns; the context stays usable for the next launch."""
import pytest
import torch

from backward_tcgen05_tma_gemms_gb300 import api, inputs

pytestmark = pytest.mark.gpu


def test_wait_timeout_is_reported_and_context_survives(orc):
    assert api.last_device_error() == 0
    api.selftest_wait_timeout(50_000_000)          # 50 ms
    assert api.last_device_error() == api.ERR_TIMEOUT
    assert api.last_device_error() == 0            # reading cleared the word
    A, B, G = inputs.matmul_case(0, 64, 32, 48)
    Y, dA, dB = api.matmul_fwd_bwd(A.cuda(), B.cuda(), G.cuda(), 2, "rows")
    assert api.last_device_error() == 0
    ref = orc.matmul(A.double().numpy(), B.double().numpy(), G.double().numpy())
    assert abs(Y.cpu().double().numpy() - ref[0]).max() < 1e-4 * abs(ref[0]).max()


def test_selftest_rejects_bad_limit():
    with pytest.raises(api.TpsError):
        api.selftest_wait_timeout(0)
