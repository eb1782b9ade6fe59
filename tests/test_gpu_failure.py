"""Failure detection without a GPU fault: a bounded device-side wait runs out (a barrier that
nothing arrives at), the host reads TP_ERR_DEVICE_TIMEOUT from tp_sync, and the context stays
usable for the next forward."""
import pytest
import torch

from megatron_tensor_transformer_gb300 import tpx
from tests.test_gpu_parity import Mlp, bits, check_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from megatron_tensor_transformer_gb300 import build
    build.build_library()
    tpx.lib()
    torch.cuda.set_device(0)
    return torch.device("cuda:0")


def test_bounded_wait_reports_and_context_survives(dev):
    assert tpx.tp_sync(timeout_ms=10000) == tpx.TP_OK        # nothing pending, no error word
    tpx.tp_selftest_bounded_wait(2000)                         # gives up after 2 ms
    assert tpx.tp_sync(timeout_ms=10000) == tpx.TP_ERR_DEVICE_TIMEOUT
    assert tpx.tp_sync(timeout_ms=10000) == tpx.TP_OK          # read once, then cleared
    m = Mlp(1024, 4096, 8, 16, dev, seed=9)                    # the context still computes
    y, _ = m.run()
    y_ref, _ = m.oracle()
    check_close(bits(y), y_ref, what="after a device timeout")


def test_sync_deadline(dev):
    """tp_sync with a deadline shorter than the queued work reports TP_ERR_TIMEOUT without
    cancelling the work, which then completes."""
    a = torch.randn(4096, 4096, device=dev)
    for _ in range(20):
        a = a @ a.T / 64.0
    st = tpx.tp_sync(timeout_ms=0)
    assert st in (tpx.TP_ERR_TIMEOUT, tpx.TP_OK)
    assert tpx.tp_sync(timeout_ms=20000) == tpx.TP_OK


def test_selftest_argument_checks(dev):
    with pytest.raises(tpx.TpxError):
        tpx.tp_selftest_bounded_wait(0)
