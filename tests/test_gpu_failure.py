"""Failure detection on the GPU without a fault: a bounded mbarrier wait that nothing
completes runs out after its limit, reports through the device error word, and leaves the
context usable — the next Newton-Schulz call reports ZOPT_ETIMEOUT once, and later calls work."""
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _clear_error_word(zopt):
    yield
    torch.cuda.synchronize()
    zopt.take_device_error()  # never leave a reported timeout for the tests that follow


def test_bounded_wait_reports_timeout_and_context_survives(zopt):
    assert zopt.take_device_error() in (0, 1)  # clear anything left over
    zopt.selftest_wait_timeout(50_000_000)  # 50 ms
    torch.cuda.synchronize()  # the kernel returned by itself
    G = torch.randn(256, 512, device="cuda").bfloat16()
    X = torch.empty_like(G)
    ws = zopt.new_ns_workspace(256, 512)
    with pytest.raises(zopt.ZoptError) as e:
        zopt.ns_orthogonalize(G, X, ws)
    assert e.value.status == 4  # ZOPT_ETIMEOUT
    zopt.ns_orthogonalize(G, X, ws)  # reported once; the context still works
    torch.cuda.synchronize()
    assert torch.isfinite(X.float()).all()
    zopt.selftest_wait_timeout(20_000_000)
    torch.cuda.synchronize()
    assert zopt.take_device_error() == 1 and zopt.take_device_error() == 0


def test_selftest_rejects_long_limits(zopt):
    with pytest.raises(zopt.ZoptError):
        zopt.selftest_wait_timeout(10_000_000_000)
