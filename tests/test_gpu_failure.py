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


def test_bounded_counter_wait_reports_timeout(zopt):
    """The fused kernel's wait on a per-matrix completion counter runs out the same way: the
    next fused call (two shapes in one launch) reports ZOPT_ETIMEOUT once, then works."""
    assert zopt.take_device_error() in (0, 1)
    zopt.selftest_count_timeout(50_000_000)
    torch.cuda.synchronize()
    pairs = [(torch.randn(2, 256, 768, device="cuda").bfloat16(), torch.empty(2, 256, 768, device="cuda",
                                                                             dtype=torch.bfloat16)),
             (torch.randn(1, 768, 256, device="cuda").bfloat16(), torch.empty(1, 768, 256, device="cuda",
                                                                             dtype=torch.bfloat16))]
    ws = zopt.new_ns_workspace_many([(256, 768, 2), (768, 256, 1)])
    with pytest.raises(zopt.ZoptError) as e:
        zopt.ns_orthogonalize_many(pairs, ws)
    assert e.value.status == 4
    zopt.ns_orthogonalize_many(pairs, ws)
    torch.cuda.synchronize()
    assert all(torch.isfinite(X.float()).all() for _, X in pairs)


def test_selftest_rejects_long_limits(zopt):
    with pytest.raises(zopt.ZoptError):
        zopt.selftest_wait_timeout(10_000_000_000)
    with pytest.raises(zopt.ZoptError):
        zopt.selftest_count_timeout(10_000_000_000)
