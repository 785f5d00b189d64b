"""Bounded device-side waits: a wait that nothing completes gives up, records
TPMLP_ERR_TIMEOUT, and the context stays usable (GPU; nothing faults or hangs)."""
import pytest

pytestmark = pytest.mark.gpu


def test_wait_timeout_is_reported_and_cleared():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from megatron_tensor_mlp_gb300 import harness, synth, tpmlp as T
    assert T.tpmlp_device_status(check=False) == T.OK
    T.tpmlp_debug_wait_timeout(20000)  # 20 ms limit
    assert T.tpmlp_device_status(check=False) == T.ERR_TIMEOUT
    assert "gave up" in T.last_error()
    assert T.tpmlp_device_status(check=False) == T.OK  # cleared
    # the context still works
    wl = synth.custom(4, 8, 64, 256, 2, dtype="bf16", seed=1)
    buf = harness.MLPBuffers(wl, backward=False)
    buf.fwd()
    assert T.tpmlp_device_status(check=False) == T.OK
    assert bool(torch.isfinite(buf.Z).all())


def test_arch_is_sm103():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    assert torch.cuda.get_device_capability(0) == (10, 3)
