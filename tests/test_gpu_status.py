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


def test_launch_count_counts_enqueued_kernels():
    """The host-side launch counter: one per kernel of the forward (column and row GEMM) and of
    the backward (dH, dB, dA and dX GEMMs and the db1 and db2 column sums) at a one-wave shape;
    nothing for a call rejected by validation."""
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from megatron_tensor_mlp_gb300 import harness, synth, tpmlp as T
    wl = synth.custom(4, 8, 64, 256, 2, dtype="bf16", seed=2)
    buf = harness.MLPBuffers(wl, backward=True)
    n0 = T.tpmlp_launch_count()
    buf.fwd()
    n1 = T.tpmlp_launch_count()
    buf.bwd()
    n2 = T.tpmlp_launch_count()
    torch.cuda.synchronize()
    T.tpmlp_device_status()
    assert n1 - n0 == 2
    assert n2 - n1 == 6
    st = T.tpmlp_mlp_fwd(buf.X, buf.A_sh, None, buf.B_sh, None, None, buf.Y, None, 4, 8, 64, 256, 2, check=False)
    assert st == T.ERR_NULL
    assert T.tpmlp_launch_count() == n2
