"""The no-allocation forward entry point (GPU).

Some callers cannot allocate device memory where they run the block (an
inference-engine plugin whose engine owns all device memory, a runtime that
forbids allocation after start-up).  tpmlp_mlp_fwd_noalloc keeps the
intermediate activation in a fixed array inside the library.  This test calls
it through the C-ABI twice in a row, on two different inputs, and checks each
result against tpmlp_mlp_fwd on the same inputs within the parity tolerance.
It is collected last, and passes alone in a fresh process as well as after the
other tests.
"""
import pytest

import gpu_util as U

pytestmark = pytest.mark.gpu


def test_noalloc_forward_matches_mlp_fwd_on_two_calls():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from megatron_tensor_mlp_gb300 import harness, synth
    from megatron_tensor_mlp_gb300 import tpmlp as T

    shapes = [(100, 3, 136, 544, 2), (64, 8, 256, 1024, 4)]  # ragged tiles; then full tiles
    for call, shape in enumerate(shapes):
        wl = synth.custom(*shape, dtype="bf16", sigma_w=0.05, sigma_bias=0.05, seed=40 + call)
        buf = harness.MLPBuffers(wl, backward=False)
        s, b, h, f, p = buf.dims()
        buf.fwd()
        Z = torch.full_like(buf.Z, float("nan"))
        T.tpmlp_mlp_fwd_noalloc(buf.X, buf.A_sh, buf.b1_sh, buf.B_sh, buf.b2, Z, s, b, h, f, p)
        T.tpmlp_device_status()
        U.assert_close(harness.to_host(Z), harness.to_host(buf.Z), "bf16", f"noalloc Z (call {call + 1})")


def test_noalloc_rejects_sizes_beyond_the_array():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from megatron_tensor_mlp_gb300 import tpmlp as T

    dummy = torch.zeros(1024, dtype=torch.bfloat16, device="cuda")
    out = torch.zeros(1024, dtype=torch.bfloat16, device="cuda")
    # 4096 tokens x ffn 8192 x 2 bytes = 64 MiB > 32 MiB
    st = T.tpmlp_mlp_fwd_noalloc(dummy, dummy, None, dummy, None, out, 4096, 1, 64, 8192, 2, check=False)
    assert st == T.ERR_SHAPE
    assert "at most" in T.last_error()
