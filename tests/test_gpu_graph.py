"""The block's entry points inside a CUDA graph (GPU).

Calls only enqueue kernels on the caller's stream (no allocation, no
synchronisation), so a forward + backward step captured once replays with
results identical to eager calls.  Per-device set-up (kernel attributes, the
pair-kernel occupancy query, the backward's second stream and its two events) happens on
the first eager call, before capture.  The second shape is large enough for the backward to
fork its bias-gradient column sums onto the second stream beside the dX GEMM, so the graph
holds that fork and join too.
"""
import pytest

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("shape", [(64, 8, 512, 2048, 4), (512, 4, 5120, 20480, 4)],
                         ids=["sums-in-line", "sums-beside-dX"])
def test_fwd_bwd_step_replays_in_a_cuda_graph(shape):
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from megatron_tensor_mlp_gb300 import harness, synth
    from megatron_tensor_mlp_gb300 import tpmlp as T

    wl = synth.custom(*shape, dtype="bf16", sigma_w=0.02, seed=5)
    buf = harness.MLPBuffers(wl, backward=True)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):  # warm-up on the capture stream
        buf.fwd(stream=side)
        buf.bwd(stream=side)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    eager = [t.clone() for t in (buf.Z, buf.dX, buf.dA_sh, buf.dB_sh, buf.db1_sh, buf.db2)]
    outs = (buf.Z, buf.dX, buf.dA_sh, buf.dB_sh, buf.db1_sh, buf.db2)
    for t in outs:
        t.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        buf.fwd()
        buf.bwd()
    for t in outs:
        t.zero_()
    for _ in range(2):
        g.replay()
    torch.cuda.synchronize()
    T.tpmlp_device_status()
    for a, b in zip(eager, outs):
        assert torch.equal(a, b)
