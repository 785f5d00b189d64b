"""The no-allocation forward entry point (GPU).

Some callers cannot allocate device memory where they run the block: an
inference-engine plugin whose engine owns all device memory, or a runtime that
forbids allocation after start-up because an allocation can synchronise the
device.  tpmlp_mlp_fwd_noalloc keeps the intermediate activation Y in a fixed
array inside the library instead of a caller workspace.

These tests call it through the C-ABI and check its Z element by element
against the fp64 oracle on the same seeded inputs (and against tpmlp_mlp_fwd):
two calls in a row on different inputs, an fp32 call, and calls exactly at
the array's size limit, where one more token must be refused.  Around a call
they check that no device memory was allocated.  The file is collected last
and passes alone in a fresh process as well as after the other tests.
"""
import pytest

import gpu_util as U

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def env():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from megatron_tensor_mlp_gb300 import harness, synth
    from megatron_tensor_mlp_gb300 import tpmlp as T
    return harness, synth, T


def _check_call(env, orc, wl, check_no_alloc=False):
    """One no-allocation forward on the workload's seeded inputs: Z against the oracle's and
    against tpmlp_mlp_fwd's on the same inputs."""
    import torch
    harness, synth, T = env
    dt = "bf16" if wl.dtype == "bf16" else "f32"
    buf = harness.MLPBuffers(wl, backward=False)
    s, b, h, f, p = buf.dims()
    buf.fwd()
    Z = torch.full_like(buf.Z, float("nan"))
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    alloc0 = torch.cuda.memory_allocated()
    T.tpmlp_mlp_fwd_noalloc(buf.X, buf.A_sh, buf.b1_sh, buf.B_sh, buf.b2, Z, s, b, h, f, p, dt=buf.dt)
    torch.cuda.synchronize()
    if check_no_alloc:
        assert torch.cuda.mem_get_info()[0] == free0, "device memory was allocated during the call"
        assert torch.cuda.memory_allocated() == alloc0
    T.tpmlp_device_status()
    x = U.host_inputs_f64(buf)
    _, _, Z_ref = orc.mlp_fwd(x["X"], x["A"], x["b1"], x["B"], x["b2"])
    got = harness.to_host(Z)
    U.assert_close(got, Z_ref, dt, f"noalloc Z vs oracle ({wl.name})")
    U.assert_close(got, harness.to_host(buf.Z), dt, f"noalloc Z vs tpmlp_mlp_fwd ({wl.name})")
    return got


def test_two_calls_in_a_row_match_the_oracle(env, orc):
    """Two calls in a row share the array: the second (other inputs, same shape) must not see
    anything of the first, and it allocates no device memory."""
    _, synth, _ = env
    shape = (100, 3, 136, 544, 2)  # ragged in every GEMM dimension
    outs = []
    for call in range(2):
        wl = synth.custom(*shape, dtype="bf16", sigma_w=0.05, sigma_bias=0.05, seed=40 + call, backward=False)
        outs.append(_check_call(env, orc, wl, check_no_alloc=(call == 1)))
    assert not (outs[0] == outs[1]).all()


def test_fp32_call_matches_the_oracle(env, orc):
    """fp32 inputs: Y takes 4 bytes per element in the array; s*b*ffn*4 is exactly the array's
    size (2048 tokens x 4096 = 32 MiB)."""
    from megatron_tensor_mlp_gb300 import tpmlp as T
    _, synth, _ = env
    s, b, h, f, p = 512, 4, 64, 4096, 4
    assert s * b * f * 4 == T.NOALLOC_SCRATCH_BYTES
    wl = synth.custom(s, b, h, f, p, dtype="f32", sigma_w=0.05, sigma_bias=0.05, seed=44, backward=False)
    _check_call(env, orc, wl)


def test_bf16_call_exactly_at_the_limit(env, orc):
    """s*b*ffn*2 equal to the array's size (4096 tokens x ffn 4096) runs and matches the oracle;
    one token more is refused with TPMLP_ERR_SHAPE before anything is enqueued."""
    import torch
    harness, synth, T = env
    s, b, h, f, p = 1024, 4, 64, 4096, 4
    assert s * b * f * 2 == T.NOALLOC_SCRATCH_BYTES
    wl = synth.custom(s, b, h, f, p, dtype="bf16", sigma_w=0.05, sigma_bias=0.05, seed=45, backward=False)
    _check_call(env, orc, wl, check_no_alloc=True)
    M1 = s * b + 1
    X = torch.zeros((M1, h), dtype=torch.bfloat16, device="cuda")
    A = torch.zeros((p, h, f // p), dtype=torch.bfloat16, device="cuda")
    B = torch.zeros((p, f // p, h), dtype=torch.bfloat16, device="cuda")
    Z = torch.zeros((M1, h), dtype=torch.bfloat16, device="cuda")
    st = T.tpmlp_mlp_fwd_noalloc(X, A, None, B, None, Z, M1, 1, h, f, p, check=False)
    assert st == T.ERR_SHAPE
    assert "at most" in T.last_error()


def test_noalloc_rejects_sizes_beyond_the_array(env):
    import torch
    _, _, T = env
    dummy = torch.zeros(1024, dtype=torch.bfloat16, device="cuda")
    out = torch.zeros(1024, dtype=torch.bfloat16, device="cuda")
    # 4096 tokens x ffn 8192 x 2 bytes = 64 MiB > 32 MiB
    st = T.tpmlp_mlp_fwd_noalloc(dummy, dummy, None, dummy, None, out, 4096, 1, 64, 8192, 2, check=False)
    assert st == T.ERR_SHAPE
    assert "at most" in T.last_error()
