"""Layout kernels against the oracle's index maps, bit for bit (GPU)."""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def T():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from megatron_tensor_mlp_gb300 import tpmlp
    return tpmlp


def _dev(a):
    import torch
    if a.size == 0:  # keep a non-NULL pointer for empty inputs
        return torch.zeros(16, dtype=torch.int16 if a.dtype == np.uint16 else torch.int32, device="cuda")
    return torch.from_numpy(a.view(np.int16) if a.dtype == np.uint16 else a.view(np.int32)).cuda()


def _host(t, dtype):
    return t.cpu().numpy().view(dtype)


@pytest.mark.parametrize("rows,cols,p,dt", [
    (5, 64, 2, 0), (7, 96, 3, 0), (16, 256, 8, 0), (3, 8, 1, 0), (1, 1024, 4, 0),
    (5, 64, 4, 1), (9, 48, 3, 1), (0, 64, 2, 0),
    (1024, 4096, 8, 0),  # several thousand 16-byte units per shard row block
])
def test_shard_columns_bitexact(T, orc, rows, cols, p, dt):
    import torch
    rng = np.random.default_rng(rows * 1000 + cols + p)
    npdt = np.uint16 if dt == T.BF16 else np.uint32
    W = rng.integers(0, np.iinfo(npdt).max, size=(rows, cols), dtype=npdt, endpoint=True)
    ref = orc.shard_columns(W, p)
    src = _dev(W)
    dst = torch.full((max(16, p * rows * (cols // p)),), -1, dtype=src.dtype, device="cuda")
    T.tpmlp_shard_columns(src, dst, rows, cols, p, dt)
    back = torch.full_like(src, -1)
    T.tpmlp_unshard_columns(dst, back, rows, cols, p, dt)
    T.tpmlp_device_status()
    n = ref.size
    assert np.array_equal(_host(dst, npdt)[:n].reshape(ref.shape), ref)
    assert np.array_equal(_host(back, npdt)[:W.size].reshape(W.shape), W)
    if n == 0:  # nothing may have been written
        assert np.all(_host(dst, npdt) == np.iinfo(npdt).max)


@pytest.mark.parametrize("rows,h,n,p,dt", [
    (4, 64, 8, 2, 0),     # d = 8 -> 16-byte units
    (3, 96, 12, 4, 0),    # d = 8
    (2, 24, 6, 3, 0),     # d = 4 -> element path
    (5, 48, 4, 4, 1),     # fp32, d = 12 -> 16-byte units
    (2, 20, 5, 5, 1),     # fp32, d = 4
    (64, 1024, 16, 8, 0),
])
def test_qkv_interleave_bitexact(T, orc, rows, h, n, p, dt):
    import torch
    rng = np.random.default_rng(h * 7 + n)
    npdt = np.uint16 if dt == T.BF16 else np.uint32
    W = rng.integers(0, np.iinfo(npdt).max, size=(rows, 3 * h), dtype=npdt, endpoint=True)
    ref = orc.qkv_interleave(W, h, n)
    src = _dev(W)
    dst = torch.full_like(src, -1)
    T.tpmlp_qkv_interleave(src, dst, rows, h, n, p, dt, inverse=0)
    inv = torch.full_like(src, -1)
    T.tpmlp_qkv_interleave(dst, inv, rows, h, n, p, dt, inverse=1)
    T.tpmlp_device_status()
    assert np.array_equal(_host(dst, npdt), ref)
    assert np.array_equal(_host(inv, npdt), W)
