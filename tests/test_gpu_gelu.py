"""The epilogue's GeLU and GeLU' against CUDA's erf on every bf16 value in [-12, 12] (GPU).

The tensor-core epilogues evaluate Phi(x) with Hastings' rational approximation of
erfc (Abramowitz & Stegun 7.1.26, |error| <= 1.5e-7).  Driven through the C-ABI
with identity weights, the column layer returns H = x exactly and Y = GeLU(x),
and the row backward with dZ = 1 returns GeLU'(x); both are compared with the
same functions computed from torch.erf / torch.exp on the GPU, allowing half a
bf16 unit in the last place of the result plus 1e-6 * max(1, |x|).
"""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu


def _all_bf16_in_range(lo, hi):
    import torch
    bits = torch.arange(0, 1 << 16, dtype=torch.int32).to(torch.int16).view(torch.bfloat16).float()
    x = bits[torch.isfinite(bits) & (bits >= lo) & (bits <= hi)]
    return torch.unique(x)


def _half_ulp_bf16(v):
    import torch
    a = v.abs().clamp_min(2.0 ** -126)
    e = torch.floor(torch.log2(a))
    return 2.0 ** (e - 8)  # bf16 has 8 significant bits: ulp = 2^(e-7), half = 2^(e-8)


def test_gelu_and_grad_match_cuda_erf():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from megatron_tensor_mlp_gb300 import tpmlp as T

    x = _all_bf16_in_range(-12.0, 12.0)
    h = 128
    n = ((x.numel() + h - 1) // h) * h
    xs = torch.zeros(n)
    xs[: x.numel()] = x
    M = n // h
    X = xs.view(M, h).to(torch.bfloat16).cuda()
    I = torch.eye(h, dtype=torch.bfloat16, device="cuda")
    Y = torch.empty((1, M, h), dtype=torch.bfloat16, device="cuda")
    H = torch.empty((1, M, h), dtype=torch.bfloat16, device="cuda")
    T.tpmlp_column_fwd(X, I, None, Y, H, M, 1, h, h, 1)
    # GeLU'(H) through the row backward: dZ = 1, B = I  ->  dY = 1, dH = GeLU'(H)
    dZ = torch.ones((M, h), dtype=torch.bfloat16, device="cuda")
    dH = torch.empty((1, M, h), dtype=torch.bfloat16, device="cuda")
    dB = torch.empty((1, h, h), dtype=torch.float32, device="cuda")
    T.tpmlp_row_bwd(Y, I, dZ, H, dH, dB, None, M, 1, h, h, 1, act=T.ACT_GELU_ERF)
    T.tpmlp_device_status()
    xf = X.float().view(-1)
    assert torch.equal(H.view(-1).float(), xf)  # identity weights: H is x exactly
    cdf = 0.5 * (1.0 + torch.erf(xf / np.sqrt(2.0)))
    ref_y = xf * cdf
    ref_g = cdf + xf * torch.exp(-0.5 * xf * xf) / np.sqrt(2.0 * np.pi)
    for got, ref, name in ((Y.view(-1).float(), ref_y, "GeLU"), (dH.view(-1).float(), ref_g, "GeLU'")):
        err = (got - ref).abs()
        bound = _half_ulp_bf16(ref) + 1e-6 * xf.abs().clamp_min(1.0)
        bad = err > bound
        assert not bool(bad.any()), f"{name}: {int(bad.sum())} values off, worst at x={float(xf[err.argmax()])}"
