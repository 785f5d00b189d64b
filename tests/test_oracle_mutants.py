"""Planted mistakes in the oracle must each fail at least one pin (CPU only).

Every mutant is a copy of the committed oracle source with one plausible
mistake (a dropped term, a wrong sign or index, a transposed operand), built
into a temporary library.  The committed oracle passes every pin; if a mutant
also passed them all, the pins would not be able to tell it apart.
"""
import os

import pytest

import oracle
import oracle_pins

MUTANTS = {
    "b1_sign": ("H[m * f + j] + (b1 ? b1[j] : 0.0)", "H[m * f + j] - (b1 ? b1[j] : 0.0)"),
    "b2_dropped": ("Z[m * h + n] += b2[n];", "Z[m * h + n] += 0.0 * b2[n];"),
    "gelu_grad_missing_term": ("return std_normal_cdf(z) + z * std_normal_pdf(z);",
                               "return std_normal_cdf(z);"),
    "cdf_sign": ("return 0.5 * erfc(-z *", "return 0.5 * erfc(z *"),
    "dgelu_at_Y_not_H": ("dH_work[m * f + j] *= act_grad(act, H[m * f + j]);",
                         "dH_work[m * f + j] *= act_grad(act, Y[m * f + j]);"),
    "matmul_nt_transposed": ("acc += a[k] * b[k];", "acc += a[k] * B[j + k * N];"),
    "matmul_tn_index": ("const double a = A[k * M + i];", "const double a = A[i * K + k];"),
    "shard_strided": ("s + (r * cols + i * cs + c) * elem_size", "s + (r * cols + c * p + i) * elem_size"),
    "qkv_identity": ("return t * h + g * d + e;", "return dst_col;"),
    "qkv_q_only": ("const int64_t g = blk / 3, t = blk % 3;", "const int64_t g = blk / 3, t = 0 * blk;"),
    "sampled_dX_transposed_A": ("for (int64_t n = 0; n < h; ++n) out[n] += dh * A[n * f + j];",
                                "for (int64_t n = 0; n < h; ++n) out[n] += dh * A[j * h + n];"),
    "sampled_dB_uses_H": ("const double y = act_fwd(act, hv);", "const double y = hv;"),
    "swiglu_b2_dropped": ("Z[m * h + n] = Z[m * h + n] + b2[n];", "Z[m * h + n] = Z[m * h + n] + 0.0 * b2[n];"),
    "silu_grad_missing_term": ("return s * (1.0 + x * (1.0 - s));", "return s;"),
    "swiglu_dHu_uses_grad": ("dHu[m * f + j] = dy * oracle_silu(g);", "dHu[m * f + j] = dy * oracle_silu_grad(g);"),
    "swiglu_pack_swapped": ("(j < 128 ? g : u)", "(j < 128 ? u : g)"),
    "swiglu_dX_missing_up": ("for (int64_t i = 0; i < M * h; ++i) dX[i] += tmp[i];",
                             "for (int64_t i = 0; i < M * h; ++i) dX[i] += 0.0 * tmp[i];"),
    "linear_bias_dropped": ("for (int64_t n = 0; n < N; ++n) Y[m * N + n] += b[n];",
                            "for (int64_t n = 0; n < N; ++n) Y[m * N + n] += 0.0 * b[n];"),
    "linear_dX_wrong_operand": ("matmul_nt(M, N, K, dY, W, dX);  /* dX = dY W^T  [M,K] */",
                                "matmul_nn(M, N, K, dY, W, dX);  /* dX = dY W^T  [M,K] */"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(oracle.SRC).read()
    assert src.count(old) == 1, f"mutation site for {name} not unique/found"
    mpath = os.path.join(tmp_path, f"mut_{name}.c")
    with open(mpath, "w") as fh:
        fh.write(src.replace(old, new))
    so = oracle.compile_source(mpath, os.path.join(tmp_path, f"libmut_{name}.so"))
    bad = oracle_pins.failing_pins(oracle.Oracle(so))
    assert bad, f"mutant {name} passed every pin"
