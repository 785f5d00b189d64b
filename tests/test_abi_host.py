"""The C-ABI library on the host: it loads, exports every declared symbol, and
rejects bad arguments before touching the device (CPU only)."""
import ctypes
import subprocess
import sys

import pytest

from megatron_tensor_mlp_gb300 import build as B

# build once here (nvcc cross-compiles without a GPU)
B.build()
from megatron_tensor_mlp_gb300 import tpmlp as T  # noqa: E402

FAKE = 0x7F0000000000  # a 16-byte aligned address that is never dereferenced


def test_exports_every_declared_symbol():
    names = T.header_functions()
    assert "tpmlp_mlp_fwd" in names and "tpmlp_qkv_interleave" in names
    lib = ctypes.CDLL(T.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), n
    # and the dynamic symbol table agrees
    out = subprocess.run(["nm", "-D", "--defined-only", T.LIB_PATH], capture_output=True, text=True).stdout
    for n in names:
        assert f" T {n}\n" in out, n


def test_version_and_strings():
    assert T.tpmlp_version() >= 200
    for code, name in T.STATUS.items():
        assert T.tpmlp_status_string(code) == name


def _fwd(**kw):
    args = dict(X=FAKE, A_sh=FAKE + 0x100000, b1_sh=None, B_sh=FAKE + 0x200000, b2=None, Z=FAKE + 0x300000,
                Y_ws=FAKE + 0x400000, H_sh=None, s=4, b=2, h=64, ffn=256, p=2, dt=T.BF16, stream=0)
    args.update(kw)
    return T.tpmlp_mlp_fwd(**args, check=False)


def test_validation_order_and_codes():
    assert _fwd(X=None) == T.ERR_NULL
    assert _fwd(Y_ws=None) == T.ERR_NULL
    assert _fwd(h=0) == T.ERR_SHAPE
    assert _fwd(s=-1) == T.ERR_SHAPE
    assert _fwd(p=0) == T.ERR_SHAPE
    assert _fwd(s=1 << 20, b=1 << 12) == T.ERR_SHAPE  # s*b >= 2^31
    assert _fwd(s=1 << 20, b=1 << 10, h=1 << 20, ffn=1 << 20, p=1) == T.ERR_SHAPE  # tensors beyond 2^40 bytes
    assert _fwd(ffn=250, p=4) == T.ERR_DIVISIBILITY   # ffn % p
    assert _fwd(h=66, p=4, ffn=256) == T.ERR_DIVISIBILITY  # the block also needs h % p
    assert _fwd(dt=7) == T.ERR_DTYPE
    assert _fwd(X=FAKE + 8) == T.ERR_ALIGNMENT        # pointer not 16-byte aligned
    assert _fwd(h=60, ffn=240, p=2) == T.ERR_ALIGNMENT  # h*2 bytes not a multiple of 16
    assert _fwd(ffn=252, p=3, h=96) == T.ERR_ALIGNMENT  # ffn/p = 84 bf16 = 168 B
    # Z overlapping X
    assert _fwd(Z=FAKE + 64) == T.ERR_ALIAS
    # Y_ws overlapping Z
    assert _fwd(Y_ws=FAKE + 0x300000 + 16) == T.ERR_ALIAS


def test_valid_arguments_reach_the_device_check():
    st = _fwd()
    # with a GPU this would launch; here the CUDA runtime has no device
    assert st in (T.ERR_CUDA, T.ERR_ARCH) or st == T.OK


def test_bwd_and_layout_validation():
    st = T.tpmlp_mlp_bwd(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, FAKE, FAKE, None, None, FAKE,
                         4, 2, 64, 256, 2, check=False)
    assert st == T.ERR_NULL
    st = T.tpmlp_mlp_bwd(*(FAKE + i * 0x100000 for i in range(9)), None, None, FAKE + 9 * 0x100000,
                         4, 2, 64, 256, 2, dt=T.F32, grad_dt=T.BF16, check=False)
    assert st == T.ERR_DTYPE
    assert T.tpmlp_shard_columns(FAKE, FAKE + 0x100000, 4, 30, 4, check=False) == T.ERR_DIVISIBILITY
    assert T.tpmlp_shard_columns(FAKE, FAKE + 0x100000, 4, 24, 4, check=False) == T.ERR_ALIGNMENT  # 6 bf16
    assert T.tpmlp_shard_columns(FAKE, FAKE + 16, 4, 64, 4, check=False) == T.ERR_ALIAS
    assert T.tpmlp_qkv_interleave(FAKE, FAKE + 0x100000, 4, 64, 6, 2, check=False) == T.ERR_DIVISIBILITY
    assert T.tpmlp_qkv_interleave(FAKE, FAKE + 0x100000, 4, 64, 8, 3, check=False) == T.ERR_DIVISIBILITY
    assert T.tpmlp_debug_wait_timeout(0, check=False) == T.ERR_SHAPE
    assert T.tpmlp_shard_columns(FAKE, FAKE + 0x100000, 1 << 30, 1 << 20, 4, check=False) == T.ERR_SHAPE
    assert T.tpmlp_qkv_interleave(FAKE, FAKE + 0x100000, 1 << 30, 1 << 20, 8, 2, check=False) == T.ERR_SHAPE
    assert T.tpmlp_swiglu_pack(FAKE, FAKE + 0x100000, FAKE + 0x200000, 1 << 30, 1 << 20, 4, check=False) \
        == T.ERR_SHAPE


def test_gemm_mode_control():
    assert T.tpmlp_set_gemm_mode(6, check=False) == T.ERR_SHAPE
    assert T.tpmlp_set_gemm_mode(-1, check=False) == T.ERR_SHAPE
    for m in (1, 2, 3, 4, 5, 0):
        assert T.tpmlp_set_gemm_mode(m) == T.OK
        assert T.tpmlp_get_gemm_mode() == m


def test_k_chunk_control():
    assert T.tpmlp_set_k_chunk(-1, check=False) == T.ERR_SHAPE
    assert T.tpmlp_set_k_chunk((1 << 24) + 1, check=False) == T.ERR_SHAPE
    assert T.tpmlp_get_k_chunk() == 4096
    for c in (1, 7, 4096):
        assert T.tpmlp_set_k_chunk(c) == T.OK
        assert T.tpmlp_get_k_chunk() == c
    assert T.tpmlp_set_k_chunk(0) == T.OK
    assert T.tpmlp_get_k_chunk() == 4096


def test_qkv_src_col_matches_oracle(orc):
    for (h, n) in [(12, 4), (64, 8), (24, 3), (8, 8), (16, 1)]:
        for c in range(3 * h):
            assert T.tpmlp_qkv_src_col(c, h, n) == orc.qkv_src_col(c, h, n)
    assert T.tpmlp_qkv_src_col(-1, 12, 4) == -1
    assert T.tpmlp_qkv_src_col(36, 12, 4) == -1
    assert T.tpmlp_qkv_src_col(0, 12, 5) == -1


def test_binding_fails_loudly_without_library(tmp_path):
    # a copy of the binding next to no library must refuse to import
    src = open(T.__file__).read()
    pkg = tmp_path / "fakepkg"
    pkg.mkdir()
    (pkg / "__init__.py").write_text("")
    (pkg / "tpmlp.py").write_text(src)
    r = subprocess.run([sys.executable, "-c", "import fakepkg.tpmlp"], cwd=tmp_path, capture_output=True, text=True)
    assert r.returncode != 0 and "is not built" in r.stderr


def test_side_stream_registration_rules():
    """All three handles or none: a partial registration is refused before any CUDA call, and
    clearing needs no device."""
    assert T.tpmlp_set_side_stream(None, None, None) == T.OK
    assert T.tpmlp_set_side_stream(0x1000, None, None, check=False) == T.ERR_NULL
    assert T.tpmlp_set_side_stream(None, 0x1000, 0x2000, check=False) == T.ERR_NULL


def test_tp_entry_points_validate_on_the_host():
    """The rank-local entry points and the finish step refuse bad arguments before any CUDA call."""
    assert T.tpmlp_sum_finish(None, None, 0x1000, 4, 8, check=False) == T.ERR_NULL
    assert T.tpmlp_sum_finish(0x1000, None, 0x2000, 4, 12, check=False) == T.ERR_ALIGNMENT  # 12 bf16 = 24 B
    assert T.tpmlp_sum_finish(0x1000, None, 0x1008, 4, 8, check=False) == T.ERR_ALIGNMENT
    assert T.tpmlp_sum_finish(0x1000, None, 0x1000, 4, 8, check=False) == T.ERR_ALIAS
    assert T.tpmlp_sum_finish(0x1000, None, 0x2000, -1, 8, check=False) == T.ERR_SHAPE
    p16 = 0x10000
    assert T.tpmlp_mlp_fwd_partial(p16, p16, None, p16, None, p16, None, 8, 2, 64, 256, 2, check=False) == T.ERR_NULL
    assert T.tpmlp_mlp_fwd_partial(p16, p16, None, p16, p16 * 2, p16 * 3, None, 8, 2, 64, 250, 2,
                                   check=False) == T.ERR_ALIGNMENT
    assert T.tpmlp_mlp_bwd_partial(p16, p16, p16, p16, p16, p16, None, p16, p16, None, None, p16, 8, 2, 64, 256, 3,
                                   check=False) == T.ERR_NULL
    assert T.tpmlp_mlp_bwd_partial(p16, p16, p16, p16, p16, p16, p16 * 2, p16 * 3, p16 * 4, None, None, p16 * 5,
                                   8, 2, 64, 256, 3, check=False) == T.ERR_DIVISIBILITY


def test_rejected_calls_launch_nothing():
    n0 = T.tpmlp_launch_count()
    assert _fwd(X=None) == T.ERR_NULL
    assert _fwd(ffn=250, p=4) == T.ERR_DIVISIBILITY
    assert T.tpmlp_sum_finish(None, None, 0x1000, 4, 8, check=False) == T.ERR_NULL
    assert T.tpmlp_launch_count() == n0
