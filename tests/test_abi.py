"""The C ABI library loads without a GPU, exports every declared symbol and
rejects bad arguments on the host before any launch."""
import ctypes
import os
import re
import subprocess

import pytest

import io_aware_exact_08_gb300 as fa

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_symbols():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names |= set(re.findall(r"\b(fa_\w+)\s*\(", text))
    return names


def test_library_builds_and_loads():
    from io_aware_exact_08_gb300 import build
    path = build.build()
    assert os.path.exists(path)
    lib = fa.load_library()
    assert lib is not None


def test_every_declared_symbol_is_exported():
    declared = _declared_symbols()
    assert {"fa_fwd", "fa_bwd", "fa_bwd_workspace_size", "fa_dropout_mask",
            "fa_check_device_status", "fa_status_string"} <= declared
    lib = ctypes.CDLL(fa.library_path())
    for name in declared:
        assert hasattr(lib, name), name
    out = subprocess.run(["nm", "-D", "--defined-only", fa.library_path()], capture_output=True, text=True)
    exported = set(re.findall(r"\bT (fa_\w+)", out.stdout))
    assert declared <= exported
    assert set(fa.EXPORTED) <= exported


def test_workspace_is_linear_in_n():
    # O(B*H*N*d): 1 KB of row statistics per 128-row tile of each head (-LSE
    # and -rowsum(dO o O) of its rows) plus the fp32 dQ accumulator, each
    # rounded to 256 bytes, plus 256 bytes for the work counter
    for B, H, N, d in [(1, 1, 128, 64), (2, 16, 8192, 128), (32, 16, 512, 64), (1, 1, 1, 64), (1, 2, 1000, 256)]:
        rows = B * H * N
        tiles = B * H * ((N + 127) // 128)
        r256 = lambda x: (x + 255) // 256 * 256
        assert fa.fa_bwd_workspace_size(B, H, N, d) == r256(1024 * tiles) + r256(4 * rows * d) + 256
    assert fa.fa_bwd_workspace_size(1, 1, 16, 96) == 0
    assert fa.fa_bwd_workspace_size(0, 1, 16, 64) == 0
    w1 = fa.fa_bwd_workspace_size(1, 1, 4096, 128) - 256
    w2 = fa.fa_bwd_workspace_size(1, 1, 8192, 128) - 256
    assert w2 == 2 * w1


FAKE = 1 << 20  # a 16-byte aligned non-null value; never dereferenced on these paths


@pytest.mark.parametrize("kw,expect", [
    (dict(d=96), -2), (dict(d=32), -2), (dict(B=0), -1), (dict(H=-1), -1), (dict(N=-5), -1),
    (dict(dropout_p=1.0), -1), (dict(dropout_p=-0.1), -1), (dict(dtype=7), -2),
    (dict(q=None), -1), (dict(lse=None), -1), (dict(o=FAKE + 8), -1), (dict(scale=float("inf")), -1),
])
def test_forward_argument_errors(kw, expect):
    args = dict(q=FAKE, k=FAKE, v=FAKE, o=FAKE, lse=FAKE, B=1, H=1, N=16, d=64, scale=0.125, causal=0,
                block_mask=None, dropout_p=0.0, seed=0, dtype=fa.FA_BF16, kv_len=None, stream=None)
    args.update(kw)
    assert fa.fa_fwd(**args) == expect


@pytest.mark.parametrize("kw,expect", [
    (dict(dtype=3), -2), (dict(d=512), -2), (dict(d=256, B=0), -1), (dict(d=256, o=FAKE + 8), -1),
    (dict(d=256, dropout_p=1.5), -1), (dict(d=256, q=None), -1),
])
def test_forward_argument_errors_fp16_and_d256(kw, expect):
    """fp16 inputs and head dim 256 go through the same host-side checks."""
    args = dict(q=FAKE, k=FAKE, v=FAKE, o=FAKE, lse=FAKE, B=1, H=1, N=16, d=64, scale=0.125, causal=0,
                block_mask=None, dropout_p=0.0, seed=0, dtype=fa.FA_FP16, kv_len=None, stream=None)
    args.update(kw)
    assert fa.fa_fwd(**args) == expect


def test_dtype_codes_match_the_header():
    torch = pytest.importorskip("torch")
    assert (fa.FA_BF16, fa.FA_FP32, fa.FA_FP16) == (0, 1, 2)
    header = open(os.path.join(os.path.dirname(__file__), "..", "include", "fa.h")).read()
    assert "FA_BF16 = 0, FA_FP32 = 1, FA_FP16 = 2" in header
    assert fa._dtype_code(torch.empty(1, dtype=torch.float16)) == fa.FA_FP16
    assert fa._dtype_code(torch.empty(1, dtype=torch.bfloat16)) == fa.FA_BF16
    with pytest.raises(TypeError):
        fa._dtype_code(torch.empty(1, dtype=torch.float64))


def test_zero_length_is_a_noop():
    assert fa.fa_fwd(None, None, None, None, None, 1, 1, 0, 64, 0.1, 0, None, 0.0, 0, fa.FA_BF16, None, None) == 0


@pytest.mark.parametrize("kw,expect", [
    (dict(workspace=None), -4), (dict(workspace_bytes=16), -4), (dict(workspace=FAKE + 16), -4),
    (dict(dq=None), -1), (dict(d=80), -2), (dict(dropout_p=2.0), -1),
])
def test_backward_argument_errors(kw, expect):
    args = dict(q=FAKE, k=FAKE, v=FAKE, o=FAKE, lse=FAKE, dO=FAKE, dq=FAKE, dk=FAKE, dv=FAKE, B=1, H=1, N=16,
                d=64, scale=0.125, causal=0, block_mask=None, dropout_p=0.0, seed=0, dtype=fa.FA_BF16,
                kv_len=None, workspace=FAKE, workspace_bytes=1 << 20, stream=None)
    args.update(kw)
    assert fa.fa_bwd(**args) == expect


@pytest.mark.parametrize("dtype", [fa.FA_BF16, fa.FA_FP16])
@pytest.mark.parametrize("kw", [
    dict(scale=0.0), dict(scale=-0.125),
    dict(N=1024 * 128 + 1, block_mask=FAKE),        # 1025 key tiles per row: over the forward's list
])
def test_forward_refuses_what_the_tensor_cores_do_not_take(kw, dtype):
    """16-bit problems outside the tensor-core kernels are refused on the
    host (FA_ERR_UNSUPPORTED), not run on the CUDA-core kernels."""
    args = dict(q=FAKE, k=FAKE, v=FAKE, o=FAKE, lse=FAKE, B=1, H=1, N=16, d=64, scale=0.125, causal=0,
                block_mask=None, dropout_p=0.0, seed=0, dtype=dtype, kv_len=None, stream=None)
    args.update(kw)
    assert fa.fa_fwd(**args) == -2
    split = dict(args, n_splits=2, workspace=FAKE, workspace_bytes=1 << 40)
    assert fa.fa_fwd_splitkv(**split) == -2


@pytest.mark.parametrize("kw", [
    dict(scale=0.0), dict(scale=-1.0),
    dict(d=128, N=256 * 128 + 1, block_mask=FAKE),  # 257 query tiles per key tile at d = 128
    dict(d=256, N=256 * 128 + 1, block_mask=FAKE),
    dict(d=64, N=1024 * 128 + 1, block_mask=FAKE),
])
def test_backward_refuses_what_the_tensor_cores_do_not_take(kw):
    args = dict(q=FAKE, k=FAKE, v=FAKE, o=FAKE, lse=FAKE, dO=FAKE, dq=FAKE, dk=FAKE, dv=FAKE, B=1, H=1, N=16,
                d=64, scale=0.125, causal=0, block_mask=None, dropout_p=0.0, seed=0, dtype=fa.FA_BF16,
                kv_len=None, workspace=FAKE, workspace_bytes=1 << 40, stream=None)
    args.update(kw)
    assert fa.fa_bwd(**args) == -2


def test_status_strings():
    for code in (0, -1, -2, -3, -4, -5):
        s = fa.fa_status_string(code)
        assert s.startswith("FA_")
    assert "unknown" in fa.fa_status_string(12345)


def test_kernel_path_switch_roundtrips():
    old = fa.fa_set_kernel_path(1)
    assert fa.fa_set_kernel_path(old) == 1


def test_splitkv_workspace_size():
    # n_splits partial O (fp32, d per row) then partial LSE, each rounded to 256 bytes
    r256 = lambda x: (x + 255) // 256 * 256
    for B, H, N, d, s in [(1, 4, 16384, 128, 4), (2, 3, 300, 64, 3), (1, 1, 1, 64, 1)]:
        rows = B * H * N
        assert fa.fa_fwd_splitkv_workspace_size(B, H, N, d, s) == r256(4 * s * rows * d) + r256(4 * s * rows)
    assert fa.fa_fwd_splitkv_workspace_size(1, 1, 128, 64, 0) == 0
    assert fa.fa_fwd_splitkv_workspace_size(1, 1, 128, 64, 65) == 0
    assert fa.fa_fwd_splitkv_workspace_size(1, 1, 128, 96, 2) == 0


@pytest.mark.parametrize("kw,expect", [
    (dict(n_splits=0), -1), (dict(n_splits=65), -1), (dict(workspace=None), -4), (dict(workspace_bytes=16), -4),
    (dict(workspace=FAKE + 16), -4), (dict(d=96), -2), (dict(o=None), -1),
])
def test_splitkv_argument_errors(kw, expect):
    args = dict(q=FAKE, k=FAKE, v=FAKE, o=FAKE, lse=FAKE, B=1, H=1, N=16, d=64, scale=0.125, causal=0,
                block_mask=None, dropout_p=0.0, seed=0, dtype=fa.FA_BF16, kv_len=None, n_splits=2,
                workspace=FAKE, workspace_bytes=1 << 20, stream=None)
    args.update(kw)
    assert fa.fa_fwd_splitkv(**args) == expect


@pytest.mark.parametrize("kw,expect", [
    (dict(d=64), -2), (dict(d=256), -2), (dict(N=100), -2), (dict(scale=0.0), -2), (dict(q=None), -1),
    (dict(descale_v=None), -1), (dict(vt=FAKE + 8), -1), (dict(B=0), -1), (dict(N=1024 * 128 + 16, block_mask=FAKE), -2),
])
def test_fp8_forward_argument_errors(kw, expect):
    args = dict(q=FAKE, k=FAKE, vt=FAKE, descale_q=FAKE, descale_k=FAKE, descale_v=FAKE, o=FAKE, lse=FAKE, B=1, H=1,
                N=16, d=128, scale=0.125, causal=0, block_mask=None, kv_len=None, stream=None)
    args.update(kw)
    assert fa.fa_fwd_fp8(**args) == expect
