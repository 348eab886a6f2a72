"""GPU vs fp64 oracle, element by element, on small seeded cases that span
several 128-row tiles and a ragged tail, with every mask and dropout, for
both the tensor-core (bf16, fp16) and the CUDA-core (fp32, and bf16 or fp16
on request) kernels. Tolerances: see parity_utils.TOL."""
import pytest
import torch

import io_aware_exact_08_gb300 as fa
from parity_utils import compare, gpu_fwd_bwd, oracle_fwd_bwd
from workloads import Workload, make_inputs, random_block_mask

pytestmark = pytest.mark.gpu


def _case(N, d, dtype, causal=False, pad=False, blocky=False, p=0.0, B=2, H=3, seed=7):
    w = Workload("case", 0, B=B, H=H, N=N, d=d, dtype=dtype, causal=causal,
                 kv_len_range=((max(1, N // 2), N) if pad else None), dropout_p=p)
    inp = make_inputs(w, seed=seed)
    if blocky:
        nb = (N + 127) // 128
        inp["block_mask"] = random_block_mask(nb, 0.5, seed + 1)
    return inp


CASES = [
    # N, d, causal, pad, blocky, dropout
    (1, 64, False, False, False, 0.0),
    (17, 64, True, False, False, 0.0),
    (127, 128, False, False, False, 0.0),
    (128, 64, True, False, False, 0.0),
    (129, 128, True, False, False, 0.0),
    (255, 64, False, True, False, 0.0),
    (300, 128, True, True, False, 0.0),
    (384, 64, False, False, True, 0.0),
    (520, 128, True, False, True, 0.0),
    (256, 64, False, False, False, 0.1),
    (333, 128, True, True, False, 0.2),
    (640, 64, False, True, True, 0.1),
    (1000, 128, False, False, False, 0.0),
    (1024, 64, True, False, False, 0.0),
]


def _ids(c):
    N, d, causal, pad, blocky, p = c
    return f"N{N}-d{d}" + ("-causal" if causal else "") + ("-pad" if pad else "") + \
        ("-block" if blocky else "") + (f"-drop{p}" if p else "")


@pytest.mark.parametrize("case", CASES, ids=_ids)
@pytest.mark.parametrize("dtype", ["bf16", "fp16", "fp32"])
def test_parity_default_path(cuda_device, case, dtype):
    N, d, causal, pad, blocky, p = case
    inp = _case(N, d, dtype, causal, pad, blocky, p)
    got = gpu_fwd_bwd(inp)
    ref = oracle_fwd_bwd(inp)
    compare(got, ref, dtype)


# head dim 256 (16-bit inputs: the one-tile tensor-core forward and the
# three-pass tensor-core backward; fp32: the CUDA-core kernels)
CASES_D256 = [
    (1, 256, False, False, False, 0.0),
    (129, 256, True, False, False, 0.0),
    (300, 256, True, True, False, 0.0),
    (384, 256, False, False, True, 0.1),
    (520, 256, True, False, False, 0.2),
]


@pytest.mark.parametrize("case", CASES_D256, ids=_ids)
@pytest.mark.parametrize("dtype", ["bf16", "fp16", "fp32"])
def test_parity_head_dim_256(cuda_device, case, dtype):
    N, d, causal, pad, blocky, p = case
    inp = _case(N, d, dtype, causal, pad, blocky, p)
    compare(gpu_fwd_bwd(inp), oracle_fwd_bwd(inp), dtype)


@pytest.mark.parametrize("case", CASES[::2] + CASES_D256[1::2], ids=_ids)
@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_parity_cuda_core_path_16bit(cuda_device, case, dtype):
    """The CUDA-core kernels on 16-bit inputs (the tensor-core path's twin)."""
    N, d, causal, pad, blocky, p = case
    inp = _case(N, d, dtype, causal, pad, blocky, p)
    old = fa.fa_set_kernel_path(1)
    try:
        got = gpu_fwd_bwd(inp)
    finally:
        fa.fa_set_kernel_path(old)
    compare(got, oracle_fwd_bwd(inp), dtype)


def test_fully_masked_rows(cuda_device):
    """Rows whose every key is masked: O = 0, LSE = -inf, no gradient."""
    inp = _case(384, 64, "bf16", B=1, H=2)
    bm = torch.ones(3, 3, dtype=torch.uint8)
    bm[1, :] = 0  # query block 1 sees nothing
    inp["block_mask"] = bm
    got = gpu_fwd_bwd(inp)
    ref = oracle_fwd_bwd(inp)
    compare(got, ref, "bf16")
    assert (got["o"][:, :, 128:256] == 0).all()


def test_repeatable(cuda_device):
    """Two runs on the same inputs agree bit for bit for O, LSE, dK, dV."""
    inp = _case(700, 128, "bf16", causal=True, p=0.1)
    a = gpu_fwd_bwd(inp)
    b = gpu_fwd_bwd(inp)
    for key in ("o", "lse", "dk", "dv"):
        assert (a[key] == b[key]).all(), key
    assert abs(a["dq"] - b["dq"]).max() <= 1e-2
