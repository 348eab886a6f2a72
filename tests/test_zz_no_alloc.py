"""fa_bwd_noalloc against fa_bwd, through the C ABI.

fa_bwd_noalloc serves callers that cannot allocate device memory (their
framework's allocator already owns the GPU, or allocation is not allowed on
their path): it takes the backward workspace from a fixed array inside the
library instead of from the caller. It must give the same gradients as
fa_bwd with a caller-provided workspace, on consecutive calls that reuse
that array, and refuse problems whose workspace does not fit.

This file is collected last on purpose: it exercises shared device state.
"""
import numpy as np
import pytest
import torch

import io_aware_exact_08_gb300 as fa
from parity_utils import TOL, max_err
from workloads import Workload, make_inputs

pytestmark = pytest.mark.gpu


def _ptr(t):
    return None if t is None else t.data_ptr()


def _run_both(w, seed):
    inp = make_inputs(w, seed=seed)
    dev = lambda t: None if t is None else t.cuda().contiguous()
    q, k, v, do = (dev(inp[n]) for n in ("q", "k", "v", "do"))
    kl = dev(inp["kv_len"])
    B, H, N, d = q.shape
    code = fa.FA_BF16 if q.dtype == torch.bfloat16 else fa.FA_FP32
    stream = torch.cuda.current_stream().cuda_stream
    o, lse = fa.attention_fwd(q, k, v, scale=inp["scale"], causal=inp["causal"], dropout_p=inp["dropout_p"],
                              seed=inp["seed"], kv_len=kl)
    args = (B, H, N, d, inp["scale"], int(inp["causal"]), None, inp["dropout_p"], inp["seed"], code, _ptr(kl))
    ref = [torch.empty_like(q) for _ in range(3)]
    ws_bytes = fa.fa_bwd_workspace_size(B, H, N, d)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=q.device)
    rc = fa.fa_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(do), *map(_ptr, ref), *args, _ptr(ws),
                   ws_bytes, stream)
    assert rc == 0, fa.fa_status_string(rc)
    got = [torch.empty_like(q) for _ in range(3)]
    rc = fa.fa_bwd_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(do), *map(_ptr, got), *args, stream)
    assert rc == 0, fa.fa_status_string(rc)
    torch.cuda.synchronize()
    st, site = fa.fa_check_device_status(stream)
    assert st == 0, (st, site)
    tol = TOL[w.dtype]
    for name, a, b in zip(("dq", "dk", "dv"), got, ref):
        a64 = a.float().cpu().numpy().astype(np.float64)
        b64 = b.float().cpu().numpy().astype(np.float64)
        assert max_err(a64, b64, allowance=w.dtype) <= tol[name], name


@pytest.mark.parametrize("w", [
    Workload("noalloc_bf16", 0, B=2, H=3, N=300, d=128, dtype="bf16", causal=True, dropout_p=0.1),
    Workload("noalloc_bf16_pad", 0, B=2, H=2, N=640, d=64, dtype="bf16", kv_len_range=(200, 640)),
    Workload("noalloc_fp32", 0, B=1, H=2, N=200, d=64, dtype="fp32", causal=True),
], ids=lambda w: w.name)
def test_noalloc_matches_fa_bwd_on_consecutive_calls(cuda_device, w):
    # two calls in a row on different inputs: the shared array is reused
    _run_both(w, seed=21)
    _run_both(w, seed=22)


def test_noalloc_refuses_oversized_problem(cuda_device):
    B, H, N, d = 8, 16, 8192, 128  # workspace far above the fixed array
    assert fa.fa_bwd_workspace_size(B, H, N, d) > fa.FA_BWD_NOALLOC_SCRATCH_BYTES
    fake = 1 << 20  # never dereferenced: the size check comes first
    rc = fa.fa_bwd_noalloc(fake, fake, fake, fake, fake, fake, fake, fake, fake, B, H, N, d, 0.1, 0, None, 0.0, 0,
                           fa.FA_BF16, None, None)
    assert rc == -4
    assert "WORKSPACE" in fa.fa_status_string(rc)
