"""The forward's O and the d = 64 backward's dK, dV leave through TMA stores of
whole 128-row tiles, and the d = 128 forward stores two 64-column boxes per
tile: rows past N lie outside the tensor and must not be written. Each output
here is a view at the start of a larger buffer whose tail holds a sentinel;
with a ragged N the last tile of the last head ends past the tensor, so a
store that is not clipped would overwrite the sentinel. The results are also
checked against the fp64 oracle on every head."""
import numpy as np
import pytest
import torch

import io_aware_exact_08_gb300 as fa
from parity_utils import compare, oracle_fwd_bwd

pytestmark = pytest.mark.gpu

SENTINEL = 1234.0


def _guarded(shape, dev):
    n = 1
    for x in shape:
        n *= x
    guard = 128 * shape[-1] * 2  # two tiles of rows past the tensor's end
    buf = torch.full((n + guard,), SENTINEL, dtype=torch.bfloat16, device=dev)
    return buf, buf[:n].view(*shape), n


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_outputs_end_at_their_tensors(cuda_device, d, causal):
    B, H, N = 1, 3, 200
    g = torch.Generator(device="cpu")
    g.manual_seed(21 + d)
    shape = (B, H, N, d)
    draw = lambda: torch.randn(shape, generator=g, dtype=torch.float32).to(torch.bfloat16)
    q, k, v, do = (draw() for _ in range(4))
    qd, kd, vd, dod = (t.to(cuda_device) for t in (q, k, v, do))
    ob, o, n = _guarded(shape, cuda_device)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=cuda_device)
    fa.attention_fwd(qd, kd, vd, causal=causal, out=o, lse=lse)
    torch.cuda.synchronize()
    tail = torch.full((ob.numel() - n,), SENTINEL, dtype=torch.bfloat16, device=cuda_device)
    assert torch.equal(ob[n:], tail), "the forward wrote past the end of O"
    grads = [_guarded(shape, cuda_device) for _ in range(3)]
    fa.attention_bwd(qd, kd, vd, o, lse, dod, causal=causal, dq=grads[0][1], dk=grads[1][1], dv=grads[2][1])
    torch.cuda.synchronize()
    st, site = fa.fa_check_device_status(torch.cuda.current_stream().cuda_stream)
    assert st == 0, f"device status {st} at site {site}"
    for name, (buf, _, _) in zip(("dq", "dk", "dv"), grads):
        assert torch.equal(buf[n:], tail), f"the backward wrote past the end of {name}"
    inp = dict(q=q, k=k, v=v, do=do, kv_len=None, block_mask=None, scale=d ** -0.5, causal=causal, dropout_p=0.0,
               seed=0)
    as64 = lambda t: t.float().cpu().numpy().astype(np.float64)
    got = {"o": as64(o), "lse": as64(lse)}
    for name, (_, t, _) in zip(("dq", "dk", "dv"), grads):
        got[name] = as64(t)
    errs = compare(got, oracle_fwd_bwd(inp), "bf16")
    print("store bounds", d, causal, errs)
