"""Full-size workloads, run exactly as the benchmark launches them, checked
against the fp64 oracle on sampled heads (the oracle computes each head
independently), plus properties that hold at any size."""
import numpy as np
import pytest

from parity_utils import compare, gpu_fwd_bwd, gpu_forward, oracle_fwd_bwd
from workloads import WORKLOADS, headdim_workloads, make_inputs, sparse_workloads, sweep_workloads

pytestmark = pytest.mark.gpu

# flat head indices (b*H + h) checked against the oracle for each workload
SAMPLED_HEADS = {
    "single_head_fp32": None,              # all
    "gpt2_causal": [0, 13, 50, 95],
    "bert_pad_dropout": [0, 17, 100, 255, 300, 511],
    "long_causal": [0, 31],
    "block_sparse": [5],
}


@pytest.mark.parametrize("name", list(WORKLOADS))
def test_workload_parity(cuda_device, name):
    w = WORKLOADS[name]
    inp = make_inputs(w)
    got = gpu_fwd_bwd(inp)
    heads = SAMPLED_HEADS[name]
    ref = oracle_fwd_bwd(inp, heads=heads)
    errs = compare(got, ref, w.dtype, heads=heads)
    print(name, errs)
    # any-size properties on every head
    for key in ("o", "dq", "dk", "dv"):
        assert np.isfinite(got[key]).all(), key
    lse = got["lse"]
    assert (np.isfinite(lse) | np.isneginf(lse)).all()


@pytest.mark.parametrize("w", sweep_workloads(), ids=lambda w: w.name)
def test_sweep_forward_parity(cuda_device, w):
    inp = make_inputs(w, with_grad_out=False)
    q, k, v, o, lse = gpu_forward(inp)
    got = {"o": o.float().cpu().numpy().astype(np.float64), "lse": lse.cpu().numpy().astype(np.float64)}
    heads = [0, w.B * w.H - 1]
    ref = oracle_fwd_bwd(inp, heads=heads, backward=False)
    compare(got, ref, w.dtype, keys=("o", "lse"), heads=heads)


@pytest.mark.parametrize("name", ["gpt2_causal", "bert_pad_dropout", "long_causal"])
def test_workload_parity_fp16(cuda_device, name):
    """The same workloads with fp16 inputs, as `bench.py --dtype fp16` runs them."""
    w = WORKLOADS[name].with_(dtype="fp16")
    inp = make_inputs(w)
    got = gpu_fwd_bwd(inp)
    heads = SAMPLED_HEADS[name]
    errs = compare(got, oracle_fwd_bwd(inp, heads=heads), "fp16", heads=heads)
    print(name, "fp16", errs)
    for key in ("o", "dq", "dk", "dv"):
        assert np.isfinite(got[key]).all(), key


@pytest.mark.parametrize("w", headdim_workloads(), ids=lambda w: w.name)
def test_headdim_workload_parity(cuda_device, w):
    """Head dim 256 at full size, as the benchmark runs it, on two sampled heads."""
    inp = make_inputs(w)
    got = gpu_fwd_bwd(inp)
    heads = [0, w.B * w.H - 1]
    errs = compare(got, oracle_fwd_bwd(inp, heads=heads), w.dtype, heads=heads)
    print(w.name, errs)


@pytest.mark.parametrize("w", sparse_workloads(), ids=lambda w: w.name)
def test_sparse_workload_parity(cuda_device, w):
    """Block-sparse at 64K and with a second pattern, as the benchmark runs
    them: the oracle on one sampled head, and on every head two identities
    that hold at any size. Softmax rows sum to 1, so sum_j dS_ij = 0 and
    sum_j dK_j = scale sum_i (sum_j dS_ij) Q_i = 0; without dropout
    sum_j dV_j = sum_i (sum_j P_ij) dO_i = sum_i dO_i (every row sees its
    diagonal block)."""
    inp = make_inputs(w)
    got = gpu_fwd_bwd(inp)
    heads = [w.B * w.H - 1]
    errs = compare(got, oracle_fwd_bwd(inp, heads=heads), w.dtype, heads=heads)
    print(w.name, errs)
    dk, dv = got["dk"], got["dv"]
    do = inp["do"].double().numpy()
    for b in range(w.B):
        for h in range(w.H):
            assert np.abs(dk[b, h].sum(0)).max() <= 1e-3 * np.abs(dk[b, h]).sum(0).max()
            gap = np.abs(dv[b, h].sum(0) - do[b, h].sum(0)).max()
            assert gap <= 1e-3 * np.abs(dv[b, h]).sum(0).max()


def test_forward_64k_d128_block_mask_on_tensor_cores(cuda_device):
    """A block mask with 512 key tiles per row at d = 128 fits the forward's
    tile lists: the forward runs on the tensor-core kernel (timed: the
    CUDA-core kernels would take far longer than the bound) and matches the
    oracle on the head. The backward's lists at d = 128 hold 256 tiles, so
    the backward is refused (FA_ERR_UNSUPPORTED) instead of being sent to the
    CUDA-core kernels."""
    import torch
    import io_aware_exact_08_gb300 as fa
    from workloads import Workload
    w = Workload("block_sparse_64k_d128", 42, B=1, H=1, N=65536, d=128, dtype="bf16", block_sparse=True)
    inp = make_inputs(w)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    for e in ev:
        e.record()
    gpu_forward(inp)  # warm-up
    fa.fa_set_main_kernel_events(ev[0].cuda_event, ev[1].cuda_event)
    try:
        q, k, v, o, lse = gpu_forward(inp)
    finally:
        fa.fa_set_main_kernel_events(None, None)
    torch.cuda.synchronize()
    kernel_ms = ev[0].elapsed_time(ev[1])
    assert kernel_ms < 3.0, kernel_ms  # ~51 GFLOP of visible work
    got = {"o": o.float().cpu().numpy().astype(np.float64), "lse": lse.cpu().numpy().astype(np.float64)}
    errs = compare(got, oracle_fwd_bwd(inp, heads=[0], backward=False), "bf16", keys=("o", "lse"), heads=[0])
    print(w.name, kernel_ms, errs)
    do = torch.zeros_like(q)
    with pytest.raises(fa.FaError) as e:
        fa.attention_bwd(q, k, v, o, lse, do, scale=inp["scale"], block_mask=inp["block_mask"].cuda())
    assert e.value.status == -2
