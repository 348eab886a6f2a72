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
