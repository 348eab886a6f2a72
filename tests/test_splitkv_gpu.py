"""Split-KV forward (fa_fwd_splitkv): the key tiles of every pair of query
tiles are cut into ranges computed by separate CTAs and merged with the
incremental-softmax combination. Checked against the fp64 oracle element by
element, and against the single-pass forward."""
import numpy as np
import pytest
import torch

import io_aware_exact_08_gb300 as fa
import oracle
from parity_utils import compare, oracle_fwd_bwd, to_dev
from workloads import Workload, make_inputs, random_block_mask

pytestmark = pytest.mark.gpu


def _inputs(N, d, causal=False, pad=False, blocky=False, p=0.0, B=2, H=3, seed=11, dtype="bf16"):
    w = Workload("splitkv", 0, B=B, H=H, N=N, d=d, dtype=dtype, causal=causal,
                 kv_len_range=((max(1, N // 2), N) if pad else None), dropout_p=p)
    inp = make_inputs(w, seed=seed, with_grad_out=False)
    if blocky:
        inp["block_mask"] = random_block_mask((N + 127) // 128, 0.5, seed + 1)
    return inp


def _run(inp, splits):
    q, k, v = (to_dev(inp[n]) for n in ("q", "k", "v"))
    o, lse = fa.attention_fwd(q, k, v, scale=inp["scale"], causal=inp["causal"],
                              block_mask=to_dev(inp["block_mask"]), dropout_p=inp["dropout_p"], seed=inp["seed"],
                              kv_len=to_dev(inp["kv_len"]), num_splits=splits)
    torch.cuda.synchronize()
    st, site = fa.fa_check_device_status(torch.cuda.current_stream().cuda_stream)
    assert st == 0, f"device status {st} at site {site}"
    return {"o": o.float().cpu().numpy().astype(np.float64), "lse": lse.cpu().numpy().astype(np.float64)}


CASES = [
    # N, d, causal, pad, blocky, dropout, splits
    (1000, 128, True, False, False, 0.0, 3),
    (768, 128, False, False, False, 0.0, 6),
    (640, 64, False, True, True, 0.1, 2),
    (300, 64, True, True, False, 0.2, 4),   # more splits than key tiles for the first pairs
    (1024, 64, True, False, False, 0.0, 8),
    (520, 128, True, False, True, 0.0, 3),
    (520, 256, True, False, False, 0.0, 3),
    (384, 256, False, True, True, 0.1, 2),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"N{c[0]}-d{c[1]}-s{c[6]}")
def test_splitkv_matches_oracle(cuda_device, case):
    N, d, causal, pad, blocky, p, splits = case
    inp = _inputs(N, d, causal, pad, blocky, p)
    got = _run(inp, splits)
    ref = oracle_fwd_bwd(inp, backward=False)
    compare(got, ref, "bf16", keys=("o", "lse"))


@pytest.mark.parametrize("case", CASES[::2], ids=lambda c: f"N{c[0]}-d{c[1]}-s{c[6]}")
def test_splitkv_fp16_matches_oracle(cuda_device, case):
    N, d, causal, pad, blocky, p, splits = case
    inp = _inputs(N, d, causal, pad, blocky, p, dtype="fp16")
    got = _run(inp, splits)
    compare(got, oracle_fwd_bwd(inp, backward=False), "fp16", keys=("o", "lse"))


def test_splitkv_agrees_with_single_pass(cuda_device):
    inp = _inputs(1024, 128, causal=True, B=1, H=4)
    a = _run(inp, 1)
    b = _run(inp, 4)
    assert np.abs(a["lse"] - b["lse"]).max() <= 1e-4
    assert np.abs(a["o"] - b["o"]).max() <= 2e-2


def test_splitkv_fully_masked_rows(cuda_device):
    inp = _inputs(384, 64, B=1, H=2)
    bm = torch.ones(3, 3, dtype=torch.uint8)
    bm[1, :] = 0
    inp["block_mask"] = bm
    got = _run(inp, 2)
    compare(got, oracle_fwd_bwd(inp, backward=False), "bf16", keys=("o", "lse"))
    assert (got["o"][:, :, 128:256] == 0).all()
    assert np.isneginf(got["lse"][:, :, 128:256]).all()
