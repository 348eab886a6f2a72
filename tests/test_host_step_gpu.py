"""fa_fwd_bwd_host on GB300: a forward + backward step on host tensors, the
copies overlapped with the kernels chunk by chunk.

Each case forces a chunk size so that several chunks pass through the ring
of device slots (more chunks than slots, so slots are reused), and checks:
 - every output against the fp64 oracle, with the parity tolerances;
 - o, lse, dk and dv bit for bit against fa_fwd + fa_bwd on device copies of
   the same inputs: per head the same kernels run in the same order whatever
   the chunk, and only dQ (fp32 reduce-adds from the key tiles, in the order
   the backward's CTAs claim them) may differ in its last bits.
"""
import numpy as np
import pytest
import torch

import io_aware_exact_08_gb300 as fa
from parity_utils import compare, gpu_fwd_bwd, oracle_fwd_bwd
from workloads import Workload, make_inputs

pytestmark = pytest.mark.gpu

CASES = [
    # name, workload, chunk_heads
    ("d64_causal_reuse", Workload("h1", 0, B=2, H=3, N=300, d=64, dtype="bf16", causal=True), 1),
    ("d128_kvlen_in_batch", Workload("h2", 0, B=2, H=3, N=333, d=128, dtype="bf16", kv_len_range=(90, 333)), 2),
    ("d128_kvlen_batches", Workload("h3", 0, B=5, H=2, N=257, d=128, dtype="fp16", causal=True,
                                    kv_len_range=(1, 257)), 2),
    ("d64_block_sparse", Workload("h4", 0, B=1, H=5, N=512, d=64, dtype="bf16", block_sparse=True), 1),
    ("d128_dropout_one_chunk", Workload("h5", 0, B=2, H=2, N=200, d=128, dtype="bf16", causal=True,
                                        dropout_p=0.15), 1),
    ("d256_causal", Workload("h6", 0, B=1, H=4, N=260, d=256, dtype="bf16", causal=True), 1),
    ("fp32_d64", Workload("h7", 0, B=1, H=4, N=130, d=64, dtype="fp32", causal=True), 1),
    ("one_row", Workload("h10", 0, B=2, H=2, N=1, d=64, dtype="bf16", causal=True), 1),
    ("kvlen_one_head_batches", Workload("h11", 0, B=4, H=1, N=190, d=128, dtype="bf16", kv_len_range=(1, 190)), 1),
]


def _host_step(inp, chunk_heads, device, pinned=True):
    pin = (lambda t: t.pin_memory()) if pinned else (lambda t: t.contiguous())
    q = pin(inp["q"])
    k, v, do = (pin(inp[n]) for n in ("k", "v", "do"))
    o, lse, dq, dk, dv = fa.attention_fwd_bwd_host(
        q, k, v, do, scale=inp["scale"], causal=inp["causal"], block_mask=inp["block_mask"],
        dropout_p=inp["dropout_p"], seed=inp["seed"], kv_len=inp["kv_len"], chunk_heads=chunk_heads,
        device=device)
    torch.cuda.synchronize(device)
    st, site = fa.fa_check_device_status(torch.cuda.current_stream(device).cuda_stream)
    assert st == 0, f"device status {st} at site {site}"
    return {n: t.float().numpy().astype(np.float64) for n, t in (("o", o), ("lse", lse), ("dq", dq),
                                                                  ("dk", dk), ("dv", dv))}


@pytest.mark.parametrize("name,w,chunk_heads", CASES, ids=[c[0] for c in CASES])
def test_host_step_matches_oracle_and_device_path(cuda_device, name, w, chunk_heads):
    inp = make_inputs(w, seed=31)
    chunks = fa.fa_fwd_bwd_host_chunks(w.B, w.H, w.N, 1 if inp["kv_len"] is not None else None, w.dropout_p,
                                       chunk_heads)
    if w.dropout_p == 0:
        assert len(chunks) > 3, "the case should reuse device slots"
    got = _host_step(inp, chunk_heads, cuda_device)
    errs = compare(got, oracle_fwd_bwd(inp), w.dtype)
    dev = gpu_fwd_bwd(inp, cuda_device)
    for key in ("o", "lse", "dk", "dv"):
        same = np.array_equal(got[key], dev[key], equal_nan=True)
        assert same, f"{key} differs from the device path (max {np.nanmax(np.abs(got[key] - dev[key]))})"
    print(name, len(chunks), "chunks", errs)


def test_automatic_chunks_on_a_larger_step(cuda_device):
    """The library's own chunk size on a step big enough to split (B=1 H=40
    N=4096 d=128, causal: 1,280 query tiles, four chunks of 10 heads): the
    device path's results, and the oracle on the first and last head of
    each chunk."""
    w = Workload("h8", 0, B=1, H=40, N=4096, d=128, dtype="bf16", causal=True)
    inp = make_inputs(w, seed=32)
    chunks = fa.fa_fwd_bwd_host_chunks(w.B, w.H, w.N, None, 0.0, 0)
    assert len(chunks) == 4
    got = _host_step(inp, 0, cuda_device)
    dev = gpu_fwd_bwd(inp, cuda_device)
    for key in ("o", "lse", "dk", "dv"):
        assert np.array_equal(got[key], dev[key], equal_nan=True), key
    assert np.max(np.abs(got["dq"] - dev["dq"])) <= 1e-2
    heads = sorted({c[0] for c in chunks} | {c[0] + c[2] - 1 for c in chunks})
    compare(got, oracle_fwd_bwd(inp, heads=heads), w.dtype, heads=heads)


def test_back_to_back_calls_share_the_workspace(cuda_device):
    """Three steps queued on one stream with one workspace, without a
    synchronisation between them: each call's copies wait for the previous
    call's work, so every step returns its own inputs' results."""
    w = Workload("h9", 0, B=1, H=6, N=256, d=64, dtype="bf16", causal=True)
    inps = [make_inputs(w, seed=40 + i) for i in range(3)]
    wsb = fa.fa_fwd_bwd_host_workspace_size(w.B, w.H, w.N, w.d, fa.FA_BF16, None, 0.0, None, 1)
    ws = torch.empty(wsb, dtype=torch.uint8, device=cuda_device)
    outs = []
    for inp in inps:
        pinned = [inp[n].pin_memory() for n in ("q", "k", "v", "do")]
        outs.append((pinned, fa.attention_fwd_bwd_host(*pinned, scale=inp["scale"], causal=True, chunk_heads=1,
                                                       workspace=ws, device=cuda_device)))
    torch.cuda.synchronize(cuda_device)
    for inp, (_, res) in zip(inps, outs):
        got = {n: t.float().numpy().astype(np.float64) for n, t in zip(("o", "lse", "dq", "dk", "dv"), res)}
        compare(got, oracle_fwd_bwd(inp), "bf16")


def test_pageable_host_memory(cuda_device):
    """Pageable (not page-locked) host tensors: the driver stages the copies
    and the call returns only after them, with the same results."""
    w = Workload("h12", 0, B=1, H=5, N=200, d=128, dtype="bf16", causal=True)
    inp = make_inputs(w, seed=33)
    assert not inp["q"].is_pinned()
    got = _host_step(inp, 1, cuda_device, pinned=False)
    ref = _host_step(inp, 1, cuda_device, pinned=True)
    for key in ("o", "lse", "dk", "dv"):
        assert np.array_equal(got[key], ref[key], equal_nan=True), key
    compare(got, oracle_fwd_bwd(inp), "bf16")
