"""The seeded input generators: mask patterns and workload shapes (no
attention arithmetic here)."""
import torch

from workloads import (BLOCK, band_butterfly_block_mask, block_mask_density, headdim_workloads,
                       local_global_block_mask, make_inputs, sparse_workloads, splitkv_workloads)


def test_local_global_pattern():
    m = local_global_block_mask(16, window=1, n_global=1)
    assert m.dtype == torch.uint8 and m.shape == (16, 16)
    assert bool((m[0] == 1).all()) and bool((m[:, 0] == 1).all())  # the global block row and column
    for i in range(16):
        for j in range(16):
            expect = abs(i - j) <= 1 or i == 0 or j == 0
            assert int(m[i, j]) == int(expect)
    assert torch.equal(m, m.t())


def test_band_butterfly_at_64k():
    m = band_butterfly_block_mask(512)
    assert bool((torch.diagonal(m) == 1).all())
    # band |i-j| <= 2 plus the 9 butterfly partners i XOR 2^k
    i = 100
    row = set(torch.nonzero(m[i]).flatten().tolist())
    assert row == set(range(98, 103)) | {i ^ (1 << k) for k in range(9)}
    assert abs(block_mask_density(m) - 0.02341) < 1e-4


def test_new_workload_shapes():
    names = {w.name: w for w in sparse_workloads() + splitkv_workloads() + headdim_workloads()}
    assert names["block_sparse_64k"].N == 65536 and names["block_sparse_64k"].block_sparse
    assert names["block_sparse_local_global"].mask_pattern == "local_global"
    assert names["d256_causal"].d == 256 and names["d256_causal"].causal
    w = names["block_sparse_local_global"].with_(N=1024, H=1)
    inp = make_inputs(w, with_grad_out=False)
    assert torch.equal(inp["block_mask"], local_global_block_mask(1024 // BLOCK))


def test_fp16_inputs_round_the_same_draws():
    w = headdim_workloads()[0].with_(N=256, H=1, B=1)
    a = make_inputs(w, with_grad_out=False)
    b = make_inputs(w.with_(dtype="fp16"), with_grad_out=False)
    assert a["q"].dtype == torch.bfloat16 and b["q"].dtype == torch.float16
    # both are the same fp32 draw rounded to nearest: they agree to bf16 precision
    assert torch.allclose(a["q"].float(), b["q"].float(), rtol=2 ** -8, atol=0)
