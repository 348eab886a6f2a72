"""The backward's persistent grid with more items than SMs: every CTA claims
further (head, key tile) items from the workspace counter, and items that no
query sees (dead key tiles) are skipped by every role. Checked against the
fp64 oracle on sampled heads, and on every head dK = dV = 0 on dead key rows."""
import numpy as np
import pytest
import torch

from parity_utils import compare, gpu_fwd_bwd, oracle_fwd_bwd
from workloads import random_block_mask

pytestmark = pytest.mark.gpu


def _inputs(B, H, N, d, seed, causal, block_mask=None, kv_len=None):
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    shape = (B, H, N, d)
    draw = lambda: torch.randn(shape, generator=g, dtype=torch.float32).to(torch.bfloat16).contiguous()
    q, k, v, do = draw(), draw(), draw(), draw()
    return dict(q=q, k=k, v=v, do=do, kv_len=kv_len, block_mask=block_mask, scale=d ** -0.5, causal=causal,
                dropout_p=0.0, seed=seed)


def test_block_mask_with_dead_key_tiles(cuda_device):
    """d = 64, 8 heads x 32 key tiles = 256 items over a grid of at most one
    CTA per SM: a random block mask with every key-tile column j = 3 mod 5
    emptied, so those items have no query tile and their dK, dV rows are 0."""
    B, H, N, d = 2, 4, 4096, 64
    nb = N // 128
    mask = random_block_mask(nb, 0.25, seed=11)
    dead = [j for j in range(nb) if j % 5 == 3]
    mask[:, dead] = 0
    inp = _inputs(B, H, N, d, seed=5, causal=False, block_mask=mask)
    got = gpu_fwd_bwd(inp)
    heads = [1, 6]
    errs = compare(got, oracle_fwd_bwd(inp, heads=heads), "bf16", heads=heads)
    print("dead key tiles", errs)
    rows = np.concatenate([np.arange(j * 128, (j + 1) * 128) for j in dead])
    assert np.all(got["dk"][:, :, rows, :] == 0) and np.all(got["dv"][:, :, rows, :] == 0)


def test_key_padding_with_dead_key_tiles_d128(cuda_device):
    """d = 128, causal, per-sequence key lengths: 4 x 4 heads x 16 key tiles
    = 256 items, those past a sequence's length dead."""
    B, H, N, d = 4, 4, 2048, 128
    kv_len = torch.tensor([2048, 700, 1, 1300], dtype=torch.int32)
    inp = _inputs(B, H, N, d, seed=9, causal=True, kv_len=kv_len)
    got = gpu_fwd_bwd(inp)
    heads = [4, 13]  # batches 1 and 3
    errs = compare(got, oracle_fwd_bwd(inp, heads=heads), "bf16", heads=heads)
    print("key padding", errs)
    for b, L in enumerate(kv_len.tolist()):
        assert np.all(got["dk"][b, :, L:, :] == 0) and np.all(got["dv"][b, :, L:, :] == 0)
