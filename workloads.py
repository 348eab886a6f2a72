"""Seeded synthetic workloads for exact tiled attention.

This module only draws inputs: Q, K, V, dO, per-sequence key lengths and the
block-sparsity mask. It holds none of the attention arithmetic, so both the
fp64 oracle (``oracle/``) and the CUDA library (``io_aware_exact_08_gb300``)
can take their inputs from it without sharing any method code.

Shapes follow the workloads the pages describe: GPT-2 self-attention at
N=1024, d=64 ("FlashAttention" blog post, section "Standard Attention"),
BERT-large at sequence length 512 and long-context / block-sparse runs up to
16K ("FlashAttention: Fast and Memory-Efficient Exact Attention with
IO-Awareness", section "Hasil"). No dataset is read: every tensor is i.i.d.
N(0,1) from a seeded CPU generator.

Recipe (identical for every workload):
  * ``torch.Generator('cpu').manual_seed(seed)``, seed = 1000 + workload index;
  * draw, in this order, fp32 N(0,1) tensors Q, K, V, dO of shape [B,H,N,d];
  * round each to the workload dtype (bf16 and fp16 rounding is round-to-nearest-even);
  * then, if the workload pads keys, kv_len[b] ~ U{lo..hi} (inclusive);
  * the block mask (block 128 x 128) is a fixed pattern, not random.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field, replace
from typing import Optional

import torch

BLOCK = 128  # block size of the block-sparsity mask (queries x keys)


@dataclass(frozen=True)
class Workload:
    name: str
    index: int
    B: int
    H: int
    N: int
    d: int
    dtype: str  # "bf16", "fp16" or "fp32"
    causal: bool = False
    kv_len_range: Optional[tuple] = None  # (lo, hi) inclusive, per sequence
    dropout_p: float = 0.0
    block_sparse: bool = False
    mask_pattern: str = "band_butterfly"  # block-sparse pattern: "band_butterfly" or "local_global"
    scale: Optional[float] = None  # default 1/sqrt(d)
    note: str = ""

    @property
    def softmax_scale(self) -> float:
        return self.scale if self.scale is not None else 1.0 / math.sqrt(self.d)

    @property
    def seed(self) -> int:
        return 1000 + self.index

    @property
    def torch_dtype(self):
        return {"bf16": torch.bfloat16, "fp16": torch.float16, "fp32": torch.float32}[self.dtype]

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)


WORKLOADS = {
    "single_head_fp32": Workload(
        "single_head_fp32", 1, B=1, H=1, N=128, d=64, dtype="fp32",
        note="single head, fp32, no mask, no dropout"),
    "gpt2_causal": Workload(
        "gpt2_causal", 2, B=8, H=12, N=1024, d=64, dtype="bf16", causal=True,
        scale=1.0 / 8.0, note="GPT-2-small-shaped causal self-attention"),
    "bert_pad_dropout": Workload(
        "bert_pad_dropout", 3, B=32, H=16, N=512, d=64, dtype="bf16",
        kv_len_range=(256, 512), dropout_p=0.1, scale=1.0 / 8.0,
        note="BERT-large-shaped attention, key padding, dropout 0.1"),
    "long_causal": Workload(
        "long_causal", 4, B=2, H=16, N=8192, d=128, dtype="bf16", causal=True,
        note="long-context dense causal attention"),
    "block_sparse": Workload(
        "block_sparse", 5, B=1, H=8, N=16384, d=64, dtype="bf16",
        block_sparse=True, note="band(2)+butterfly block-sparse attention"),
}


def sweep_workloads():
    """Forward-only sweep at fixed B*N = 16K tokens, H=16, d=128, causal."""
    out = []
    for i, n in enumerate((1024, 2048, 4096, 8192, 16384)):
        out.append(Workload(f"sweep_n{n}", 10 + i, B=16384 // n, H=16, N=n,
                            d=128, dtype="bf16", causal=True,
                            note="forward sweep at B*N=16K"))
    return out


def splitkv_workloads():
    """Long sequences with few heads, where the two-tile forward grid
    (B*H*ceil(N/256) CTAs) would not fill the GPU: the case split-KV serves."""
    return [Workload("longctx_b1h4", 20, B=1, H=4, N=16384, d=128, dtype="bf16", causal=True,
                     note="few heads, long context"),
            Workload("longctx_b1h2_d64", 21, B=1, H=2, N=8192, d=64, dtype="bf16", causal=False,
                     note="few heads, long context")]


def headdim_workloads():
    """Head dimension 256, the widest the FlashAttention-2 section of the
    "Flash Attention" guide supports ("Dukungan untuk dimensi head yang lebih
    besar"), at 16K tokens per step like the sweep."""
    return [Workload("d256_causal", 30, B=2, H=8, N=4096, d=256, dtype="bf16", causal=True,
                     note="head dim 256")]


def band_butterfly_block_mask(nb: int, band: int = 2) -> torch.Tensor:
    """Block mask M[i][j] (uint8, nb x nb): |i-j| <= band, or j == i XOR 2^k.

    The block-sparse extension restricts attention to the non-zero blocks of
    a fixed mask M in {0,1}^{N/B_r x N/B_c} ("FlashAttention: Fast and
    Memory-Efficient Exact Attention with IO-Awareness", section
    "Ekstensi: Block-Sparse FlashAttention"). The pattern (a diagonal band
    plus butterfly partners) is the workload's choice.
    """
    m = torch.zeros(nb, nb, dtype=torch.uint8)
    for i in range(nb):
        for j in range(max(0, i - band), min(nb, i + band + 1)):
            m[i, j] = 1
        k = 0
        while (1 << k) < nb:
            j = i ^ (1 << k)
            if j < nb:
                m[i, j] = 1
            k += 1
    return m


def local_global_block_mask(nb: int, window: int = 1, n_global: int = 1) -> torch.Tensor:
    """Block mask M[i][j] (uint8, nb x nb): |i-j| <= window, or i < n_global,
    or j < n_global: a sliding window of blocks plus global blocks that see
    and are seen by every block. A second fixed pattern for the block-sparse
    iterator, which accepts any M."""
    m = torch.zeros(nb, nb, dtype=torch.uint8)
    for i in range(nb):
        m[i, max(0, i - window):min(nb, i + window + 1)] = 1
    m[:n_global, :] = 1
    m[:, :n_global] = 1
    return m


def sparse_workloads():
    """Block-sparse attention beyond the 16K workload: the band + butterfly
    pattern at N = 64K (the length of the Path-256 task in the paper
    summary's results, "Hasil (beserta Angka Terpenting)"), and a second
    pattern (sliding window + global blocks) at 16K."""
    return [Workload("block_sparse_64k", 40, B=1, H=8, N=65536, d=64, dtype="bf16", block_sparse=True,
                     note="band(2)+butterfly block-sparse attention at 64K"),
            Workload("block_sparse_local_global", 41, B=1, H=8, N=16384, d=64, dtype="bf16", block_sparse=True,
                     mask_pattern="local_global", note="window(1)+global(1) block-sparse attention")]


def block_mask_density(mask: torch.Tensor) -> float:
    return float(mask.to(torch.float64).mean())


def make_inputs(w: Workload, seed: Optional[int] = None, with_grad_out: bool = True):
    """Draw the workload's tensors on the CPU.

    Returns a dict with q, k, v, do (torch CPU tensors in the workload dtype,
    layout [B,H,N,d] contiguous), kv_len (int32 [B] or None), block_mask
    (uint8 [nb,nb] or None, nb = ceil(N/128)), and the scalars the attention
    call takes (scale, causal, dropout_p, philox seed).
    """
    seed = w.seed if seed is None else seed
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    shape = (w.B, w.H, w.N, w.d)

    def draw():
        return torch.randn(shape, generator=g, dtype=torch.float32).to(w.torch_dtype).contiguous()

    q = draw()
    k = draw()
    v = draw()
    do = draw() if with_grad_out else None
    kv_len = None
    if w.kv_len_range is not None:
        lo, hi = w.kv_len_range
        kv_len = torch.randint(lo, hi + 1, (w.B,), generator=g, dtype=torch.int64).to(torch.int32)
    block_mask = None
    if w.block_sparse:
        nb = (w.N + BLOCK - 1) // BLOCK
        if w.mask_pattern == "local_global":
            block_mask = local_global_block_mask(nb)
        else:
            block_mask = band_butterfly_block_mask(nb)
    return dict(q=q, k=k, v=v, do=do, kv_len=kv_len, block_mask=block_mask,
                scale=w.softmax_scale, causal=w.causal, dropout_p=w.dropout_p,
                seed=seed)


def random_block_mask(nb: int, density: float, seed: int) -> torch.Tensor:
    """A random block mask for edge-case tests (diagonal forced on)."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    m = (torch.rand(nb, nb, generator=g) < density).to(torch.uint8)
    for i in range(nb):
        m[i, i] = 1
    return m


FP8_MAX = 448.0  # largest finite E4M3 magnitude


def quantize_e4m3(x: torch.Tensor):
    """Per-head E4M3 quantisation of a [B,H,N,d] tensor for the FP8 forward.

    Returns (codes, descale): codes are the uint8 E4M3 bytes of x / descale,
    rounded to nearest even by torch's float8_e4m3fn conversion, and descale
    (fp32 [B*H]) is each head's max |x| / 448, so the real input is
    code * descale (1 where a head is all zeros). Only input preparation: the
    oracle and the library both take these bytes and factors as they are.
    """
    B, H, N, d = x.shape
    xf = x.to(torch.float32).reshape(B * H, N * d)
    amax = xf.abs().amax(dim=1)
    descale = torch.where(amax > 0, amax / FP8_MAX, torch.ones_like(amax))
    scaled = (xf / descale[:, None]).clamp_(-FP8_MAX, FP8_MAX)
    codes = scaled.to(torch.float8_e4m3fn).view(torch.uint8).reshape(B, H, N, d).contiguous()
    return codes, descale.contiguous()


def make_fp8_inputs(w: Workload, seed: Optional[int] = None):
    """The workload's Q, K, V (drawn as for the 16-bit workloads, in fp32)
    quantised per head to E4M3: codes q8, k8, v8 ([B,H,N,d] uint8), their
    factors (fp32 [B*H]), and v8 transposed to [B,H,d,N] for the library."""
    w32 = w.with_(dtype="fp32")
    inp = make_inputs(w32, seed=seed, with_grad_out=False)
    out = dict(inp)
    for n in ("q", "k", "v"):
        codes, ds = quantize_e4m3(inp[n])
        out[n + "8"] = codes
        out["descale_" + n] = ds
    out["vt8"] = out["v8"].transpose(2, 3).contiguous()
    return out
