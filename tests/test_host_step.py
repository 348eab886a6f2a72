"""Host logic of fa_fwd_bwd_host (no GPU): how a step on host tensors is cut
into chunks of heads, the workspace those chunks need, and the argument
checks that run before anything touches the device."""
import itertools

import pytest

import io_aware_exact_08_gb300 as fa

FAKE = 1 << 20  # a 256-byte aligned non-null value; never dereferenced on these paths


def r256(x):
    return (x + 255) // 256 * 256


def _check_partition(B, H, chunks, kv_len, dropout):
    """Every head exactly once, in order; each chunk is a valid problem."""
    nxt = 0
    for head0, cb, ch, b0 in chunks:
        assert head0 == nxt
        assert cb >= 1 and ch >= 1
        nxt += cb * ch
        if dropout:
            assert (head0, cb, ch, b0) == (0, B, H, 0)
        elif kv_len:
            if cb > 1 or ch == H:
                # whole batches starting at batch b0
                assert ch == H and head0 == b0 * H
            else:
                # a run of heads inside batch b0
                assert b0 * H <= head0 and head0 + ch <= (b0 + 1) * H
        else:
            assert cb == 1
    assert nxt == B * H


@pytest.mark.parametrize("B,H,N", [(1, 1, 128), (2, 3, 300), (2, 16, 8192), (8, 12, 1024), (32, 16, 512),
                                   (3, 40, 4096), (1, 1000, 64), (7, 5, 129)])
@pytest.mark.parametrize("kv_len", [None, FAKE])
@pytest.mark.parametrize("dropout", [0.0, 0.1])
@pytest.mark.parametrize("chunk_heads", [0, 1, 2, 5, 16, 10 ** 6])
def test_chunks_partition_the_heads(B, H, N, kv_len, dropout, chunk_heads):
    chunks = fa.fa_fwd_bwd_host_chunks(B, H, N, kv_len, dropout, chunk_heads)
    _check_partition(B, H, chunks, kv_len is not None, dropout > 0)
    if dropout == 0 and chunk_heads > 0:
        assert all(cb * ch <= chunk_heads for _, cb, ch, _ in chunks)
        # as few chunks as that size allows, as even as possible
        G = min(chunk_heads, B * H)
        ceil = lambda a, b: -(-a // b)
        if kv_len is None:  # runs of heads
            n_expect, sizes = ceil(B * H, G), [ch for _, _, ch, _ in chunks]
        elif G >= H:  # whole batches
            n_expect, sizes = ceil(B, G // H), [cb for _, cb, _, _ in chunks]
        else:  # runs of heads inside each batch
            n_expect, sizes = B * ceil(H, G), [ch for _, _, ch, _ in chunks]
        assert len(chunks) == n_expect
        assert max(sizes) - min(sizes) <= 1


@pytest.mark.parametrize("B,H,N", [(2, 16, 8192), (8, 12, 1024), (32, 16, 512), (1, 8, 16384), (1, 2, 256),
                                   (4, 64, 2048)])
def test_automatic_chunks(B, H, N):
    """At most four chunks; every chunk holds at least min(512, max(256,
    8 heads)) query tiles unless the whole step has fewer; a step too small
    to split stays one chunk."""
    nt = (N + 127) // 128
    least = min(512, max(256, 8 * nt))
    chunks = fa.fa_fwd_bwd_host_chunks(B, H, N, None, 0.0, 0)
    assert 1 <= len(chunks) <= 4
    if B * H * nt < 2 * least:
        assert len(chunks) == 1
    for _, cb, ch, _ in chunks:
        assert cb * ch * nt >= min(least, B * H * nt)
    sizes = [cb * ch for _, cb, ch, _ in chunks]
    assert max(sizes) - min(sizes) <= 1  # balanced


def test_example_plans():
    # B=2 H=16 N=8K: 64 tiles per head, 8 heads (512 tiles) per chunk
    assert fa.fa_fwd_bwd_host_chunks(2, 16, 8192, None, 0.0, 0) == [(0, 1, 8, 0), (8, 1, 8, 0), (16, 1, 8, 0),
                                                                   (24, 1, 8, 0)]
    # B=8 H=12 N=1K: 8 tiles per head, 32 heads for 256 tiles, 3 chunks
    assert fa.fa_fwd_bwd_host_chunks(8, 12, 1024, None, 0.0, 0) == [(0, 1, 32, 0), (32, 1, 32, 0), (64, 1, 32, 0)]
    # B=1 H=4 N=16K: 128 tiles per head, 4 heads for 512 tiles, one chunk
    assert fa.fa_fwd_bwd_host_chunks(1, 4, 16384, None, 0.0, 0) == [(0, 1, 4, 0)]
    # B=2 H=8 N=4K: 32 tiles per head, 8 heads (256 tiles) per chunk
    assert fa.fa_fwd_bwd_host_chunks(2, 8, 4096, None, 0.0, 0) == [(0, 1, 8, 0), (8, 1, 8, 0)]
    # key padding, 2 heads per chunk of 3-head batches: pieces inside each batch
    assert fa.fa_fwd_bwd_host_chunks(2, 3, 300, FAKE, 0.0, 2) == [(0, 1, 2, 0), (2, 1, 1, 0), (3, 1, 2, 1),
                                                                  (5, 1, 1, 1)]
    # key padding, 6 heads per chunk of 3-head batches: two whole batches, then one
    assert fa.fa_fwd_bwd_host_chunks(3, 3, 300, FAKE, 0.0, 6) == [(0, 2, 3, 0), (6, 1, 3, 2)]
    # dropout: one chunk
    assert fa.fa_fwd_bwd_host_chunks(2, 16, 8192, None, 0.1, 4) == [(0, 2, 16, 0)]


@pytest.mark.parametrize("B,H,N,d,dt", [(2, 16, 8192, 128, fa.FA_BF16), (2, 3, 300, 64, fa.FA_FP16),
                                        (1, 5, 1000, 256, fa.FA_FP32), (8, 12, 1024, 64, fa.FA_BF16)])
@pytest.mark.parametrize("mask,kv_len,dropout,chunk_heads", list(itertools.product(
    [None, FAKE], [None, FAKE], [0.0, 0.2], [0, 1, 4])))
def test_workspace_size(B, H, N, d, dt, mask, kv_len, dropout, chunk_heads):
    """kv_len and the block mask first, then min(3, chunks) slots of eight
    tensors, the lse and the backward workspace of the largest chunk."""
    chunks = fa.fa_fwd_bwd_host_chunks(B, H, N, kv_len, dropout, chunk_heads)
    heads = max(cb * ch for _, cb, ch, _ in chunks)
    es = 4 if dt == fa.FA_FP32 else 2
    nb = (N + 127) // 128
    head = (r256(4 * B) if kv_len else 0) + (r256(nb * nb) if mask else 0)
    slot = 8 * r256(heads * N * d * es) + r256(heads * N * 4) + r256(fa.fa_bwd_workspace_size(1, heads, N, d))
    want = head + min(3, len(chunks)) * slot
    assert fa.fa_fwd_bwd_host_workspace_size(B, H, N, d, dt, mask, dropout, kv_len, chunk_heads) == want


def test_workspace_size_of_invalid_sizes_is_zero():
    ws = fa.fa_fwd_bwd_host_workspace_size
    assert ws(0, 1, 16, 64, fa.FA_BF16, None, 0.0, None, 0) == 0
    assert ws(1, 1, 16, 96, fa.FA_BF16, None, 0.0, None, 0) == 0
    assert ws(1, 1, 16, 64, 9, None, 0.0, None, 0) == 0
    assert ws(1, 1, 16, 64, fa.FA_BF16, None, 0.0, None, -1) == 0
    assert ws(1, 1, 0, 64, fa.FA_BF16, None, 0.0, None, 0) == 0


def _args(**kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, dO=FAKE, o=FAKE, lse=FAKE, dq=FAKE, dk=FAKE, dv=FAKE, B=1, H=2, N=16, d=64,
             scale=0.125, causal=0, block_mask=None, dropout_p=0.0, seed=0, dtype=fa.FA_BF16, kv_len=None,
             chunk_heads=0, workspace=FAKE, workspace_bytes=1 << 30, stream=None)
    a.update(kw)
    return a


@pytest.mark.parametrize("kw,expect", [
    (dict(q=None), -1), (dict(dO=None), -1), (dict(lse=None), -1), (dict(dv=None), -1),
    (dict(B=0), -1), (dict(N=-1), -1), (dict(chunk_heads=-2), -1), (dict(dropout_p=1.0), -1),
    (dict(d=96), -2), (dict(dtype=5), -2),
    (dict(workspace=None), -4), (dict(workspace_bytes=4096), -4), (dict(workspace=FAKE + 16), -4),
])
def test_argument_errors(kw, expect):
    """Refused on the host before any CUDA call."""
    assert fa.fa_fwd_bwd_host(**_args(**kw)) == expect


def test_zero_length_is_a_noop():
    assert fa.fa_fwd_bwd_host(**_args(N=0, q=None, workspace=None)) == 0


def test_binding_checks_host_tensors():
    """attention_fwd_bwd_host refuses device tensors and masks of the wrong
    type or size before calling the library."""
    torch = pytest.importorskip("torch")
    q = torch.zeros((1, 2, 130, 64), dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        fa.attention_fwd_bwd_host(q, q, q, q.float())  # dO of another dtype
    with pytest.raises(ValueError):
        fa.attention_fwd_bwd_host(q, q, q, q, kv_len=torch.tensor([130], dtype=torch.int64))
    with pytest.raises(ValueError):
        fa.attention_fwd_bwd_host(q, q, q, q, kv_len=torch.tensor([130, 1], dtype=torch.int32))
    with pytest.raises(ValueError):
        fa.attention_fwd_bwd_host(q, q, q, q, block_mask=torch.ones(3, dtype=torch.uint8))


def test_device_binding_checks_masks():
    """attention_fwd / attention_bwd refuse masks the kernels would misread
    (wrong dtype, size or device) before calling the library."""
    torch = pytest.importorskip("torch")
    q = torch.zeros((1, 1, 300, 64), dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        fa._check_masks(torch.ones(3, 3, dtype=torch.uint8), None, 1, 300, q.device)  # a CPU mask
    with pytest.raises(ValueError):
        fa._check_masks(None, torch.tensor([300], dtype=torch.int64), 1, 300, q.device)


@pytest.mark.parametrize("B,H,N", [(65535, 1, 128), (1, 65535, 64), (255, 257, 1)])
@pytest.mark.parametrize("kv_len", [None, FAKE])
def test_chunks_at_the_largest_head_counts(B, H, N, kv_len):
    """B * H up to 65535 (the kernels' limit): one head per chunk, and the
    library's own plan, still partition the heads; one more head is refused."""
    for chunk_heads in (1, 0):
        chunks = fa.fa_fwd_bwd_host_chunks(B, H, N, kv_len, 0.0, chunk_heads)
        _check_partition(B, H, chunks, kv_len is not None, False)
    with pytest.raises(fa.FaError):
        fa.fa_fwd_bwd_host_chunks(B * H + 1, 1, N, kv_len, 0.0, 0)
    assert fa.fa_fwd_bwd_host_workspace_size(B * H + 1, 1, N, 64, fa.FA_BF16, None, 0.0, kv_len, 0) == 0


def test_chunk_query_writes_at_most_max_chunks_records():
    """fa_fwd_bwd_host_chunks returns the full count but writes only the
    first max_chunks records of four ints, and accepts a NULL buffer."""
    import ctypes
    lib = fa.load_library()
    n = lib.fa_fwd_bwd_host_chunks(2, 3, 300, None, 0.0, 1, None, 0)
    assert n == 6
    buf = (ctypes.c_int * (4 * 4))(*([-7] * 16))
    assert lib.fa_fwd_bwd_host_chunks(2, 3, 300, None, 0.0, 1, buf, 2) == 6
    assert list(buf[:8]) == [0, 1, 1, 0, 1, 1, 1, 0]
    assert list(buf[8:]) == [-7] * 8
