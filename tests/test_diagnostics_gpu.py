"""The library's diagnostic entry points on the GPU: the events it records
around a call's main kernel (bench.py's kernel-level roofline) and its
exponential-throughput probe (bench.py's exponential roofline)."""
import pytest
import torch

import io_aware_exact_08_gb300 as fa

pytestmark = pytest.mark.gpu


def test_main_kernel_events_bracket_the_kernel(cuda_device):
    B, H, N, d = 1, 4, 2048, 128
    g = torch.Generator().manual_seed(1)
    q, k, v = (torch.randn(B, H, N, d, generator=g).to(torch.bfloat16).cuda() for _ in range(3))
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    call_a, call_b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for e in (start, stop):
        e.record()  # torch reads elapsed times only of events it has seen recorded
    fa.attention_fwd(q, k, v, causal=True)  # warm-up
    assert fa.fa_set_main_kernel_events(start.cuda_event, stop.cuda_event) == 0
    try:
        call_a.record()
        fa.attention_fwd(q, k, v, causal=True)
        call_b.record()
    finally:
        assert fa.fa_set_main_kernel_events(None, None) == 0
    torch.cuda.synchronize()
    kernel_ms = start.elapsed_time(stop)
    call_ms = call_a.elapsed_time(call_b)
    assert 0 < kernel_ms <= call_ms * 1.05
    # one event without the other is refused
    assert fa.fa_set_main_kernel_events(start.cuda_event, None) == -1


def test_ex2_probe_rate_is_plausible(cuda_device):
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    blocks, iters = sms * 4, 1024
    out = torch.empty(blocks * 512, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    assert fa.fa_ex2_probe(out.data_ptr(), blocks, iters, stream) == 0
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    assert fa.fa_ex2_probe(out.data_ptr(), blocks, iters, stream) == 0
    b.record()
    torch.cuda.synchronize()
    rate = blocks * 512 * iters * 8 / (a.elapsed_time(b) * 1e-3)
    per_clock_per_sm = rate / sms / 2.07e9  # at the GB300's maximum SM clock
    # the multifunction unit's documented order of magnitude: between 8 and 64 a clock per SM
    assert 8 <= per_clock_per_sm <= 64, per_clock_per_sm
    assert torch.isfinite(out).all()
    assert fa.fa_ex2_probe(out.data_ptr(), 0, iters, stream) == -1
