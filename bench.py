"""Benchmark: exact attention forward + backward on one GB300 (or N replicas).

One step = one forward and one backward over one batch of the workload
(inputs resident in HBM), through the library's C ABI. Prints ONE JSON line.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                  [--impl fa|reference] [--no-cpu-baseline]

Default workload: long-context dense causal attention (B=2 H=16 N=8192
d=128, bf16), the largest configuration and one the N >= 4K throughput
target applies to; --workload selects any other. Metric: TFLOP/s with FLOPs = 4*B*H*N^2*d for the forward and
2.5x that for the backward, halved for causal and scaled by the block
density for block-sparse masks (the literal formula; key padding counts the
dense N^2). For N > 1 GPUs (torchrun), every rank runs the same workload on
its own GPU with no collective on the data path (independent heads/batches:
weak scaling); the step time is the max over ranks.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "attention fwd / fwd+bwd TFLOP/s at 1 GB300 and % of dense BF16 tensor peak"
UNIT = "TFLOP/s"
L2_BYTES = 129 * 1024 * 1024


# ---------------------------------------------------------------------------
# FLOP and byte models
# ---------------------------------------------------------------------------

def density_of(inp, w):
    if inp.get("block_mask") is None:
        return 1.0
    return float(inp["block_mask"].double().mean())


def flops(w, density=1.0):
    f = 4.0 * w.B * w.H * w.N * w.N * w.d
    if w.causal:
        f *= 0.5
    f *= density
    return f, 2.5 * f


def algorithmic_bytes(w):
    """Forward: read Q, K, V, write O (elements) + write LSE (fp32).
    Backward: read Q, K, V, O, dO, LSE; write dQ, dK, dV."""
    e = 2 if w.dtype in ("bf16", "fp16") else 4
    bhnd = w.B * w.H * w.N * w.d
    bhn = w.B * w.H * w.N
    return 4 * bhnd * e + 4 * bhn, 8 * bhnd * e + 8 * bhn


def visible_pairs(w, inp):
    """Number of unmasked (query, key) pairs of the workload: the
    exponentials the forward needs (the backward recomputes each once more)."""
    import numpy as np
    N = w.N
    kv = inp["kv_len"].numpy().astype(np.int64) if inp.get("kv_len") is not None else np.full(w.B, N)
    bm = inp["block_mask"].numpy().astype(bool) if inp.get("block_mask") is not None else None
    total = 0
    rows = np.arange(N)
    for b in range(w.B):
        L = int(min(max(kv[b], 0), N))
        if bm is None:
            per_row = np.minimum(rows + 1, L) if w.causal else np.full(N, L)
            total += int(per_row.sum())
            continue
        # block mask: per query block, count keys block by block
        nb = bm.shape[0]
        for ib in range(nb):
            r = rows[ib * 128:(ib + 1) * 128]
            for jb in np.nonzero(bm[ib])[0]:
                lo, hi = jb * 128, min((jb + 1) * 128, L)
                if hi <= lo:
                    continue
                if w.causal:
                    total += int(np.clip(np.minimum(r + 1, hi) - lo, 0, None).sum())
                else:
                    total += int(hi - lo) * len(r)
    return int(total) * w.H


def measure_ex2_rate(device):
    """Exponentials per second of the GPU's ex2.approx.f32 (the library's
    throughput probe, timed with CUDA events)."""
    import torch
    import io_aware_exact_08_gb300 as fa
    sms = torch.cuda.get_device_properties(device).multi_processor_count
    blocks, iters = sms * 4, 4096
    out = torch.empty(blocks * 512, dtype=torch.float32, device=device)
    stream = torch.cuda.current_stream(device)
    for _ in range(2):
        assert fa.fa_ex2_probe(out.data_ptr(), blocks, iters, stream.cuda_stream) == 0
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    assert fa.fa_ex2_probe(out.data_ptr(), blocks, iters, stream.cuda_stream) == 0
    b.record(stream)
    torch.cuda.synchronize(device)
    return blocks * 512 * iters * 8 / (a.elapsed_time(b) * 1e-3)


def bwd_main_bytes(w):
    """Algorithmic bytes of the backward's main kernel: read Q, K, V, dO,
    LSE and rowsum(dO o O); write dQ, dK, dV."""
    e = 2 if w.dtype in ("bf16", "fp16") else 4
    bhnd = w.B * w.H * w.N * w.d
    bhn = w.B * w.H * w.N
    return 7 * bhnd * e + 8 * bhn


def main_kernel_names(w, splits=1):
    """(forward, backward) main kernels of a workload's calls, as the events
    of fa_set_main_kernel_events bracket them."""
    if w.dtype not in ("bf16", "fp16"):
        return "fwd_simt_kernel", "bwd_simt_kernels"
    fwd = "fwd_d256_kernel" if w.d == 256 else "fwd_1t_kernel" if (w.d == 64 and splits == 1) else "fwd_pp_kernel"
    bwd = "bwd256_kernel (3 passes)" if w.d == 256 else "bwd_tc_kernel"
    return fwd, bwd


KERNEL_SOURCES = {
    "fwd_pp_kernel": ["fa_fwd_sm103.cu"],
    "fwd_d256_kernel": ["fa_fwd_sm103.cu"],
    "fwd_1t_kernel": ["fa_fwd1t_sm103.cu"],
    "fwd_fp8_kernel": ["fa_fwd_fp8_sm103.cu"],
    "bwd_tc_kernel": ["fa_bwd_sm103.cu"],
    "bwd256_kernel (3 passes)": ["fa_bwd256_sm103.cu"],
    "fwd_simt_kernel": ["fa_simt.cu"],
    "bwd_simt_kernels": ["fa_simt.cu"],
}
SHARED_HEADERS = ["fa_sm103.cuh", "fa_device.cuh", "fa_internal.h"]


def kernel_source_hash(kernel=None):
    """SHA-256 over the CUDA sources a kernel is built from (its own file and
    the shared device headers; every source file when kernel is None)."""
    import hashlib
    d = os.path.join(ROOT, "io_aware_exact_08_gb300", "csrc")
    if kernel is None:
        files = sorted(fn for fn in os.listdir(d) if fn.endswith((".cu", ".cuh", ".h")))
    else:
        files = sorted(KERNEL_SOURCES.get(kernel, []) + SHARED_HEADERS)
    h = hashlib.sha256()
    for fn in files:
        h.update(fn.encode())
        h.update(open(os.path.join(d, fn), "rb").read())
    return h.hexdigest()


def recorded_traffic(workload, kernel):
    """DRAM bytes (read + write) of one launch of `kernel` on `workload`, as
    ncu counted them in the capture recorded under profiles/, or None when
    there is no record or the kernel's sources have changed since."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    ent = rec.get("kernels", {}).get(workload, {}).get(kernel)
    if not ent or ent.get("source_sha256") != kernel_source_hash(kernel):
        return None
    return int(ent["dram_bytes"])


def traffic_key(w, splits=1):
    """Key of a (workload, dtype, split count) in the DRAM traffic record."""
    from workloads import WORKLOADS, headdim_workloads, sparse_workloads, splitkv_workloads, sweep_workloads
    base = {x.name: x for x in list(WORKLOADS.values()) + sweep_workloads() + splitkv_workloads() +
            headdim_workloads() + sparse_workloads()}.get(w.name)
    key = w.name
    if base is not None and base.dtype != w.dtype:
        key += f"/{w.dtype}"
    if splits > 1:
        key += f"/splits={splits}"
    return key


def workload_config(w, density, splits, ws):
    """The `config` object of a bench line: the workload and the step, the
    same for the library arm and the reference arm."""
    return {"workload": w.name, "B": w.B, "H": w.H, "N": w.N, "d": w.d, "dtype": w.dtype, "causal": w.causal,
            "dropout_p": w.dropout_p, "kv_len_range": w.kv_len_range, "block_density": round(density, 5),
            "scale": w.softmax_scale,
            "step": "fa_fwd + fa_bwd" if splits == 1 else f"fa_fwd_splitkv ({splits} splits) + fa_bwd",
            "l2": "flushed before every timed step", "parallelism": f"replicas x{ws}"}


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            pk = json.load(f)
        return dict(bf16=float(pk["bf16_tflops"]), bf16_sustained=float(pk.get("bf16_tflops_sustained", 0) or 0),
                    hbm=float(pk["hbm_gbs"]), source="measured")
    except Exception:
        return dict(bf16=1900.0, bf16_sustained=1700.0, hbm=6800.0, source="fallback")


# ---------------------------------------------------------------------------
# Clock sampling during the timed region
# ---------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu_index = gpu_index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu_index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        sm, mx, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for nm, val in zip(names, parts[5:9]):
                if val.lower() in ("active", "1"):
                    reasons.add(nm)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "samples": len(sm),
                "reasons": sorted(reasons)}


# ---------------------------------------------------------------------------
# Distributed helpers (torchrun); N == 1 runs without a process group.
# ---------------------------------------------------------------------------

def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(value, device=None):
    """Max of a float over all ranks (identity without a process group)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_tflops(flops_per_rank, ms_per_rank, world_size, device=None):
    """Whole-job throughput: the units every rank processed divided by the
    slowest rank's time (each rank runs the same workload: weak scaling)."""
    ms_max = max_over_ranks(ms_per_rank, device)
    return flops_per_rank * world_size / (ms_max * 1e-3) / 1e12, ms_max


def barrier(device=None):
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        if device is not None and device.type == "cuda":
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


# ---------------------------------------------------------------------------
# CPU baseline: the oracle, as it stands, on a bounded sample of heads
# ---------------------------------------------------------------------------

def cpu_model():
    """Model name of the host CPU (lscpu, else /proc/cpuinfo, else the ISA)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    import platform
    return platform.machine()


def head_sample(inp, w, n):
    """The first n heads (flat order b*H + h) of the inputs as a smaller
    problem the oracle can run on its own (heads are independent): the
    first n heads of batch 0 if n <= H, else the first ceil(n/H) whole
    batches. Returns (inputs, heads taken)."""
    if n <= w.H:
        nb, nh = 1, n
    else:
        nb, nh = min(w.B, -(-n // w.H)), w.H
    out = dict(inp)
    for key in ("q", "k", "v", "do", "q8", "k8", "v8"):
        if inp.get(key) is not None:
            out[key] = inp[key][:nb, :nh].contiguous()
    for key in ("descale_q", "descale_k", "descale_v"):
        if inp.get(key) is not None:
            out[key] = inp[key].reshape(w.B, w.H)[:nb, :nh].reshape(-1).contiguous()
    if inp.get("kv_len") is not None:
        out["kv_len"] = inp["kv_len"][:nb].contiguous()
    return out, nb * nh


def oracle_heads_for(w, inp, budget_s, backward=True):
    """How many whole heads of the workload the oracle runs in about
    budget_s seconds (at least one), from one timed head."""
    t1 = oracle_run(w, inp, [0], backward)
    return max(1, min(w.B * w.H, int(budget_s / max(t1, 1e-6))))


def oracle_run(w, inp, heads, backward=True):
    """Wall time of the fp64 oracle on the first len(heads) heads (forward,
    and backward), given only those heads' inputs. The dropout mask is drawn
    for the heads' own (b, h) indices, which the sample keeps."""
    import oracle
    sub, _ = head_sample(inp, w, len(heads))
    kw = dict(causal=w.causal, block_mask=sub["block_mask"], block=128, kv_len=sub["kv_len"],
              dropout_p=w.dropout_p, seed=sub["seed"])
    q, k, v, do = (sub[n] for n in ("q", "k", "v", "do"))
    t0 = time.perf_counter()
    oracle.attention_fwd(q, k, v, w.softmax_scale, **kw)
    if backward:
        oracle.attention_bwd(q, k, v, do, w.softmax_scale, **kw)
    return time.perf_counter() - t0


def oracle_sample(w, inp, budget_s=12.0, backward=True):
    """Times the fp64 oracle on whole heads of the workload (fwd+bwd)."""
    import oracle
    total_heads = w.B * w.H
    fwd_f, bwd_f = flops(w, density_of(inp, w))
    per_head = (fwd_f + (bwd_f if backward else 0.0)) / total_heads
    n = head_sample(inp, w, oracle_heads_for(w, inp, budget_s, backward))[1]
    t = oracle_run(w, inp, list(range(n)), backward)
    value = per_head * n / t / 1e12
    return {"value": value, "unit": UNIT, "cores": oracle.max_threads(), "cpu_model": cpu_model(),
            "kind": "oracle",
            "sample": f"{n} of {total_heads} heads, fp64 {'fwd+bwd' if backward else 'fwd'}, {t:.2f} s"}


# ---------------------------------------------------------------------------
# Our arm
# ---------------------------------------------------------------------------

def run_fa(args, w, ws, rank, device):
    import torch
    import io_aware_exact_08_gb300 as fa
    from workloads import make_inputs

    inp = make_inputs(w)
    dens = density_of(inp, w)
    fwd_f, bwd_f = flops(w, dens)
    fwd_b, bwd_b = algorithmic_bytes(w)
    dev = lambda t: None if t is None else t.to(device).contiguous()
    q, k, v, do = (dev(inp[n]) for n in ("q", "k", "v", "do"))
    bm, kl = dev(inp["block_mask"]), dev(inp["kv_len"])
    B, H, N, d = w.B, w.H, w.N, w.d
    dtype = {"bf16": fa.FA_BF16, "fp16": fa.FA_FP16, "fp32": fa.FA_FP32}[w.dtype]
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=device)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(q), torch.empty_like(q)
    wsb = fa.fa_bwd_workspace_size(B, H, N, d)
    work = torch.empty(wsb, dtype=torch.uint8, device=device)
    flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=device)
    stream = torch.cuda.current_stream(device)
    sh = stream.cuda_stream
    ptr = lambda t: None if t is None else t.data_ptr()
    scale, causal, p, seed = w.softmax_scale, int(w.causal), float(w.dropout_p), int(inp["seed"])

    splits = max(1, int(getattr(args, "splits", 1)))
    kv_ws = None
    if splits > 1:
        kv_wsb = fa.fa_fwd_splitkv_workspace_size(B, H, N, d, splits)
        kv_ws = torch.empty(kv_wsb, dtype=torch.uint8, device=device)

    def fwd():
        if kv_ws is not None:
            rc = fa.fa_fwd_splitkv(ptr(q), ptr(k), ptr(v), ptr(o), ptr(lse), B, H, N, d, scale, causal, ptr(bm), p,
                                   seed, dtype, ptr(kl), splits, kv_ws.data_ptr(), kv_ws.numel(), sh)
        else:
            rc = fa.fa_fwd(ptr(q), ptr(k), ptr(v), ptr(o), ptr(lse), B, H, N, d, scale, causal, ptr(bm), p, seed,
                           dtype, ptr(kl), sh)
        assert rc == 0, fa.fa_status_string(rc)

    def bwd():
        rc = fa.fa_bwd(ptr(q), ptr(k), ptr(v), ptr(o), ptr(lse), ptr(do), ptr(dq), ptr(dk), ptr(dv), B, H, N, d,
                       scale, causal, ptr(bm), p, seed, dtype, ptr(kl), ptr(work), wsb, sh)
        assert rc == 0, fa.fa_status_string(rc)

    for _ in range(args.warmup):
        fwd()
        bwd()
    torch.cuda.synchronize(device)
    st, site = fa.fa_check_device_status(sh)
    assert st == 0, f"device status {st} at site {site}"

    # timed region: K steps; L2 flushed before each step, outside the events
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True),
           torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    clocks = ClockSampler(device.index if device.index is not None else 0)
    clocks.start()
    time.sleep(0.3)
    barrier(device)
    torch.cuda.synchronize(device)
    launches0 = fa.fa_launch_count()
    for i in range(args.steps):
        flush.zero_()
        ev[i][0].record(stream)
        fwd()
        ev[i][1].record(stream)
        bwd()
        ev[i][2].record(stream)
    torch.cuda.synchronize(device)
    launches = fa.fa_launch_count() - launches0
    barrier(device)
    clk = clocks.stop()
    st, site = fa.fa_check_device_status(sh)
    assert st == 0, f"device status {st} at site {site}"
    fwd_ms = [a.elapsed_time(b) for a, b, c in ev]
    bwd_ms = [b.elapsed_time(c) for a, b, c in ev]
    step_ms = sum(f + g for f, g in zip(fwd_ms, bwd_ms)) / args.steps
    value, step_ms_max = whole_job_tflops(fwd_f + bwd_f, step_ms, ws, device)
    fwd_avg = max_over_ranks(sum(fwd_ms) / args.steps, device)
    bwd_avg = max_over_ranks(sum(bwd_ms) / args.steps, device)

    # end to end through the public API with host buffers (pinned): every
    # step copies Q, K, V, dO (and the masks) in and O, LSE, dQ, dK, dV out.
    # fa_fwd_bwd_host overlaps those copies with the kernels chunk by chunk;
    # the split-KV forward has no host entry point, so with --splits the
    # step copies around fa_fwd_splitkv + fa_bwd one after the other.
    host_in = [inp[n].pin_memory() for n in ("q", "k", "v", "do")]
    host_out = [torch.empty(q.shape, dtype=q.dtype).pin_memory() for _ in range(4)]
    host_lse = torch.empty((B, H, N), dtype=torch.float32).pin_memory()
    host_bm = None if inp["block_mask"] is None else inp["block_mask"].contiguous()
    host_kl = None if inp["kv_len"] is None else inp["kv_len"].contiguous()
    h2d = sum(t.numel() * t.element_size() for t in host_in)
    d2h = sum(t.numel() * t.element_size() for t in host_out)
    chunk_heads = int(getattr(args, "chunk_heads", 0))
    if kv_ws is None:
        h2d += sum(t.numel() * t.element_size() for t in (host_bm, host_kl) if t is not None)
        d2h += host_lse.numel() * host_lse.element_size()
        hws_b = fa.fa_fwd_bwd_host_workspace_size(B, H, N, d, dtype, ptr(host_bm), p, ptr(host_kl), chunk_heads)
        hws = torch.empty(hws_b, dtype=torch.uint8, device=device)

        def e2e_step():
            rc = fa.fa_fwd_bwd_host(*(t.data_ptr() for t in host_in), ptr(host_out[0]), ptr(host_lse),
                                    *(t.data_ptr() for t in host_out[1:]), B, H, N, d, scale, causal, ptr(host_bm),
                                    p, seed, dtype, ptr(host_kl), chunk_heads, hws.data_ptr(), hws_b, sh)
            assert rc == 0, fa.fa_status_string(rc)
    else:
        def e2e_step():
            for dst, src in zip((q, k, v, do), host_in):
                dst.copy_(src, non_blocking=True)
            fwd()
            bwd()
            for dst, src in zip(host_out, (o, dq, dk, dv)):
                dst.copy_(src, non_blocking=True)
    e_start, e_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e2e_steps = max(1, min(args.steps, 10))
    e2e_step()  # first call: the library's copy streams, pinned pages
    barrier(device)
    torch.cuda.synchronize(device)
    e_start.record(stream)
    for _ in range(e2e_steps):
        e2e_step()
    e_end.record(stream)
    torch.cuda.synchronize(device)
    e2e_ms = max_over_ranks(e_start.elapsed_time(e_end) / e2e_steps, device)

    # the main kernel of each call, timed on its own in a second pass of K
    # steps (same L2 flush): the library records the events right around its
    # launch (fa_set_main_kernel_events), so the backward's preprocess and dQ
    # conversion are outside them
    kev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    for e in sum(kev, []):
        e.record(stream)  # torch reads elapsed times only of events it has seen recorded
    barrier(device)
    torch.cuda.synchronize(device)
    for i in range(args.steps):
        flush.zero_()
        fa.fa_set_main_kernel_events(kev[i][0].cuda_event, kev[i][1].cuda_event)
        fwd()
        fa.fa_set_main_kernel_events(kev[i][2].cuda_event, kev[i][3].cuda_event)
        bwd()
        fa.fa_set_main_kernel_events(None, None)
    torch.cuda.synchronize(device)
    fwd_k_ms = max_over_ranks(sum(e[0].elapsed_time(e[1]) for e in kev) / args.steps, device)
    bwd_k_ms = max_over_ranks(sum(e[2].elapsed_time(e[3]) for e in kev) / args.steps, device)

    total_f = (fwd_f + bwd_f) * ws
    e2e_value = total_f / (e2e_ms * 1e-3) / 1e12
    fwd_tflops = fwd_f * ws / (fwd_avg * 1e-3) / 1e12
    bwd_tflops = bwd_f * ws / (bwd_avg * 1e-3) / 1e12
    peaks = load_peaks()
    # dominant kernel of the step: the forward kernel, or the backward's main
    # kernel (all of the backward's FLOPs; its algorithmic bytes are those of
    # the call minus the O read that the preprocess does)
    names = main_kernel_names(w, splits)
    fwd_is_dom = fwd_k_ms > bwd_k_ms
    dom_name = names[0] if fwd_is_dom else names[1]
    dom_ms = fwd_k_ms if fwd_is_dom else bwd_k_ms
    dom_f = fwd_f if fwd_is_dom else bwd_f
    dom_b = fwd_b if fwd_is_dom else bwd_main_bytes(w)
    tensor_ach = dom_f / (dom_ms * 1e-3) / 1e12
    hbm_ach = dom_b / (dom_ms * 1e-3) / 1e9
    # fp16 and bf16 share the dense tensor rate (2.25 PFLOP/s nominal each), so
    # an fp16 contraction takes the measured bf16 peak times 1
    sixteen = w.dtype in ("bf16", "fp16")
    tensor_frac = tensor_ach / peaks["bf16"]
    hbm_frac = hbm_ach / peaks["hbm"]
    if sixteen and tensor_frac >= hbm_frac:
        roof = {"bound": "tensor", "achieved": round(tensor_ach, 2), "peak": peaks["bf16"], "unit": "TFLOP/s",
                "frac": round(tensor_frac, 4)}
    elif sixteen:
        roof = {"bound": "hbm", "achieved": round(hbm_ach, 1), "peak": peaks["hbm"], "unit": "GB/s",
                "frac": round(hbm_frac, 4)}
    else:
        roof = {"bound": "alu", "achieved": round(tensor_ach, 3), "peak": None, "unit": "TFLOP/s", "frac": None}
    roof.update({"kernel": dom_name,
                 "traffic": recorded_traffic(traffic_key(w, splits), dom_name),
                 "peak_source": peaks["source"] + " (burst)" + (", bf16 peak x 1 for fp16" if w.dtype == "fp16" else ""),
                 "tensor_frac": round(tensor_frac, 4), "hbm_frac": round(hbm_frac, 4),
                 "algorithmic_flops": dom_f, "algorithmic_bytes": dom_b, "kernel_avg_ms": round(dom_ms, 4),
                 "kernel_ms": {names[0]: round(fwd_k_ms, 4), names[1]: round(bwd_k_ms, 4)}})

    # secondary roofline: the exponentials (one per visible score in the
    # forward, one more in the backward's recompute) against the measured
    # ex2 throughput
    ex2_rate = measure_ex2_rate(device)
    exps = 2 * visible_pairs(w, inp)
    exp_ms = exps / ex2_rate * 1e3
    mufu = {"exp_per_step": exps, "ex2_per_s": round(ex2_rate, 1), "bound_ms": round(exp_ms, 5),
            "frac_of_step": round(exp_ms / step_ms_max, 4),
            "fwd_frac": round(exp_ms / 2 / fwd_avg, 4), "bwd_frac": round(exp_ms / 2 / bwd_avg, 4)}

    line = {
        "metric": METRIC, "value": round(value, 3), "unit": UNIT, "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(step_ms_max, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": w.dtype, "data": "synthetic",
        "config": workload_config(w, dens, splits, ws),
        "fwd_tflops": round(fwd_tflops, 3), "bwd_tflops": round(bwd_tflops, 3),
        "fwd_ms": round(fwd_avg, 4), "bwd_ms": round(bwd_avg, 4),
        "frac_of_bf16_peak": round(value / ws / peaks["bf16"], 4) if sixteen else None,
        "fwd_frac_of_bf16_peak": round(fwd_tflops / ws / peaks["bf16"], 4) if sixteen else None,
        "roofline": roof,
        "exp_roofline": mufu,
        "e2e": {"value": round(e2e_value, 3), "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": round(e2e_ms, 4),
                "call": "fa_fwd_bwd_host" if kv_ws is None else "copies + fa_fwd_splitkv + fa_bwd"},
        "gpu_launches": int(launches),
        "clocks": clk,
    }
    if rank == 0 and not args.no_cpu_baseline and ws == 1:
        line["cpu_baseline"] = oracle_sample(w, inp, budget_s=args.cpu_budget)
    return line


def oracle_run_fp8(inp, w, heads):
    """Wall time of the oracle's FP8 forward on the first len(heads) heads."""
    import oracle
    sub, _ = head_sample(inp, w, len(heads))
    t0 = time.perf_counter()
    oracle.attention_fwd_fp8(sub["q8"], sub["k8"], sub["v8"], sub["descale_q"], sub["descale_k"], sub["descale_v"],
                             w.softmax_scale, causal=w.causal, block_mask=sub["block_mask"], block=128,
                             kv_len=sub["kv_len"])
    return time.perf_counter() - t0


def fp8_config(w, density, ws):
    cfg = workload_config(w, density, 1, ws)
    cfg.update({"dtype": "e4m3", "step": "fa_fwd_fp8 (forward only; E4M3 Q, K, V with per-head factors, bf16 O)"})
    return cfg


def run_fa_fp8(args, w, ws, rank, device):
    """The E4M3 forward alone: one step = one fa_fwd_fp8 call over the
    workload (inputs resident in HBM), FLOPs = the forward's 4 B H N^2 d
    (halved for causal, times the block density)."""
    import torch
    import io_aware_exact_08_gb300 as fa
    from workloads import make_fp8_inputs

    inp = make_fp8_inputs(w)
    dens = density_of(inp, w)
    fwd_f, _ = flops(w, dens)
    dev = lambda t: None if t is None else t.to(device).contiguous()
    q8, k8, vt8 = dev(inp["q8"]), dev(inp["k8"]), dev(inp["vt8"])
    dsq, dsk, dsv = dev(inp["descale_q"]), dev(inp["descale_k"]), dev(inp["descale_v"])
    bm, kl = dev(inp["block_mask"]), dev(inp["kv_len"])
    B, H, N, d = w.B, w.H, w.N, w.d
    o = torch.empty((B, H, N, d), dtype=torch.bfloat16, device=device)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=device)
    flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=device)
    stream = torch.cuda.current_stream(device)
    sh = stream.cuda_stream
    ptr = lambda t: None if t is None else t.data_ptr()

    def fwd():
        rc = fa.fa_fwd_fp8(ptr(q8), ptr(k8), ptr(vt8), ptr(dsq), ptr(dsk), ptr(dsv), ptr(o), ptr(lse), B, H, N, d,
                           w.softmax_scale, int(w.causal), ptr(bm), ptr(kl), sh)
        assert rc == 0, fa.fa_status_string(rc)

    for _ in range(args.warmup):
        fwd()
    torch.cuda.synchronize(device)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    clocks = ClockSampler(device.index if device.index is not None else 0)
    clocks.start()
    time.sleep(0.3)
    barrier(device)
    torch.cuda.synchronize(device)
    launches0 = fa.fa_launch_count()
    for i in range(args.steps):
        flush.zero_()
        ev[i][0].record(stream)
        fwd()
        ev[i][1].record(stream)
    torch.cuda.synchronize(device)
    launches = fa.fa_launch_count() - launches0
    barrier(device)
    clk = clocks.stop()
    st, site = fa.fa_check_device_status(sh)
    assert st == 0, f"device status {st} at site {site}"
    step_ms = sum(a.elapsed_time(b) for a, b in ev) / args.steps
    value, step_ms_max = whole_job_tflops(fwd_f, step_ms, ws, device)

    host_in = [inp[n].pin_memory() for n in ("q8", "k8", "vt8")]
    host_out = torch.empty(o.shape, dtype=o.dtype).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in host_in)
    d2h = host_out.numel() * host_out.element_size()
    e_start, e_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e2e_steps = max(1, min(args.steps, 10))
    barrier(device)
    torch.cuda.synchronize(device)
    e_start.record(stream)
    for _ in range(e2e_steps):
        for dst, src in zip((q8, k8, vt8), host_in):
            dst.copy_(src, non_blocking=True)
        fwd()
        host_out.copy_(o, non_blocking=True)
    e_end.record(stream)
    torch.cuda.synchronize(device)
    e2e_ms = max_over_ranks(e_start.elapsed_time(e_end) / e2e_steps, device)

    peaks = load_peaks()
    # E4M3 dense tensor rate is twice the bf16 rate (4.5 vs 2.25 PFLOP/s
    # nominal): the measured bf16 peak times 2
    peak = 2.0 * peaks["bf16"]
    ach = value / ws
    e = 1
    bhnd = B * H * N * d
    alg_bytes = 3 * bhnd * e + 2 * bhnd + 4 * B * H * N
    roof = {"bound": "tensor", "achieved": round(ach, 2), "peak": round(peak, 1), "unit": "TFLOP/s",
            "frac": round(ach / peak, 4), "kernel": "fwd_fp8_kernel",
            "traffic": recorded_traffic(w.name + "/fp8", "fwd_fp8_kernel"),
            "peak_source": peaks["source"] + " (burst) bf16 peak x 2 for E4M3",
            "algorithmic_flops": fwd_f, "algorithmic_bytes": alg_bytes, "kernel_avg_ms": round(step_ms_max, 4)}
    line = {
        "metric": METRIC, "value": round(value, 3), "unit": UNIT, "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(step_ms_max, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "e4m3", "data": "synthetic",
        "config": fp8_config(w, dens, ws),
        "fwd_tflops": round(value, 3), "fwd_ms": round(step_ms_max, 4),
        "frac_of_bf16_peak": round(ach / peaks["bf16"], 4),
        "roofline": roof,
        "e2e": {"value": round(fwd_f * ws / (e2e_ms * 1e-3) / 1e12, 3), "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
        "gpu_launches": int(launches),
        "clocks": clk,
    }
    if rank == 0 and not args.no_cpu_baseline and ws == 1:
        import oracle
        t1 = oracle_run_fp8(inp, w, [0])
        n = head_sample(inp, w, max(1, min(B * H, int(args.cpu_budget / max(t1, 1e-6)))))[1]
        t = oracle_run_fp8(inp, w, list(range(n))) if n > 1 else t1
        line["cpu_baseline"] = {"value": fwd_f / (B * H) * n / t / 1e12, "unit": UNIT, "cores": oracle.max_threads(),
                                "cpu_model": cpu_model(), "kind": "oracle",
                                "sample": f"{n} of {B * H} heads, fp64 forward on the dequantised inputs, {t:.2f} s"}
    return line


def run_reference_fp8(args, w, ws, rank):
    """The oracle's FP8 forward (fp64 on the dequantised inputs) as the
    reference arm, on a fixed sample of whole heads per step."""
    from workloads import make_fp8_inputs
    if rank != 0:
        return None
    import oracle
    inp = make_fp8_inputs(w)
    dens = density_of(inp, w)
    fwd_f, _ = flops(w, dens)
    total = w.B * w.H
    t1 = oracle_run_fp8(inp, w, [0])
    n = head_sample(inp, w, max(1, min(total, int(args.cpu_budget / max(1, args.steps) / max(t1, 1e-6)))))[1]
    heads = list(range(n))
    for _ in range(args.warmup):
        oracle_run_fp8(inp, w, [0])
    times = [oracle_run_fp8(inp, w, heads) for _ in range(args.steps)]
    step_s = sum(times) / len(times)
    value = fwd_f * n / total / step_s / 1e12
    sample = f"{n} of {total} heads per step, fp64 forward on the dequantised E4M3 inputs"
    cfg = fp8_config(w, dens, ws)
    cfg["sample"] = sample
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(step_s * 1e3, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic", "config": cfg,
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": oracle.max_threads(), "cpu_model": cpu_model(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def run_reference(args, w, ws, rank):
    """The oracle (fp64, host cores) as the reference arm: each step runs it
    on the same fixed sample of whole heads of the workload, and the step's
    wall time is measured (nothing is extrapolated)."""
    from workloads import make_inputs
    if rank != 0:
        return None
    import oracle
    inp = make_inputs(w)
    dens = density_of(inp, w)
    fwd_f, bwd_f = flops(w, dens)
    total_heads = w.B * w.H
    # sample size: whole heads filling about cpu_budget / steps seconds per step
    n = head_sample(inp, w, oracle_heads_for(w, inp, args.cpu_budget / max(1, args.steps)))[1]
    heads = list(range(n))
    for _ in range(args.warmup):
        oracle_run(w, inp, [0])
    times = [oracle_run(w, inp, heads) for _ in range(args.steps)]
    step_s = sum(times) / len(times)
    sample_f = (fwd_f + bwd_f) * n / total_heads
    value = sample_f / step_s / 1e12
    sample = f"{n} of {total_heads} heads per step, fp64 fwd+bwd"
    cfg = workload_config(w, dens, max(1, int(getattr(args, "splits", 1))), ws)
    cfg["sample"] = sample
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(step_s * 1e3, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": cfg,
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": oracle.max_threads(), "cpu_model": cpu_model(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="long_causal")
    ap.add_argument("--impl", default="fa", choices=["fa", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=12.0)
    ap.add_argument("--dtype", choices=["bf16", "fp16", "fp8"], default=None,
                    help="run a 16-bit workload with this input type instead of its own; fp8 times the "
                         "E4M3 forward (fa_fwd_fp8, head dim 128) alone")
    ap.add_argument("--splits", type=int, default=1,
                    help="forward through fa_fwd_splitkv with this many key-tile ranges per query-tile pair")
    ap.add_argument("--chunk-heads", type=int, default=0,
                    help="heads per chunk of the end-to-end step on host buffers (fa_fwd_bwd_host); 0 lets "
                         "the library choose")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    from workloads import WORKLOADS, headdim_workloads, sparse_workloads, splitkv_workloads, sweep_workloads
    table = dict(WORKLOADS)
    table.update({w.name: w for w in sweep_workloads() + splitkv_workloads() + headdim_workloads() +
                  sparse_workloads()})
    w = table[args.workload]
    fp8 = args.dtype == "fp8"
    if args.dtype is not None:
        if w.dtype not in ("bf16", "fp16"):
            ap.error("--dtype applies to the 16-bit workloads only")
        if fp8:
            if w.d != 128 or w.dropout_p > 0 or args.splits > 1:
                ap.error("--dtype fp8 needs a head-dim-128 workload without dropout or splits")
        else:
            w = w.with_(dtype=args.dtype)
    ws, rank, local = dist_env()

    if args.impl == "reference":
        line = run_reference_fp8(args, w, ws, rank) if fp8 else run_reference(args, w, ws, rank)
        if line is not None:
            print(json.dumps(line), flush=True)
        return 0

    import torch
    if ws > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    device = torch.device("cuda", local if ws > 1 else 0)
    torch.cuda.set_device(device)
    import io_aware_exact_08_gb300 as fa
    fa.load_library()
    line = run_fa_fp8(args, w, ws, rank, device) if fp8 else run_fa(args, w, ws, rank, device)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
