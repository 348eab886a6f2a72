"""Device failure path, tested without faulting the GPU: a kernel's bounded
mbarrier wait on a barrier nothing arrives at gives up, the status word
reports FA_ERR_DEVICE_TIMEOUT with its site, the call returns normally and
the context keeps working."""
import numpy as np
import pytest
import torch

import io_aware_exact_08_gb300 as fa
from parity_utils import compare, gpu_fwd_bwd, oracle_fwd_bwd
from workloads import Workload, make_inputs

pytestmark = pytest.mark.gpu


def test_bounded_wait_reports_timeout_and_context_survives(cuda_device):
    stream = torch.cuda.current_stream().cuda_stream
    assert fa.fa_check_device_status(stream)[0] == 0
    assert fa.fa_test_wait_timeout(50_000_000, stream) == 0  # 50 ms limit
    st, site = fa.fa_check_device_status(stream)
    assert st == -5 and site == 900
    assert "TIMEOUT" in fa.fa_status_string(st)
    assert fa.fa_check_device_status(stream)[0] == 0  # cleared by the read
    # the context is still usable: a normal forward/backward matches the oracle
    inp = make_inputs(Workload("after", 0, B=1, H=2, N=200, d=64, dtype="bf16", causal=True), seed=3)
    compare(gpu_fwd_bwd(inp), oracle_fwd_bwd(inp), "bf16")
