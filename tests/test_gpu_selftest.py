"""Failure detection on the GPU without a fault: a bounded wait that nothing
completes expires after about 2 s and reports ATTN_ERR_DEVICE_TIMEOUT through
dev_status; the context stays usable (a forward runs afterwards)."""
import time

import numpy as np
import pytest
import torch

import exact_attention_58_gb300 as ea
from exact_attention_58_gb300.workloads import make_inputs
from gpu_helpers import O_ATOL, f64, gpu_fwd, oracle_fwd

pytestmark = pytest.mark.gpu


def test_completed_wait_reports_nothing():
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ea.attn_selftest_wait(status, arrive=True)
    torch.cuda.synchronize()
    assert int(status.item()) == 0


def test_expired_wait_reports_timeout_and_the_context_survives():
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    t0 = time.monotonic()
    ea.attn_selftest_wait(status, arrive=False)
    torch.cuda.synchronize()
    elapsed = time.monotonic() - t0
    assert int(status.item()) == 6          # ATTN_ERR_DEVICE_TIMEOUT
    assert 1.0 < elapsed < 30.0
    inp = make_inputs(1, 1, 130, 64, gen_seed=1)
    o, _ = gpu_fwd(inp)
    O_ref, _ = oracle_fwd(inp)
    assert float(np.abs(f64(o) - O_ref).max()) <= O_ATOL
