"""Device-side failure detection without a GPU fault: a bounded wait that
runs out reports BA_ERR_DEVICE_TIMEOUT through the status word, and the
context stays usable for the next correct call."""

import numpy as np
import pytest
import torch

import oracle
from branch_attention_speculative_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def api():
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required for -m gpu tests")
    from branch_attention_speculative_gb300 import build as B
    B.build()
    from branch_attention_speculative_gb300 import api as A
    return A


def test_expired_wait_reports_timeout_and_context_survives(api):
    wl = W.small("ttt", [64], heads_q=2, heads_kv=1, head_dim=64, cp=2, depth=2)
    plan = api.Plan.from_workload(wl)
    ws = plan.workspace()
    plan.selftest_wait_timeout(ws, cycles=1 << 22)   # ~2 ms of waiting, then give up
    assert plan.check_device_status(ws) == -4        # BA_ERR_DEVICE_TIMEOUT
    assert plan.check_device_status(ws) == 0         # the check clears the word
    # the same context still computes correctly
    t = W.make_tensors(wl, device="cuda", gen_device="cpu")
    o, lse = plan.forward(t["q_b"], t["k_m"], t["v_m"], t["k_b"], t["v_b"], workspace=ws)
    assert plan.check_device_status(ws) == 0
    host = {k: v.float().cpu().double().numpy() for k, v in t.items()}
    ro, rl = oracle.attention.forward(wl, host)
    assert np.abs(o.float().cpu().double().numpy() - ro).max() < 2e-2
    assert np.abs(lse.cpu().double().numpy() - rl).max() < 1e-3


def test_bad_arguments_never_launch(api):
    wl = W.small("ttt", [64], heads_q=2, heads_kv=1, head_dim=64, cp=2, depth=2)
    plan = api.Plan.from_workload(wl)
    t = W.make_tensors(wl, device="cuda", gen_device="cpu")
    small_ws = torch.empty(256, dtype=torch.uint8, device="cuda")
    with pytest.raises(api.BaError) as e:
        plan.forward(t["q_b"], t["k_m"], t["v_m"], t["k_b"], t["v_b"], workspace=small_ws)
    assert e.value.code == -6
    with pytest.raises(ValueError):
        plan.forward(t["q_b"][:, :32], t["k_m"], t["v_m"], t["k_b"], t["v_b"])
