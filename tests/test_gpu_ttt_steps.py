"""EAGLE-3 TTT one step at a time through ba_forward_step / ba_backward_step:
each step alone matches the oracle element by element, reads no branch key
slot above its own, and the steps together reproduce the all-steps call."""

import numpy as np
import pytest
import torch

import oracle
from branch_attention_speculative_gb300 import workloads as W
from tests import gpu_support as S

pytestmark = pytest.mark.gpu

CASES = [
    W.config(1),
    W.small("ttt", [1280, 768], heads_q=8, heads_kv=2, head_dim=128, cp=2, depth=3, seed=7, name="ttt_d128_steps"),
]


@pytest.fixture(scope="module")
def api():
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required for -m gpu tests")
    from branch_attention_speculative_gb300 import build as B
    B.build()
    from branch_attention_speculative_gb300 import api as A
    return A


def _np(t):
    return t.float().cpu().double().numpy()


@pytest.mark.parametrize("wl", CASES, ids=lambda w: w.name)
def test_steps_match_oracle_and_all_steps_call(api, wl):
    D = wl.depth
    t = W.make_tensors(wl, device="cuda", gen_device="cpu")
    plan = api.Plan.from_workload(wl)
    ws = plan.workspace()
    # all steps at once
    o_all, l_all = plan.forward(t["q_b"], t["k_m"], t["v_m"], t["k_b"], t["v_b"], workspace=ws)
    g_all = plan.backward(t["q_b"], t["k_m"], t["v_m"], t["k_b"], t["v_b"], o_all, l_all, t["d_o"], workspace=ws)
    assert plan.check_device_status(ws) == 0
    host = {k: _np(v) for k, v in t.items()}
    ro, rl = oracle.attention.forward(wl, host)
    rg = oracle.attention.backward(wl, host, ro, rl)

    # forward, step by step; the branch slots above the step hold NaN, as if
    # the later steps' keys and values did not exist yet
    o_s, l_s = [], []
    for s in range(D):
        kb = t["k_b"].clone()
        vb = t["v_b"].clone()
        kb[s + 1:] = float("nan")
        vb[s + 1:] = float("nan")
        o, l = plan.forward_step(s, t["q_b"][s], t["k_m"], t["v_m"], kb, vb, workspace=ws)
        assert plan.check_device_status(ws) == 0
        torch.cuda.synchronize()
        assert torch.equal(o, o_all[s]) and torch.equal(l, l_all[s]), f"step {s} differs from the all-steps call"
        S.check_o(_np(o), ro[s], f"o step {s}")
        S.check_lse(l.cpu().double().numpy(), rl[s], f"lse step {s}")
        o_s.append(o)
        l_s.append(l)

    # backward, last step first, key gradients accumulated in fp32
    acc = {"dk_m": torch.zeros(plan.km_shape(), dtype=torch.float32, device="cuda"),
           "dv_m": torch.zeros(plan.km_shape(), dtype=torch.float32, device="cuda"),
           "dk_b": torch.zeros(plan.kb_shape(), dtype=torch.float32, device="cuda"),
           "dv_b": torch.zeros(plan.kb_shape(), dtype=torch.float32, device="cuda")}
    for s in reversed(range(D)):
        kb = t["k_b"].clone()
        vb = t["v_b"].clone()
        kb[s + 1:] = float("nan")
        vb[s + 1:] = float("nan")
        before_b = acc["dk_b"][s + 1:].clone()
        dq = plan.backward_step(s, t["q_b"][s], t["k_m"], t["v_m"], kb, vb, o_s[s], l_s[s], t["d_o"][s], acc,
                                workspace=ws)
        assert plan.check_device_status(ws) == 0
        torch.cuda.synchronize()
        assert torch.equal(acc["dk_b"][s + 1:], before_b), "a step touched branch slots above its own"
        assert torch.equal(dq, g_all["dq_b"][s]), f"dq of step {s} differs from the all-steps call"
        S.check_grad(_np(dq), rg["dq_b"][s], f"dq step {s}")
    for n, name in (("dk_m", "dk_m"), ("dv_m", "dv_m"), ("dk_b", "dk_b"), ("dv_b", "dv_b")):
        got = acc[n].cpu().double().numpy()
        S.check_grad(got, rg[name], f"{n} (accumulated over steps)")
        # the all-steps call rounds the same sums to bf16 once
        allb = _np(g_all[name])
        assert np.abs(got - allb).max() <= 2.0 ** -7 * np.abs(allb).max() + 1e-6, n


def test_step_arguments_are_checked(api):
    wl = W.config(1)
    plan = api.Plan.from_workload(wl)
    t = W.make_tensors(wl, device="cuda", gen_device="cpu")
    for bad in (-1, wl.depth):
        with pytest.raises(api.BaError) as e:
            plan.forward_step(bad, t["q_b"][0], t["k_m"], t["v_m"], t["k_b"], t["v_b"])
        assert e.value.code == -1
    blk = api.Plan.from_workload(W.small("block", [64], heads_q=2, heads_kv=1, head_dim=64, cp=2, block=2,
                                         anchors_per_seq=3))
    with pytest.raises(ValueError):
        blk.forward_step(0, t["q_b"][0], t["k_m"], t["v_m"], t["k_b"], t["v_b"])
