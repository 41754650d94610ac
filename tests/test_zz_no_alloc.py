"""ba_forward_noalloc: the forward for callers that cannot allocate device
memory where they run attention (e.g. a plugin inside another framework's
execution loop).  It must give the same results as ba_forward, call after
call, using only the library's static scratch array.  Collected last."""

import numpy as np
import pytest
import torch

from branch_attention_speculative_gb300 import workloads as W

pytestmark = pytest.mark.gpu

O_MAX_ABS, O_REL_RMS, LSE_MAX_ABS = 2e-2, 1e-2, 1e-3


@pytest.fixture(scope="module")
def api():
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required for -m gpu tests")
    from branch_attention_speculative_gb300 import build as B
    B.build()
    from branch_attention_speculative_gb300 import api as A
    return A


def _close(got_o, got_l, ref_o, ref_l):
    a = got_o.float().cpu().double().numpy()
    b = ref_o.float().cpu().double().numpy()
    assert np.abs(a - b).max() <= O_MAX_ABS
    assert np.sqrt(((a - b) ** 2).mean() / (b ** 2).mean()) <= O_REL_RMS
    assert np.abs(got_l.cpu().double().numpy() - ref_l.cpu().double().numpy()).max() <= LSE_MAX_ABS


@pytest.mark.parametrize("wl", [W.config(1),
                                W.small("block", [256, 128], heads_q=4, heads_kv=1, head_dim=128, cp=2, block=16,
                                        anchors_per_seq=13, seed=3, name="block16_c2")],
                         ids=lambda w: w.name)
def test_noalloc_forward_matches_forward_twice(api, wl):
    plan = api.Plan.from_workload(wl)
    assert plan.workspace_bytes <= 64 << 20
    t = W.make_tensors(wl, device="cuda", gen_device="cpu")
    ref_o, ref_l = plan.forward(t["q_b"], t["k_m"], t["v_m"], t["k_b"], t["v_b"])
    torch.cuda.synchronize()
    for _ in range(2):  # two calls in a row share the static scratch
        o = torch.full_like(t["q_b"], float("nan"))
        l = torch.full(t["q_b"].shape[:-1], float("nan"), dtype=torch.float32, device="cuda")
        plan.forward_noalloc(t["q_b"], t["k_m"], t["v_m"], t["k_b"], t["v_b"], o=o, lse=l)
        torch.cuda.synchronize()
        _close(o, l, ref_o, ref_l)


def test_noalloc_rejects_plans_beyond_the_static_scratch(api):
    wl = W.config(2)  # about 5 GB of workspace
    plan = api.Plan.from_workload(wl)
    assert plan.workspace_bytes > 64 << 20
    q = torch.empty(plan.q_shape(), dtype=torch.bfloat16, device="cuda")
    km = torch.empty(plan.km_shape(), dtype=torch.bfloat16, device="cuda")
    kb = torch.empty(plan.kb_shape(), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(api.BaError) as e:
        plan.forward_noalloc(q, km, km, kb, kb)
    assert e.value.code == -6
