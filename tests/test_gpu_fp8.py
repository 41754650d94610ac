"""The 8-bit main forward (ba_forward_fp8) against the fp64 oracle, with the
tolerances e4m3 arithmetic allows.

e4m3 keeps 3 mantissa bits: round to nearest errs by at most 2^-4 relative
(about 3.6% RMS).  Three roundings reach the output: q and k (the score
sc * <q, k> over d = 128 terms moves by about 0.05 in natural-log units), P
and v.  For softmax rows spread over many keys each error enters O as a
relative error of the same size, so O is off by about 5-7% RMS
(an e4m3 emulation of this kernel's arithmetic in fp64 gives 4.5-5.8% for 16 to
32768 keys per row); the largest single deviation is one rounding of the
largest |v| (about 4.5 * 2^-4 = 0.28).  lse carries the weighted mean of the
score errors: about 0.05 for a row with one key, falling with more keys.
Bars: O rel-RMS <= 0.1 and max-abs <= 0.35; lse max-abs <= 0.25 and RMS
<= 0.03."""

import numpy as np
import pytest
import torch

import oracle
from branch_attention_speculative_gb300 import workloads as W
from tests import gpu_support as S

pytestmark = pytest.mark.gpu

F8_O_REL_RMS, F8_O_MAX_ABS = 0.1, 0.35
F8_LSE_MAX_ABS, F8_LSE_RMS = 0.25, 0.03


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


def _check(o, ro, l, rl, what):
    d = np.abs(o - ro)
    rr = S.rel_rms(o, ro)
    assert rr <= F8_O_REL_RMS and d.max() <= F8_O_MAX_ABS, f"{what} o: rel-rms {rr:.3e} max-abs {d.max():.3e}"
    e = np.abs(l - rl)
    assert e.max() <= F8_LSE_MAX_ABS and np.sqrt((e ** 2).mean()) <= F8_LSE_RMS, \
        f"{what} lse: max-abs {e.max():.3e} rms {np.sqrt((e ** 2).mean()):.3e}"


SMALL = [
    W.small("ttt", [1024, 512], heads_q=8, heads_kv=2, head_dim=128, cp=2, depth=2, seed=11, name="ttt_f8_c2"),
    W.small("block", [1536, 512], heads_q=8, heads_kv=2, head_dim=128, cp=2, block=16, anchors_per_seq=40,
            seed=12, name="block16_f8_c2"),
    W.small("causal", [256, 768], heads_q=4, heads_kv=4, head_dim=128, cp=2, seed=13, name="causal_f8_c2"),
]


@pytest.mark.parametrize("wl", SMALL, ids=lambda w: w.name)
def test_fp8_forward_small_full(api, wl):
    t = W.make_tensors(wl, device="cuda", gen_device="cpu")
    if wl.family == "causal":
        t["k_b"] = t["v_b"] = None
    plan = api.Plan.from_workload(wl)
    ws = torch.empty(plan.workspace_bytes_fp8, dtype=torch.uint8, device="cuda")
    o, lse = plan.forward_fp8(t["q_b"], t["k_m"], t["v_m"], t.get("k_b"), t.get("v_b"), workspace=ws)
    assert plan.check_device_status(ws) == 0
    host = {k: _np(v) for k, v in t.items() if v is not None}
    ro, rl = oracle.attention.forward(wl, host)
    _check(_np(o), ro, lse.cpu().double().numpy(), rl, wl.name)


@pytest.mark.parametrize("k,n_units", [(3, 32), (4, 24), (5, 24)])
def test_fp8_forward_sampled(api, k, n_units):
    wl = W.config(k)
    t = W.make_tensors(wl, device="cuda")
    plan = api.Plan.from_workload(wl)
    ws = torch.empty(plan.workspace_bytes_fp8, dtype=torch.uint8, device="cuda")
    o, lse = plan.forward_fp8(t["q_b"], t["k_m"], t["v_m"], t["k_b"], t["v_b"], workspace=ws)
    assert plan.check_device_status(ws) == 0
    del ws
    src = S.TorchSource(wl, t)
    res = oracle.attention.unit_eval(wl, src, S.sample_units(wl, n_units), grads=False)
    qids = np.concatenate([e["qids"] for e in res])
    assert len(qids) * wl.heads_q >= 4096
    idx = torch.as_tensor(qids, device="cuda")
    og = _np(o.reshape(-1, wl.heads_q, wl.head_dim).index_select(0, idx))
    lg = lse.reshape(-1, wl.heads_q).index_select(0, idx).cpu().double().numpy()
    _check(og, np.concatenate([e["o"] for e in res]), lg, np.concatenate([e["lse"] for e in res]), wl.name)


@pytest.mark.parametrize("wl", [
    W.small("ttt", [200, 56], heads_q=2, heads_kv=1, head_dim=128, cp=2, depth=2),  # chunks of 50 and 14 tokens
    W.small("ttt", [256], heads_q=2, heads_kv=1, head_dim=64, cp=2, depth=2),       # head_dim 64
], ids=["unaligned_chunks", "head_dim_64"])
def test_fp8_rejects_what_it_does_not_cover(api, wl):
    plan = api.Plan.from_workload(wl)
    t = W.make_tensors(wl, device="cuda", gen_device="cpu")
    with pytest.raises(api.BaError) as e:
        plan.forward_fp8(t["q_b"], t["k_m"], t["v_m"], t["k_b"], t["v_b"])
    assert e.value.code == -2
