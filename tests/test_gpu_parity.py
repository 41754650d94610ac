"""GPU parity: the CUDA path through the C ABI against the CPU oracle on the
same seeded inputs."""

import numpy as np
import pytest
import torch

import oracle
from branch_attention_speculative_gb300 import workloads as W
from tests import gpu_support as S

pytestmark = pytest.mark.gpu


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


def _run(api, wl, tensors, bwd=True):
    plan = api.Plan.from_workload(wl)
    ws = plan.workspace()
    o, lse = plan.forward(tensors["q_b"], tensors["k_m"], tensors["v_m"], tensors.get("k_b"), tensors.get("v_b"),
                          workspace=ws)
    assert plan.check_device_status(ws) == 0
    g = None
    if bwd:
        g = plan.backward(tensors["q_b"], tensors["k_m"], tensors["v_m"], tensors.get("k_b"), tensors.get("v_b"),
                          o, lse, tensors["d_o"], workspace=ws)
        assert plan.check_device_status(ws) == 0
    torch.cuda.synchronize()
    return plan, o, lse, g


def _tensors(wl):
    t = W.make_tensors(wl, device="cuda", gen_device="cpu")
    if wl.family == "causal":
        t["k_b"] = t["v_b"] = None
    return t


def _full_compare(api, wl):
    t = _tensors(wl)
    plan, o, lse, g = _run(api, wl, t)
    host = {k: _np(v) for k, v in t.items() if v is not None}
    ro, rl = oracle.attention.forward(wl, host)
    rg = oracle.attention.backward(wl, host, ro, rl)
    S.check_o(_np(o), ro)
    S.check_lse(_np(lse), rl)
    names = ["dq_b", "dk_m", "dv_m"] + ([] if wl.family == "causal" else ["dk_b", "dv_b"])
    for n in names:
        S.check_grad(_np(g[n]), rg[n], n)


# ---------------------------------------------------------------- K1 pack


@pytest.mark.parametrize("wl", [W.config(2), W.small("block", [64, 128], cp=4, block=4, anchors_per_seq=9),
                                W.small("ttt", [16, 48], cp=2, depth=3)], ids=lambda w: w.name)
def test_zigzag_pack_matches_oracle_permutation_bit_exact(api, wl):
    plan = api.Plan.from_workload(wl)
    ws = plan.workspace()
    g = torch.Generator(device="cuda").manual_seed(7)
    perm = torch.as_tensor(oracle.zigzag.packed_token_order(wl.cu_seqlens, wl.cp), device="cuda")
    # main K/V: rows permuted by the token order
    x = torch.randn(wl.km_shape(), generator=g, device="cuda").to(torch.bfloat16)
    y = plan.zigzag_pack("main_kv", x, workspace=ws)
    assert torch.equal(y, x[perm])
    assert torch.equal(plan.zigzag_pack("main_kv", y, inverse=True, workspace=ws), x)
    # query-shaped: tokens (TTT) or anchors (block) permuted
    q = torch.randn(wl.q_shape(), generator=g, device="cuda").to(torch.bfloat16)
    yq = plan.zigzag_pack("query", q, workspace=ws)
    if wl.family == "block":
        ap = torch.as_tensor(oracle.zigzag.packed_anchor_order(wl.cu_seqlens, wl.cp, wl.anchors), device="cuda")
        assert torch.equal(yq, q[ap])
    else:
        assert torch.equal(yq, q[:, perm])
    assert torch.equal(plan.zigzag_pack("query", yq, inverse=True, workspace=ws), q)
    assert plan.check_device_status(ws) == 0


# ---------------------------------------------------------------- K4 merge


@pytest.mark.parametrize("d", [64, 128])
def test_lse_merge_matches_eq2(api, d):
    rng = np.random.default_rng(d)
    rows = 3001
    om = rng.standard_normal((rows, d)).astype(np.float32)
    ob = rng.standard_normal((rows, d)).astype(np.float32)
    lm = (rng.standard_normal(rows) * 5).astype(np.float32)
    lb = (rng.standard_normal(rows) * 5).astype(np.float32)
    lm[6::17] = 80.0             # far apart
    lb[6::17] = -60.0
    lm[::7] = -np.inf            # empty main part
    lb[3::11] = -np.inf          # empty branch part
    lm[5::13] = lb[5::13] = -np.inf  # both empty
    ro, rl = oracle.merge.lse_merge(om, lm, ob, lb)
    om_dev = om.copy()
    om_dev[np.isneginf(lm)] = np.nan  # an empty part's O must never be read
    T = lambda a: torch.as_tensor(a, device="cuda")
    o, l = api.lse_merge(T(om_dev), T(lm), T(ob), T(lb))
    o, l = _np(o), l.cpu().double().numpy()
    assert np.array_equal(np.isneginf(l), np.isneginf(rl))
    fin = np.isfinite(rl)
    assert np.abs(l[fin] - rl[fin]).max() < 1e-5
    # bf16 output: within one rounding of the fp64 merge
    assert np.abs(o - ro).max() <= 2.0 ** -8 * np.abs(ro).max() + 1e-6
    assert (o[~fin] == 0).all()


# ---------------------------------------------------------------- full fwd + bwd, small


SMALL = [
    W.small("ttt", [64], heads_q=2, heads_kv=1, head_dim=64, cp=1, depth=2, name="ttt_c1"),
    W.small("ttt", [200, 56, 320], heads_q=4, heads_kv=2, head_dim=64, cp=2, depth=3, seed=1, name="ttt_ragged_c2"),
    W.small("ttt", [264, 136], heads_q=8, heads_kv=2, head_dim=128, cp=4, depth=2, seed=2, name="ttt_d128_c4"),
    W.small("block", [256, 128], heads_q=4, heads_kv=1, head_dim=128, cp=2, block=16, anchors_per_seq=13, seed=3,
            name="block16_c2"),
    W.small("block", [96, 32, 160], heads_q=4, heads_kv=2, head_dim=64, cp=4, block=3, anchors_per_seq=7, seed=4,
            name="block3_ragged_c4"),
    W.small("causal", [136, 8, 256], heads_q=4, heads_kv=4, head_dim=64, cp=2, seed=5, name="causal_mha"),
    W.small("block", [64], heads_q=2, heads_kv=1, head_dim=64, cp=2, block=1, anchors_per_seq=1, seed=6,
            name="block_one_anchor"),
    # chunks of several whole 128-key / 128-query tiles plus a ragged
    # tail, at head_dim 128: every main key's dK/dV, including the unmasked
    # key tiles away from the diagonal, is checked against the full oracle
    W.small("ttt", [1280, 768], heads_q=8, heads_kv=2, head_dim=128, cp=2, depth=2, seed=7,
            name="ttt_d128_tiles_c2"),
    W.small("block", [1536, 512], heads_q=8, heads_kv=2, head_dim=128, cp=2, block=16, anchors_per_seq=40, seed=8,
            name="block16_d128_tiles_c2"),
    # the planner's limits on branch keys per query: block size 64, TTT depth 16
    W.small("block", [512, 256], heads_q=4, heads_kv=2, head_dim=64, cp=2, block=64, anchors_per_seq=5, seed=10,
            name="block64_c2"),
    W.small("ttt", [128, 64], heads_q=2, heads_kv=1, head_dim=128, cp=2, depth=16, seed=11, name="ttt_depth16"),
    W.small("causal", [384, 640], heads_q=4, heads_kv=2, head_dim=128, cp=2, seed=9, name="causal_d128_gqa"),
    # head_dim 128, one q head per kv head and an odd number of query streams
    W.small("ttt", [256, 96], heads_q=3, heads_kv=3, head_dim=128, cp=2, depth=3, seed=12, name="ttt_d128_odd_streams"),
]


@pytest.mark.parametrize("wl", SMALL, ids=lambda w: w.name)
def test_small_full_parity(api, wl):
    _full_compare(api, wl)


def test_config1_full_parity(api):
    _full_compare(api, W.config(1))


# ---------------------------------------------------------------- measured shapes, sampled


# Main-key gradient windows at the end of the last sequence: at the 256K shape
# one whole 128-key tile, whose attending query rows sit more than 2^31
# elements into q_b; at the 128K block shape four tiles, two clusters of the
# dK/dV kernel.
@pytest.mark.parametrize("k,n_units,window", [(2, 48, 64), (3, 32, 256), (4, 24, 512), (5, 24, 128)])
def test_config_sampled_parity(api, k, n_units, window):
    wl = W.config(k)
    t = W.make_tensors(wl, device="cuda")
    plan, o, lse, g = _run(api, wl, t)
    src = S.TorchSource(wl, t)
    units = S.sample_units(wl, n_units)
    res = oracle.attention.unit_eval(wl, src, units)
    of = o.reshape(-1, wl.heads_q, wl.head_dim)
    lf = lse.reshape(-1, wl.heads_q)
    dqf = g["dq_b"].reshape(-1, wl.heads_q, wl.head_dim)
    dkbf = g["dk_b"].reshape(-1, wl.heads_kv, wl.head_dim)
    dvbf = g["dv_b"].reshape(-1, wl.heads_kv, wl.head_dim)
    idx = lambda ids: torch.as_tensor(np.asarray(ids), device="cuda")
    ro = np.concatenate([e["o"] for e in res])
    rl = np.concatenate([e["lse"] for e in res])
    rdq = np.concatenate([e["dq"] for e in res])
    qids = np.concatenate([e["qids"] for e in res])
    assert len(qids) * wl.heads_q >= 4096
    S.check_o(_np(of.index_select(0, idx(qids))), ro)
    S.check_lse(lf.index_select(0, idx(qids)).cpu().double().numpy(), rl)
    S.check_grad(_np(dqf.index_select(0, idx(qids))), rdq, "dq_b")
    bids = np.concatenate([oracle.keysets.branch_keys_of_unit(wl, e["unit"]) for e in res])
    S.check_grad(_np(dkbf.index_select(0, idx(bids))), np.concatenate([e["dk_b"] for e in res]), "dk_b")
    S.check_grad(_np(dvbf.index_select(0, idx(bids))), np.concatenate([e["dv_b"] for e in res]), "dv_b")
    # main keys in the tail window of the last sequence, first and last kv head
    hi = int(wl.cu_seqlens[-1])
    lo = hi - window
    heads = sorted({0, wl.heads_kv - 1})
    rdk, rdv = oracle.attention.main_key_grads(wl, src, lo, hi, kv_heads=heads)
    S.check_grad(_np(g["dk_m"][lo:hi][:, heads]), rdk, "dk_m")
    S.check_grad(_np(g["dv_m"][lo:hi][:, heads]), rdv, "dv_m")
    # exact identities over the whole gradients
    inv = S.invariant_errors_torch(wl, t, g)
    assert max(inv.values()) <= S.INVARIANT_REL, inv
