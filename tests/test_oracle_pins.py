"""Pins of the CPU oracle against the pages' definitions, closed forms,
library routines and hand-worked fixtures (no GPU)."""

import math
import os

import numpy as np
import pytest
import torch

import oracle
from branch_attention_speculative_gb300 import workloads as W
from tests import oracle_pins as P

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _small_cases():
    return [
        W.small("ttt", [8], heads_q=2, heads_kv=1, head_dim=16, cp=2, depth=3),
        W.small("ttt", [8, 12], heads_q=4, heads_kv=2, head_dim=16, cp=2, depth=2, seed=1),
        W.small("block", [16, 8], heads_q=4, heads_kv=2, head_dim=16, cp=2, block=3,
                anchors_per_seq=4, seed=2),
        W.small("causal", [12, 4], heads_q=2, heads_kv=1, head_dim=16, cp=2, seed=3),
    ]


@pytest.mark.parametrize("wl", _small_cases(), ids=lambda w: w.name)
def test_uniform_attention_reveals_key_sets(wl):
    # q = 0: l = log|K(i)| exactly and O = indicator(K(i)) / |K(i)|
    assert P.uniform_keyset_error(wl) < 1e-13


@pytest.mark.parametrize("wl", _small_cases(), ids=lambda w: w.name)
def test_matches_torch_sdpa_with_loop_built_mask(wl):
    assert P.sdpa_error(wl) < 1e-12


@pytest.mark.parametrize("wl", _small_cases(), ids=lambda w: w.name)
def test_gradients_match_finite_differences(wl):
    assert P.fd_error(wl) < 1e-6


@pytest.mark.parametrize("wl", _small_cases(), ids=lambda w: w.name)
def test_gradient_invariants_hold(wl):
    rng = np.random.default_rng(5)
    t = P.rand_inputs(wl, rng)
    g = oracle.attention.backward(wl, t)
    e = P.invariant_errors(wl, g, t)
    assert max(e.values()) < 1e-12, e


@pytest.mark.parametrize("wl", _small_cases(), ids=lambda w: w.name)
def test_probability_rows_sum_to_one(wl):
    rng = np.random.default_rng(7)
    t = P.rand_inputs(wl, rng)
    _, lse = oracle.attention.forward(wl, t)
    q = t["q_b"].reshape(-1, wl.heads_q, wl.head_dim)
    lse = lse.reshape(-1, wl.heads_q)
    kb = t["k_b"].reshape(-1, wl.heads_kv, wl.head_dim)
    G = wl.heads_q // wl.heads_kv
    for s in range(wl.num_seqs):
        qids = oracle.keysets.queries_of_seq(wl, s)
        a, b = int(wl.cu_seqlens[s]), int(wl.cu_seqlens[s + 1])
        bids = oracle.keysets.branch_keys_of_seq(wl, s)
        mask = np.concatenate([oracle.keysets.main_mask(wl, qids, np.arange(a, b)),
                               oracle.keysets.branch_mask(wl, qids, bids)], axis=1)
        for h in range(wl.heads_q):
            K = np.concatenate([t["k_m"][a:b, h // G], kb[bids, h // G]], axis=0)
            p = oracle.attention.masked_attention_probs(q[qids, h], K, mask, wl.scale, lse[qids, h])
            assert np.abs(p.sum(1) - 1.0).max() < 1e-12


@pytest.mark.parametrize("wl", _small_cases(), ids=lambda w: w.name)
def test_key_count_closed_form_matches_mask(wl):
    for s in range(wl.num_seqs):
        qids = oracle.keysets.queries_of_seq(wl, s)
        a, b = int(wl.cu_seqlens[s]), int(wl.cu_seqlens[s + 1])
        bids = oracle.keysets.branch_keys_of_seq(wl, s)
        n = oracle.keysets.main_mask(wl, qids, np.arange(a, b)).sum(1) + \
            oracle.keysets.branch_mask(wl, qids, bids).sum(1)
        assert np.array_equal(n, oracle.keysets.key_count(wl, qids))
        for i, q in enumerate(qids):
            assert n[i] == len(P.key_set_by_loops(wl, int(q)))


# ---------------------------------------------------------------- decomposition


@pytest.mark.parametrize("family", ["ttt", "block", "causal"])
@pytest.mark.parametrize("cp", [1, 2, 4])
def test_decomposition_equals_single_softmax(family, cp):
    lens = [8 * cp, 16 * cp, 8 * cp]
    wl = W.small(family, lens, heads_q=4, heads_kv=2, head_dim=16, cp=cp, depth=3, block=4,
                 anchors_per_seq=5, seed=cp)
    assert P.decomposition_error(wl) < 1e-10


def test_ring_steps_cover_every_visible_pair_once():
    wl = W.small("ttt", [16, 32], heads_q=2, heads_kv=1, head_dim=8, cp=4, depth=2, seed=4)
    C = wl.cp
    _, owner = oracle.zigzag.token_chunk(wl.cu_seqlens, C)
    count = {}
    for r in range(C):
        qids = oracle.decomposed._rank_queries(wl, r, owner)
        for s in range(C):
            src = oracle.zigzag.ring_source(r, s, C)
            kpos = np.concatenate([np.arange(a, b) for a, b in
                                   oracle.zigzag.rank_token_ranges(wl.cu_seqlens, C, src)])
            m = oracle.keysets.main_mask(wl, qids, kpos)
            for i, j in zip(*np.nonzero(m)):
                count[(int(qids[i]), int(kpos[j]))] = count.get((int(qids[i]), int(kpos[j])), 0) + 1
    want = set()
    for qid in range(wl.steps * wl.tokens):
        for kind, idx in P.key_set_by_loops(wl, qid):
            if kind == "m":
                want.add((qid, idx))
    assert set(count) == want
    assert set(count.values()) == {1}


@pytest.mark.parametrize("family", ["ttt", "block"])
def test_chunk_pair_kinds(family):
    wl = W.small(family, [32, 48], heads_q=2, heads_kv=1, head_dim=8, cp=4, depth=2, block=2,
                 anchors_per_seq=12, seed=9)
    for (s, qc, qa, qb, _) in oracle.zigzag.chunk_table(wl.cu_seqlens, wl.cp):
        units = [u for u in range(oracle.keysets.num_units(wl))
                 if qa <= oracle.keysets.unit_position(wl, u) < qb]
        if not units:
            continue
        qids = np.concatenate([oracle.keysets.queries_of_unit(wl, u) for u in units])
        for (s2, kc, ka, kb, _) in oracle.zigzag.chunk_table(wl.cu_seqlens, wl.cp):
            m = oracle.keysets.main_mask(wl, qids, np.arange(ka, kb))
            if s2 != s:
                assert not m.any()
                continue
            kind = oracle.decomposed.chunk_pair_kind(wl, qc, kc)
            if kind == "full":
                assert m.all()
            elif kind == "empty":
                assert not m.any()
            else:  # diagonal pair: the per-row causal limit decides
                p = oracle.keysets.query_anchor_position(wl, qids)
                assert np.array_equal(m, np.arange(ka, kb)[None, :] <= p[:, None])


def test_zigzag_golden():
    rows = P.parse_golden(os.path.join(GOLDEN, "zigzag_c2_L256.txt"))
    table = oracle.zigzag.chunk_table(np.array([0, 256]), 2)
    chunk_rows = [r for r in rows if r[0] != "packed"]
    assert len(chunk_rows) == len(table)
    for r, (s, c, a, b, owner) in zip(chunk_rows, table):
        assert [int(x) for x in r] == [c, a, b, owner]
    perm = oracle.zigzag.packed_token_order(np.array([0, 256]), 2)
    want = np.concatenate([np.arange(int(r[1]), int(r[2])) for r in rows if r[0] == "packed"])
    assert np.array_equal(perm, want)


def _anchor_cases():
    out = []
    for r in P.parse_golden(os.path.join(GOLDEN, "zigzag_anchors_c2.txt")):
        ints = lambda tok: np.array([int(x) for x in tok.split(";")], dtype=np.int64)
        out.append((r[0], ints(r[1]), ints(r[2]), ints(r[3]), ints(r[4])))
    return out


@pytest.mark.parametrize("case", _anchor_cases(), ids=lambda c: c[0])
def test_packed_anchor_order_golden(case):
    _, cu, anchors, want_order, want_lim = case
    order = oracle.zigzag.packed_anchor_order(cu, 2, anchors)
    assert np.array_equal(order, want_order)
    # every packed anchor's rows are limited at the anchor's own position
    assert np.array_equal(anchors[order], want_lim)


def test_ring_source_golden():
    rows = [[int(x) for x in r] for r in P.parse_golden(os.path.join(GOLDEN, "ring_c4.txt"))]
    assert [r[0] for r in rows] == [0, 1, 2, 3]
    for s, *src in rows:
        assert [oracle.zigzag.ring_source(r, s, 4) for r in range(4)] == src


def test_eq3_volume_golden_and_branch_independence():
    rows = P.parse_golden(os.path.join(GOLDEN, "eq3_volume.txt"))
    for T, C, hkv, d, want in [[int(x) for x in r] for r in rows]:
        vol = oracle.zigzag.comm_volume_fwd(np.array([0, T]), C, hkv, d, 2)
        assert (vol == want).all()
    # the schedule's volume is the same for every config drawn from the five shapes
    for k in (2, 3, 4):
        wl = W.config(k)
        vol = oracle.zigzag.comm_volume_fwd(wl.cu_seqlens, wl.cp, wl.heads_kv, wl.head_dim, 2)
        assert (vol == 2 * (wl.cp - 1) * (wl.tokens // wl.cp) * wl.heads_kv * wl.head_dim * 2).all()


def test_packed_order_is_rank_major_permutation():
    wl = W.config(2)
    perm = oracle.zigzag.packed_token_order(wl.cu_seqlens, wl.cp)
    assert np.array_equal(np.sort(perm), np.arange(wl.tokens))
    _, owner = oracle.zigzag.token_chunk(wl.cu_seqlens, wl.cp)
    assert (np.diff(owner[perm]) >= 0).all()
    # every rank holds T / C tokens
    assert (np.bincount(owner, minlength=wl.cp) == wl.tokens // wl.cp).all()


# ---------------------------------------------------------------- Eq. 2


def test_eq2_worked_examples():
    for r in P.parse_golden(os.path.join(GOLDEN, "eq2_merge_worked.txt")):
        v = [P.golden_value(x) for x in r]
        lm, lb = v[0], v[1]
        om, ob = np.array(v[2:4]), np.array(v[4:6])
        l_want, o_want = v[6], np.array(v[7:9])
        o, l = oracle.merge.lse_merge(om[None], np.array([lm]), ob[None], np.array([lb]))
        if math.isinf(l_want):
            assert np.isneginf(l[0])
        else:
            assert abs(l[0] - l_want) < 1e-14
        assert np.abs(o[0] - o_want).max() < 1e-14


def test_eq2_merge_of_halves_is_full_softmax_and_identities():
    rng = np.random.default_rng(3)
    q = rng.standard_normal((5, 8))
    k = rng.standard_normal((11, 8))
    v = rng.standard_normal((11, 8))
    full = np.ones((5, 11), bool)
    o, l = oracle.attention.masked_attention_fwd(q, k, v, full, 0.3)
    o1, l1 = oracle.attention.masked_attention_fwd(q, k[:4], v[:4], full[:, :4], 0.3)
    o2, l2 = oracle.attention.masked_attention_fwd(q, k[4:], v[4:], full[:, 4:], 0.3)
    o3, l3 = oracle.merge.lse_merge(o1, l1, o2, l2)
    assert np.abs(o3 - o).max() < 1e-14 and np.abs(l3 - l).max() < 1e-13
    # commutative
    o4, l4 = oracle.merge.lse_merge(o2, l2, o1, l1)
    assert np.abs(o4 - o3).max() < 1e-15 and np.abs(l4 - l3).max() < 1e-15
    # associative over three parts
    oa, la = oracle.attention.masked_attention_fwd(q, k[:3], v[:3], full[:, :3], 0.3)
    ob, lb = oracle.attention.masked_attention_fwd(q, k[3:7], v[3:7], full[:, 3:7], 0.3)
    oc, lc = oracle.attention.masked_attention_fwd(q, k[7:], v[7:], full[:, 7:], 0.3)
    x = oracle.merge.lse_merge(*oracle.merge.lse_merge(oa, la, ob, lb), oc, lc)
    y = oracle.merge.lse_merge(oa, la, *oracle.merge.lse_merge(ob, lb, oc, lc))
    assert np.abs(x[0] - o).max() < 1e-14 and np.abs(y[0] - o).max() < 1e-14


# ---------------------------------------------------------------- sampled evaluators


@pytest.mark.parametrize("wl", _small_cases(), ids=lambda w: w.name)
def test_sampled_evaluators_match_full(wl):
    rng = np.random.default_rng(11)
    t = P.rand_inputs(wl, rng)
    o, lse = oracle.attention.forward(wl, t)
    g = oracle.attention.backward(wl, t, o, lse)
    of = o.reshape(-1, wl.heads_q, wl.head_dim)
    lf = lse.reshape(-1, wl.heads_q)
    dq = g["dq_b"].reshape(-1, wl.heads_q, wl.head_dim)
    units = list(range(oracle.keysets.num_units(wl)))
    res = oracle.attention.unit_eval(wl, t, units)
    dkb = np.zeros_like(t["k_b"].reshape(-1, wl.heads_kv, wl.head_dim))
    for e in res:
        assert np.abs(e["o"] - of[e["qids"]]).max() < 1e-13
        assert np.abs(e["lse"] - lf[e["qids"]]).max() < 1e-13
        assert np.abs(e["dq"] - dq[e["qids"]]).max() < 1e-13
        if wl.family != "causal":
            dkb[oracle.keysets.branch_keys_of_unit(wl, e["unit"])] += e["dk_b"]
    if wl.family != "causal":
        assert np.abs(dkb - g["dk_b"].reshape(dkb.shape)).max() < 1e-13
    # main-key gradients over a window at the end of the last sequence
    s = wl.num_seqs - 1
    hi = int(wl.cu_seqlens[s + 1])
    lo = max(int(wl.cu_seqlens[s]), hi - 5)
    dk, dv = oracle.attention.main_key_grads(wl, t, lo, hi)
    assert np.abs(dk - g["dk_m"][lo:hi]).max() < 1e-13
    assert np.abs(dv - g["dv_m"][lo:hi]).max() < 1e-13


def test_useful_pairs_matches_mask_count():
    wl = W.small("block", [16, 8], heads_q=4, heads_kv=2, head_dim=16, cp=2, block=3,
                 anchors_per_seq=4, seed=2)
    n = 0
    for qid in range(wl.num_anchors * wl.block):
        n += len(P.key_set_by_loops(wl, qid))
    assert oracle.attention.useful_pairs(wl) == n * wl.heads_q
