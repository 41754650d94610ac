"""Plant plausible mistakes in the oracle (on the CPU) and check that at least
one pin catches each of them: the pins are sensitive, not just self-consistent."""

import os

import numpy as np
import pytest

import oracle
from branch_attention_speculative_gb300 import workloads as W
from tests import oracle_pins as P

TTT = W.small("ttt", [8, 8], heads_q=4, heads_kv=2, head_dim=16, cp=2, depth=3, seed=1)
BLK = W.small("block", [16, 8], heads_q=4, heads_kv=2, head_dim=16, cp=2, block=3,
              anchors_per_seq=4, seed=2)


def _pins_fail(wl):
    errs = [P.uniform_keyset_error(wl), P.sdpa_error(wl), P.fd_error(wl, n_dirs=1)]
    return max(errs[0], errs[1]) > 1e-6 or errs[2] > 1e-4


def test_unmutated_pins_pass():
    assert not _pins_fail(TTT)
    assert not _pins_fail(BLK)


def test_anchor_key_dropped_is_caught(monkeypatch):
    orig = oracle.keysets.main_mask

    def wrong(wl, qids, kpos):
        p = oracle.keysets.query_anchor_position(wl, qids)
        return orig(wl, qids, kpos) & (np.asarray(kpos)[None, :] < p[:, None])

    monkeypatch.setattr(oracle.keysets, "main_mask", wrong)
    assert _pins_fail(TTT)


def test_ttt_own_step_key_dropped_is_caught(monkeypatch):
    def wrong(wl, qids, kids):
        T = wl.tokens
        qids, kids = np.asarray(qids), np.asarray(kids)
        return ((kids[None, :] % T) == (qids[:, None] % T)) & ((kids[None, :] // T) < (qids[:, None] // T))

    monkeypatch.setattr(oracle.keysets, "branch_mask", wrong)
    assert _pins_fail(TTT)


def test_block_made_causal_is_caught(monkeypatch):
    def wrong(wl, qids, kids):
        qids, kids = np.asarray(qids), np.asarray(kids)
        B = wl.block
        return ((kids[None, :] // B) == (qids[:, None] // B)) & ((kids[None, :] % B) <= (qids[:, None] % B))

    monkeypatch.setattr(oracle.keysets, "branch_mask", wrong)
    assert _pins_fail(BLK)


def test_missing_softmax_scale_is_caught(monkeypatch):
    orig = oracle.attention.masked_attention_fwd
    monkeypatch.setattr(oracle.attention, "masked_attention_fwd",
                        lambda q, k, v, m, scale: orig(q, k, v, m, 1.0))
    assert _pins_fail(TTT)


def test_wrong_backward_term_is_caught(monkeypatch):
    def wrong(q, k, v, mask, scale, o, lse, do):
        p = oracle.attention.masked_attention_probs(q, k, mask, scale, lse)
        dv = p.T @ do
        dp = do @ v.T
        ds = p * dp  # Delta term dropped
        return scale * (ds @ k), scale * (ds.T @ q), dv

    monkeypatch.setattr(oracle.attention, "masked_attention_bwd", wrong)
    assert _pins_fail(TTT)


def test_wrong_eq2_weight_is_caught(monkeypatch):
    orig = oracle.merge.lse_merge

    def wrong(o_m, l_m, o_b, l_b):
        o, l = orig(o_m, l_m, o_b, l_b)
        return o, l + 1e-3

    monkeypatch.setattr(oracle.decomposed, "lse_merge", wrong)
    assert P.decomposition_error(TTT) > 1e-6


def test_wrong_zigzag_owner_is_caught(monkeypatch):
    monkeypatch.setattr(oracle.zigzag, "chunk_owner", lambda c, C: c % C)
    table = oracle.zigzag.chunk_table(np.array([0, 256]), 2)
    rows = [r for r in P.parse_golden(os.path.join(os.path.dirname(__file__), "golden", "zigzag_c2_L256.txt")) if r[0] != "packed"]
    assert any(int(r[3]) != t[4] for r, t in zip(rows, table))


def _anchor_golden():
    rows = P.parse_golden(os.path.join(os.path.dirname(__file__), "golden", "zigzag_anchors_c2.txt"))
    ints = lambda tok: np.array([int(x) for x in tok.split(";")], dtype=np.int64)
    return [(ints(r[1]), ints(r[2]), ints(r[3])) for r in rows]


def test_anchors_left_in_natural_order_are_caught(monkeypatch):
    monkeypatch.setattr(oracle.zigzag, "packed_anchor_order",
                        lambda cu, C, anchors: np.arange(len(anchors)))
    assert any(not np.array_equal(oracle.zigzag.packed_anchor_order(cu, 2, a), want)
               for cu, a, want in _anchor_golden())


def test_tail_chunk_before_head_chunk_is_caught(monkeypatch):
    # rank-major, but each rank's tail chunk (2C-1-r) listed before its head chunk (r)
    def wrong(cu, C, anchors):
        chunk, owner = oracle.zigzag.token_chunk(cu, C)
        a = np.asarray(anchors)
        seq = np.searchsorted(np.asarray(cu), a, side="right") - 1
        head = (chunk[a] == owner[a]).astype(np.int64)
        return np.lexsort((a, head, seq, owner[a]))

    monkeypatch.setattr(oracle.zigzag, "packed_anchor_order", wrong)
    assert any(not np.array_equal(oracle.zigzag.packed_anchor_order(cu, 2, a), want)
               for cu, a, want in _anchor_golden())


def test_reversed_ring_direction_is_caught(monkeypatch):
    monkeypatch.setattr(oracle.zigzag, "ring_source", lambda r, s, C: (r + s) % C)
    rows = [[int(x) for x in r] for r in
            P.parse_golden(os.path.join(os.path.dirname(__file__), "golden", "ring_c4.txt"))]
    assert any([oracle.zigzag.ring_source(r, s, 4) for r in range(4)] != src for s, *src in rows)
