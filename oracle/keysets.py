"""Which keys a branch query attends — the branch mask.

Source: "Online Draft Co-Training ..." — ai.info summary, Key Contributions 1
and "Methodology in Plain English" (each branch query looks at the causal
prefix of the main sequence and at a small set of keys of its own branch);
paperlens walkthrough, "The two walls" / Wall 1 (EAGLE-3 TTT grows a branch
from every position; DFlash generates a whole block in one pass; every branch
attends the causal prefix and its own branch-local KV); rainbus page,
prerequisites on the three draft families.

Readings taken where the pages are silent:
* TTT: the step-j query (j = 1..D) anchored at main position p attends main
  keys [seq_start, p] (inclusive) and branch keys (p, i) for 1 <= i <= j.
  Stored 0-based: row (jj, p) attends branch keys (ii, p), ii <= jj.
* Block (DFlash, DSpark): every one of the B branch queries of anchor p
  attends main keys [seq_start, p] and all B branch keys of that anchor
  (bidirectional inside the block).
* Causal: main queries with no branch keys (plain causal varlen attention).

Query ids are flat indices into q_b reshaped to [-1, Hq, d]; TTT: jj*T + t,
block: a*B + u, causal: t.  Branch key ids are flat indices into k_b reshaped
to [-1, Hkv, d] in the same way.
"""

from __future__ import annotations

import numpy as np


def seq_of_position(cu_seqlens: np.ndarray, pos: np.ndarray) -> np.ndarray:
    return np.searchsorted(cu_seqlens, pos, side="right") - 1


def query_anchor_position(wl, qids: np.ndarray) -> np.ndarray:
    """The main position p that a query's branch hangs from."""
    qids = np.asarray(qids, dtype=np.int64)
    if wl.family == "block":
        return np.asarray(wl.anchors, dtype=np.int64)[qids // wl.block]
    return qids % wl.tokens


def main_mask(wl, qids: np.ndarray, kpos: np.ndarray) -> np.ndarray:
    """[len(qids), len(kpos)] bool: query attends main key at position kpos
    iff the key lies in the query's sequence and at or before its anchor."""
    p = query_anchor_position(wl, qids)
    cu = np.asarray(wl.cu_seqlens, dtype=np.int64)
    start = cu[seq_of_position(cu, p)]
    kpos = np.asarray(kpos, dtype=np.int64)
    return (kpos[None, :] >= start[:, None]) & (kpos[None, :] <= p[:, None])


def branch_mask(wl, qids: np.ndarray, kids: np.ndarray) -> np.ndarray:
    """[len(qids), len(kids)] bool: query attends branch key kids."""
    qids = np.asarray(qids, dtype=np.int64)
    kids = np.asarray(kids, dtype=np.int64)
    if wl.family == "ttt":
        T = wl.tokens
        jj, tq = qids // T, qids % T
        ii, tk = kids // T, kids % T
        return (tk[None, :] == tq[:, None]) & (ii[None, :] <= jj[:, None])
    if wl.family == "block":
        B = wl.block
        return (kids[None, :] // B) == (qids[:, None] // B)
    return np.zeros((len(qids), len(kids)), dtype=bool)


def queries_of_seq(wl, s: int) -> np.ndarray:
    """Flat query ids whose anchor lies in sequence s."""
    a, b = int(wl.cu_seqlens[s]), int(wl.cu_seqlens[s + 1])
    if wl.family == "block":
        an = np.asarray(wl.anchors, dtype=np.int64)
        idx = np.nonzero((an >= a) & (an < b))[0]
        return (idx[:, None] * wl.block + np.arange(wl.block)[None, :]).reshape(-1)
    T = wl.tokens
    return (np.arange(wl.steps)[:, None] * T + np.arange(a, b)[None, :]).reshape(-1)


def branch_keys_of_seq(wl, s: int) -> np.ndarray:
    """Flat branch-key ids whose anchor lies in sequence s."""
    if wl.family == "causal":
        return np.zeros(0, dtype=np.int64)
    return queries_of_seq(wl, s)  # branch keys are laid out exactly like the queries


def queries_of_unit(wl, unit: int) -> np.ndarray:
    """All queries hanging from one anchor unit: position t (TTT, causal) or
    anchor index a (block)."""
    if wl.family == "block":
        return unit * wl.block + np.arange(wl.block, dtype=np.int64)
    return np.arange(wl.steps, dtype=np.int64) * wl.tokens + unit


def branch_keys_of_unit(wl, unit: int) -> np.ndarray:
    if wl.family == "causal":
        return np.zeros(0, dtype=np.int64)
    return queries_of_unit(wl, unit)


def unit_position(wl, unit: int) -> int:
    if wl.family == "block":
        return int(wl.anchors[unit])
    return int(unit)


def num_units(wl) -> int:
    return wl.num_anchors if wl.family == "block" else wl.tokens


def key_count(wl, qids: np.ndarray) -> np.ndarray:
    """|key set| per query in closed form: (p - seq_start + 1) main keys plus
    jj + 1 (TTT) or B (block) branch keys.  Pinned against the mask."""
    p = query_anchor_position(wl, qids)
    cu = np.asarray(wl.cu_seqlens, dtype=np.int64)
    n_main = p - cu[seq_of_position(cu, p)] + 1
    if wl.family == "ttt":
        return n_main + (np.asarray(qids) // wl.tokens) + 1
    if wl.family == "block":
        return n_main + wl.block
    return n_main
