"""The decomposed path: main ring partials + rank-local branch part + Eq. 2.

Source: "Online Draft Co-Training ..." — ai.info summary, Key Contributions 1
and "Methodology in Plain English" (main part by packed zigzag-ring attention
with K/V circulating and queries staying put, branch part computed locally on
the anchor's rank, the two merged with the log-sum-exp trick that ring
attention already uses between steps); rainbus page, Figure 1(b) (each rank
merges the ring result with its local branch attention via Eq. 2) and step 2
of the method.

This is the method's own order of work, kept separate from ``attention`` so
the tests can show that it reaches the plain definition (to 1e-10 in fp64):
for every virtual rank r and ring step s, the rank's queries attend the main
keys held by rank (r - s) mod C (causal mask inside the same sequence); the C
partials are merged in ring order with Eq. 2; the branch partial over the
rank-local branch keys is merged last with Eq. 2.
"""

from __future__ import annotations

import numpy as np

from . import keysets, zigzag
from .attention import masked_attention_fwd, _flat, _group
from .merge import lse_merge


def _rank_queries(wl, r, owner_of_token):
    """Flat query ids whose anchor position is held by rank r."""
    units = np.arange(keysets.num_units(wl))
    pos = np.array([keysets.unit_position(wl, u) for u in units], dtype=np.int64)
    mine = units[owner_of_token[pos] == r] if len(units) else units
    if len(mine) == 0:
        return np.zeros(0, dtype=np.int64)
    return np.concatenate([keysets.queries_of_unit(wl, int(u)) for u in mine])


def forward(wl, t, record_steps=False):
    """Decomposed forward.  Returns (o, lse) like ``attention.forward`` and,
    with record_steps, the list of per (rank, step) partial lse arrays."""
    C = wl.cp
    q = _flat(t["q_b"], wl.heads_q)
    km = np.asarray(t["k_m"], dtype=np.float64)
    vm = np.asarray(t["v_m"], dtype=np.float64)
    causal = wl.family == "causal"
    kb = None if causal else _flat(t["k_b"], wl.heads_kv)
    vb = None if causal else _flat(t["v_b"], wl.heads_kv)
    _, owner = zigzag.token_chunk(wl.cu_seqlens, C)
    G = _group(wl)
    o = np.zeros_like(q)
    lse = np.full(q.shape[:2], -np.inf)
    steps = []
    for r in range(C):
        qids = _rank_queries(wl, r, owner)
        if len(qids) == 0:
            continue
        for h in range(wl.heads_q):
            kh = h // G
            Q = q[qids, h]
            o_m = np.zeros((len(qids), wl.head_dim))
            l_m = np.full(len(qids), -np.inf)
            for s in range(C):
                src = zigzag.ring_source(r, s, C)
                kpos = np.concatenate([np.arange(a, b) for (a, b) in
                                       zigzag.rank_token_ranges(wl.cu_seqlens, C, src)])
                mask = keysets.main_mask(wl, qids, kpos)
                o_s, l_s = masked_attention_fwd(Q, km[kpos, kh], vm[kpos, kh], mask, wl.scale)
                if record_steps:
                    steps.append((r, s, h, qids, l_s))
                o_m, l_m = lse_merge(o_m, l_m, o_s, l_s)
            if causal:
                o_f, l_f = o_m, l_m
            else:
                bids = np.unique(qids)  # branch keys are laid out like the queries
                bmask = keysets.branch_mask(wl, qids, bids)
                o_b, l_b = masked_attention_fwd(Q, kb[bids, kh], vb[bids, kh], bmask, wl.scale)
                o_f, l_f = lse_merge(o_m, l_m, o_b, l_b)
            o[qids, h] = o_f
            lse[qids, h] = l_f
    o = o.reshape(np.shape(t["q_b"]))
    lse = lse.reshape(np.shape(t["q_b"])[:-1])
    if record_steps:
        return o, lse, steps
    return o, lse


def chunk_pair_kind(wl, qc: int, kc: int) -> str:
    """Classification of a (query chunk, key chunk) pair of one sequence under
    the causal main mask: 'full' if kc < qc, 'diag' if kc == qc, 'empty' if
    kc > qc."""
    if kc < qc:
        return "full"
    if kc == qc:
        return "diag"
    return "empty"
