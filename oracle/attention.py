"""Dense masked softmax attention over main + branch keys, and its gradients.

What the path computes, stated plainly ("Online Draft Co-Training ..." —
ai.info summary, "Methodology in Plain English": the decomposition is
mathematically equivalent to computing the full attention at once; rainbus
page, core method: the merge restores the exact output; the backward replays
the ring and accumulates gradients locally).  For a branch query i with key
set K(i) (see ``keysets``):

    s_ij = scale * <q_i, k_j>
    l_i  = log sum_{j in K(i)} exp(s_ij)                (natural log)
    O_i  = sum_{j in K(i)} exp(s_ij - l_i) v_j

and the gradients of <dO, O> with respect to q_b, k_m, v_m, k_b, v_b:

    P = exp(S - l), dV = P^T dO, dP = dO V^T, Delta_i = <dO_i, O_i>,
    dS = P * (dP - Delta), dQ = scale dS K, dK = scale dS^T Q.

Query head h reads kv head h // (Hq / Hkv); key gradients are summed over the
query heads of a group.  All arithmetic is fp64 on the given values; the mask
is materialised (``keysets``) and applied as -inf before the row max.
"""

from __future__ import annotations

import numpy as np

from . import keysets


# --------------------------------------------------------------------------
# the core: one dense masked softmax attention


def masked_attention_fwd(q, k, v, mask, scale):
    """q [n, d], k [m, d], v [m, d], mask [n, m] bool -> (o [n, d], lse [n]).
    Rows with no visible key give o = 0 and lse = -inf."""
    s = scale * (q @ k.T)
    s = np.where(mask, s, -np.inf)
    rowmax = s.max(axis=1, initial=-np.inf)
    shift = np.where(np.isneginf(rowmax), 0.0, rowmax)
    e = np.where(mask, np.exp(s - shift[:, None]), 0.0)
    z = e.sum(axis=1)
    with np.errstate(divide="ignore"):
        lse = np.where(z > 0, shift + np.log(np.where(z > 0, z, 1.0)), -np.inf)
    p = e / np.where(z > 0, z, 1.0)[:, None]
    return p @ v, lse


def masked_attention_probs(q, k, mask, scale, lse):
    s = scale * (q @ k.T)
    safe = np.where(np.isneginf(lse), 0.0, lse)
    return np.where(mask, np.exp(np.where(mask, s, 0.0) - safe[:, None]), 0.0)


def masked_attention_bwd(q, k, v, mask, scale, o, lse, do):
    """Gradients of <do, o> -> (dq, dk, dv) for one dense masked attention."""
    p = masked_attention_probs(q, k, mask, scale, lse)
    dv = p.T @ do
    dp = do @ v.T
    delta = (do * o).sum(axis=1)
    ds = p * (dp - delta[:, None])
    dq = scale * (ds @ k)
    dk = scale * (ds.T @ q)
    return dq, dk, dv


# --------------------------------------------------------------------------
# helpers over the natural layouts


def _flat(x, heads):
    x = np.asarray(x, dtype=np.float64)
    return x.reshape(-1, heads, x.shape[-1])


def _group(wl):
    return wl.heads_q // wl.heads_kv


# --------------------------------------------------------------------------
# full evaluation (small workloads): per sequence, all keys of the sequence


def forward(wl, t):
    """Full forward.  t: dict of arrays in natural layout (q_b, k_m, v_m, k_b,
    v_b).  Returns (o like q_b, lse [q_b.shape[:-1]]) in fp64."""
    q = _flat(t["q_b"], wl.heads_q)
    km = np.asarray(t["k_m"], dtype=np.float64)
    vm = np.asarray(t["v_m"], dtype=np.float64)
    kb = _flat(t["k_b"], wl.heads_kv) if wl.family != "causal" else None
    vb = _flat(t["v_b"], wl.heads_kv) if wl.family != "causal" else None
    o = np.zeros_like(q)
    lse = np.full(q.shape[:2], -np.inf)
    G = _group(wl)
    for s in range(wl.num_seqs):
        qids = keysets.queries_of_seq(wl, s)
        if len(qids) == 0:
            continue
        a, b = int(wl.cu_seqlens[s]), int(wl.cu_seqlens[s + 1])
        kpos = np.arange(a, b)
        bids = keysets.branch_keys_of_seq(wl, s)
        mask = np.concatenate([keysets.main_mask(wl, qids, kpos),
                               keysets.branch_mask(wl, qids, bids)], axis=1)
        for h in range(wl.heads_q):
            kh = h // G
            K = km[a:b, kh]
            V = vm[a:b, kh]
            if len(bids):
                K = np.concatenate([K, kb[bids, kh]], axis=0)
                V = np.concatenate([V, vb[bids, kh]], axis=0)
            oo, ll = masked_attention_fwd(q[qids, h], K, V, mask, wl.scale)
            o[qids, h] = oo
            lse[qids, h] = ll
    return o.reshape(np.shape(t["q_b"])), lse.reshape(np.shape(t["q_b"])[:-1])


def backward(wl, t, o=None, lse=None):
    """Full backward of <d_o, O>.  Returns dict dq_b, dk_m, dv_m, dk_b, dv_b
    (fp64, natural layouts)."""
    if o is None or lse is None:
        o, lse = forward(wl, t)
    q = _flat(t["q_b"], wl.heads_q)
    do = _flat(t["d_o"], wl.heads_q)
    of = _flat(o, wl.heads_q)
    lf = np.asarray(lse, dtype=np.float64).reshape(q.shape[:2])
    km = np.asarray(t["k_m"], dtype=np.float64)
    vm = np.asarray(t["v_m"], dtype=np.float64)
    causal = wl.family == "causal"
    kb = None if causal else _flat(t["k_b"], wl.heads_kv)
    vb = None if causal else _flat(t["v_b"], wl.heads_kv)
    dq = np.zeros_like(q)
    dkm = np.zeros_like(km)
    dvm = np.zeros_like(vm)
    dkb = None if causal else np.zeros_like(kb)
    dvb = None if causal else np.zeros_like(vb)
    G = _group(wl)
    for s in range(wl.num_seqs):
        qids = keysets.queries_of_seq(wl, s)
        if len(qids) == 0:
            continue
        a, b = int(wl.cu_seqlens[s]), int(wl.cu_seqlens[s + 1])
        n_main = b - a
        kpos = np.arange(a, b)
        bids = keysets.branch_keys_of_seq(wl, s)
        mask = np.concatenate([keysets.main_mask(wl, qids, kpos),
                               keysets.branch_mask(wl, qids, bids)], axis=1)
        for h in range(wl.heads_q):
            kh = h // G
            K = km[a:b, kh]
            V = vm[a:b, kh]
            if len(bids):
                K = np.concatenate([K, kb[bids, kh]], axis=0)
                V = np.concatenate([V, vb[bids, kh]], axis=0)
            gq, gk, gv = masked_attention_bwd(q[qids, h], K, V, mask, wl.scale, of[qids, h],
                                              lf[qids, h], do[qids, h])
            dq[qids, h] = gq
            dkm[a:b, kh] += gk[:n_main]
            dvm[a:b, kh] += gv[:n_main]
            if len(bids):
                dkb[bids, kh] += gk[n_main:]
                dvb[bids, kh] += gv[n_main:]
    out = {
        "dq_b": dq.reshape(np.shape(t["q_b"])),
        "dk_m": dkm,
        "dv_m": dvm,
    }
    if not causal:
        out["dk_b"] = dkb.reshape(np.shape(t["k_b"]))
        out["dv_b"] = dvb.reshape(np.shape(t["v_b"]))
    return out


# --------------------------------------------------------------------------
# sampled evaluation (large workloads)


class ArraySource:
    """Input access for the sampled evaluators.  ``rows(name, ids)`` returns
    flat rows of q_b / d_o (over Hq) or k_b / v_b (over Hkv) as fp64
    [len(ids), H, d]; ``main(name, kh)`` returns the whole main k_m / v_m
    column of kv head kh as fp64 [T, d].  This one reads in-memory arrays;
    callers with inputs elsewhere supply an object with the same two methods."""

    def __init__(self, wl, t):
        self.wl = wl
        self.t = t
        self._main = {}

    def rows(self, name, ids):
        heads = self.wl.heads_q if name in ("q_b", "d_o") else self.wl.heads_kv
        x = np.asarray(self.t[name])
        return np.asarray(x.reshape(-1, heads, x.shape[-1])[np.asarray(ids)], dtype=np.float64)

    def main(self, name, kh):
        key = (name, kh)
        if key not in self._main:
            self._main[key] = np.asarray(np.asarray(self.t[name])[:, kh], dtype=np.float64)
        return self._main[key]


def _as_source(wl, src):
    return src if hasattr(src, "rows") and hasattr(src, "main") else ArraySource(wl, src)


def _unit_span(wl, unit):
    p = keysets.unit_position(wl, unit)
    s = int(keysets.seq_of_position(wl.cu_seqlens, np.array([p]))[0])
    return int(wl.cu_seqlens[s]), p


def _unit_problem(wl, src, unit, grads):
    """Queries, key mask and inputs of one anchor unit."""
    qids = keysets.queries_of_unit(wl, unit)
    bids = keysets.branch_keys_of_unit(wl, unit)
    a, p = _unit_span(wl, unit)
    kpos = np.arange(a, p + 1)
    mask = np.concatenate([keysets.main_mask(wl, qids, kpos),
                           keysets.branch_mask(wl, qids, bids)], axis=1)
    causal = wl.family == "causal"
    return dict(qids=qids, bids=bids, a=a, p=p, kpos=kpos, mask=mask, Q=src.rows("q_b", qids),
                dO=src.rows("d_o", qids) if grads else None,
                Kb=None if causal else src.rows("k_b", bids), Vb=None if causal else src.rows("v_b", bids))


def _unit_kv(wl, src, u, kh):
    K = src.main("k_m", kh)[u["a"]:u["p"] + 1]
    V = src.main("v_m", kh)[u["a"]:u["p"] + 1]
    if u["Kb"] is not None:
        K = np.concatenate([K, u["Kb"][:, kh]], axis=0)
        V = np.concatenate([V, u["Vb"][:, kh]], axis=0)
    return K, V


def unit_eval(wl, src, units, heads=None, grads=True):
    """Row-local evaluation of every query hanging from the given anchor
    units (positions for TTT/causal, anchor indices for block), restricted to
    the listed q heads.  Each query's key set is built from its own unit:
    main keys [seq_start, p] and the unit's branch keys, with the mask of
    ``keysets`` applied over them.

    ``src`` is an ``ArraySource`` (or a dict of natural-layout arrays).
    Returns one dict per unit with arrays indexed [query-in-unit,
    head-in-list]: o, lse and (if grads) dq, plus the unit's branch-key
    gradients dk_b, dv_b [branch-key-in-unit, kv head] summed over the listed
    heads."""
    src = _as_source(wl, src)
    heads = list(range(wl.heads_q)) if heads is None else list(heads)
    G = _group(wl)
    res = []
    for unit in units:
        u = _unit_problem(wl, src, int(unit), grads)
        nq, nb = len(u["qids"]), len(u["bids"])
        entry = {"unit": int(unit), "qids": u["qids"],
                 "o": np.zeros((nq, len(heads), wl.head_dim)), "lse": np.zeros((nq, len(heads)))}
        if grads:
            entry["dq"] = np.zeros((nq, len(heads), wl.head_dim))
            entry["dk_b"] = np.zeros((nb, wl.heads_kv, wl.head_dim))
            entry["dv_b"] = np.zeros((nb, wl.heads_kv, wl.head_dim))
        for hi, h in enumerate(heads):
            kh = h // G
            K, V = _unit_kv(wl, src, u, kh)
            oo, ll = masked_attention_fwd(u["Q"][:, h], K, V, u["mask"], wl.scale)
            entry["o"][:, hi] = oo
            entry["lse"][:, hi] = ll
            if grads:
                gq, gk, gv = masked_attention_bwd(u["Q"][:, h], K, V, u["mask"], wl.scale, oo, ll, u["dO"][:, h])
                entry["dq"][:, hi] = gq
                n_main = len(u["kpos"])
                entry["dk_b"][:, kh] += gk[n_main:]
                entry["dv_b"][:, kh] += gv[n_main:]
        res.append(entry)
    return res


def main_key_grads(wl, src, key_lo: int, key_hi: int, kv_heads=None):
    """dK_m, dV_m for the main keys [key_lo, key_hi) (one sequence), summed
    over every query that attends them.  Each attending query's lse and O come
    from its own full key set (row-local forward), so the cost is bounded by
    the number of queries anchored at or after key_lo.

    Returns (dk [key_hi-key_lo, len(kv_heads), d], dv likewise)."""
    src = _as_source(wl, src)
    kv_heads = list(range(wl.heads_kv)) if kv_heads is None else list(kv_heads)
    cu = np.asarray(wl.cu_seqlens, dtype=np.int64)
    s = int(keysets.seq_of_position(cu, np.array([key_lo]))[0])
    if key_hi > cu[s + 1]:
        raise ValueError("window crosses a sequence end")
    G = _group(wl)
    n = key_hi - key_lo
    dk = np.zeros((n, len(kv_heads), wl.head_dim))
    dv = np.zeros((n, len(kv_heads), wl.head_dim))
    # units whose anchor lies in [key_lo, seq_end): only they attend these keys
    if wl.family == "block":
        an = np.asarray(wl.anchors, dtype=np.int64)
        units = np.nonzero((an >= key_lo) & (an < cu[s + 1]))[0]
    else:
        units = np.arange(key_lo, cu[s + 1])
    for unit in units:
        u = _unit_problem(wl, src, int(unit), True)
        a, p = u["a"], u["p"]
        m = min(p + 1, key_hi) - key_lo  # window keys this unit sees
        for ki, kh in enumerate(kv_heads):
            K, V = _unit_kv(wl, src, u, kh)
            for h in range(kh * G, (kh + 1) * G):
                oo, ll = masked_attention_fwd(u["Q"][:, h], K, V, u["mask"], wl.scale)
                _, gk, gv = masked_attention_bwd(u["Q"][:, h], K, V, u["mask"], wl.scale, oo, ll, u["dO"][:, h])
                dk[:m, ki] += gk[key_lo - a:key_lo - a + m]
                dv[:m, ki] += gv[key_lo - a:key_lo - a + m]
    return dk, dv


def useful_pairs(wl) -> int:
    """Number of unmasked (query-head row, key) pairs: the useful work."""
    total = 0
    for s in range(wl.num_seqs):
        qids = keysets.queries_of_seq(wl, s)
        total += int(keysets.key_count(wl, qids).sum())
    return total * wl.heads_q
