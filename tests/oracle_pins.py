"""Checks that pin the oracle to something other than itself.

Each function returns a scalar error so the same check can serve as a pin
(error ~ 0) and, in the mutation tests, show that a planted mistake in the
oracle is caught (error large).  The expected values here come from the
definitions on the pages restated independently (explicit Python loops), from
closed forms, or from library routines (torch SDPA) — never from the oracle.
"""

from __future__ import annotations

import math

import numpy as np
import torch

import oracle
from branch_attention_speculative_gb300 import workloads as W


# --------------------------------------------------------------------------
# key sets restated from the definition, by explicit loops


def key_set_by_loops(wl, qid):
    """Key set of one flat query id as a python set of ('m', pos) / ('b', id):
    TTT step-j query at p sees main [start, p] and branch (p, i<=j); block
    query of anchor a sees main [start, p_a] and all B keys of a."""
    cu = [int(x) for x in wl.cu_seqlens]
    if wl.family == "block":
        a = qid // wl.block
        p = int(wl.anchors[a])
    else:
        p = qid % wl.tokens
    s = 0
    while not (cu[s] <= p < cu[s + 1]):
        s += 1
    keys = set()
    for pos in range(cu[s], p + 1):
        keys.add(("m", pos))
    if wl.family == "ttt":
        j = qid // wl.tokens
        for i in range(j + 1):
            keys.add(("b", i * wl.tokens + p))
    elif wl.family == "block":
        for u in range(wl.block):
            keys.add(("b", a * wl.block + u))
    return keys


def rand_inputs(wl, rng, dtype=np.float64):
    sh = W.tensor_shapes(wl)
    return {k: rng.standard_normal(v).astype(dtype) for k, v in sh.items()}


# --------------------------------------------------------------------------
# pin 1: uniform attention reveals the key sets exactly


def uniform_keyset_error(wl):
    """q = 0 makes every visible key equally weighted, so l_i = log|K(i)| and,
    with one-hot values, O_i is the indicator of K(i) divided by |K(i)|."""
    T = wl.tokens
    nb = int(np.prod(wl.kb_shape()[:2]))
    d = T + nb
    wl2 = W.Workload(wl.name, wl.family, wl.cu_seqlens, wl.heads_q, wl.heads_kv, d, wl.cp,
                     wl.depth, wl.block, wl.anchors, wl.seed)
    t = {
        "q_b": np.zeros(wl2.q_shape()),
        "k_m": np.random.default_rng(0).standard_normal(wl2.km_shape()),
        "v_m": np.zeros(wl2.km_shape()),
        "k_b": np.random.default_rng(1).standard_normal(wl2.kb_shape()),
        "v_b": np.zeros(wl2.kb_shape()),
    }
    for pos in range(T):
        t["v_m"][pos, :, pos] = 1.0
    vb = t["v_b"].reshape(-1, wl2.heads_kv, d)
    for i in range(nb):
        vb[i, :, T + i] = 1.0
    t["v_b"] = vb.reshape(wl2.kb_shape())
    o, lse = oracle.attention.forward(wl2, t)
    o = o.reshape(-1, wl2.heads_q, d)
    lse = lse.reshape(-1, wl2.heads_q)
    err = 0.0
    for qid in range(o.shape[0]):
        ks = key_set_by_loops(wl2, qid)
        want = np.zeros(d)
        for (kind, idx) in ks:
            want[idx if kind == "m" else T + idx] = 1.0 / len(ks)
        for h in range(wl2.heads_q):
            err = max(err, float(np.abs(o[qid, h] - want).max()))
            err = max(err, abs(float(lse[qid, h]) - math.log(len(ks))))
    return err


# --------------------------------------------------------------------------
# pin 2: torch SDPA (fp64, CPU) with a mask built by loops


def sdpa_error(wl, seed=0):
    """Oracle O against torch.nn.functional.scaled_dot_product_attention fed
    all keys of the workload and a boolean mask built by ``key_set_by_loops``."""
    rng = np.random.default_rng(seed)
    t = rand_inputs(wl, rng)
    o, _ = oracle.attention.forward(wl, t)
    o = o.reshape(-1, wl.heads_q, wl.head_dim)
    T = wl.tokens
    q = t["q_b"].reshape(-1, wl.heads_q, wl.head_dim)
    nq = q.shape[0]
    kb = t["k_b"].reshape(-1, wl.heads_kv, wl.head_dim)
    vb = t["v_b"].reshape(-1, wl.heads_kv, wl.head_dim)
    nb = kb.shape[0]
    mask = np.zeros((nq, T + nb), dtype=bool)
    for qid in range(nq):
        for (kind, idx) in key_set_by_loops(wl, qid):
            mask[qid, idx if kind == "m" else T + idx] = True
    G = wl.heads_q // wl.heads_kv
    err = 0.0
    for h in range(wl.heads_q):
        kh = h // G
        K = np.concatenate([t["k_m"][:, kh], kb[:, kh]], axis=0)
        V = np.concatenate([t["v_m"][:, kh], vb[:, kh]], axis=0)
        ref = torch.nn.functional.scaled_dot_product_attention(
            torch.from_numpy(q[:, h])[None], torch.from_numpy(K)[None], torch.from_numpy(V)[None],
            attn_mask=torch.from_numpy(mask)[None], scale=wl.scale)[0].numpy()
        err = max(err, float(np.abs(ref - o[:, h]).max()))
    return err


# --------------------------------------------------------------------------
# pin 3: finite differences of f = <dO, O> and of l


def fd_error(wl, seed=0, eps=1e-6, n_dirs=3):
    """Relative error of the oracle's gradients against central differences
    along random directions, per input tensor; and of dl/dq against the
    central difference of l."""
    rng = np.random.default_rng(seed)
    t = rand_inputs(wl, rng)
    g = oracle.attention.backward(wl, t)
    names = [("q_b", "dq_b"), ("k_m", "dk_m"), ("v_m", "dv_m")]
    if wl.family != "causal":
        names += [("k_b", "dk_b"), ("v_b", "dv_b")]

    def f(tt):
        o, _ = oracle.attention.forward(wl, tt)
        return float((o * tt["d_o"]).sum())

    worst = 0.0
    for x, gx in names:
        for _ in range(n_dirs):
            u = rng.standard_normal(t[x].shape)
            tp = dict(t)
            tm = dict(t)
            tp[x] = t[x] + eps * u
            tm[x] = t[x] - eps * u
            num = (f(tp) - f(tm)) / (2 * eps)
            ana = float((g[gx] * u).sum())
            worst = max(worst, abs(num - ana) / max(1.0, abs(num)))
    # d l_i / d q_i = scale * sum_j P_ij k_j : check on the lse sum
    u = rng.standard_normal(t["q_b"].shape)
    tp = dict(t)
    tm = dict(t)
    tp["q_b"] = t["q_b"] + eps * u
    tm["q_b"] = t["q_b"] - eps * u
    num = (oracle.attention.forward(wl, tp)[1].sum() - oracle.attention.forward(wl, tm)[1].sum()) / (2 * eps)
    # analytic: with V := K the output is sum_j P_ij k_j
    t2 = dict(t)
    t2["v_m"] = t["k_m"]
    if wl.family != "causal":
        t2["v_b"] = t["k_b"]
    ok, _ = oracle.attention.forward(wl, t2)
    ana = wl.scale * float((ok * u).sum())
    worst = max(worst, abs(num - ana) / max(1.0, abs(num)))
    return worst


# --------------------------------------------------------------------------
# pin 4: exact gradient invariants


def invariant_errors(wl, g, t):
    """Relative errors of the three identities that follow from
    sum_j P_ij = 1 and sum_j dS_ij = 0, per kv head:
      sum over all keys of dK = 0;  sum of dV = sum of dO over the group's
      queries;  sum_i <q_i, dq_i> = sum_j <k_j, dk_j>."""
    Hkv, G, d = wl.heads_kv, wl.heads_q // wl.heads_kv, wl.head_dim
    dq = np.asarray(g["dq_b"], dtype=np.float64).reshape(-1, wl.heads_q, d)
    q = np.asarray(t["q_b"], dtype=np.float64).reshape(-1, wl.heads_q, d)
    do = np.asarray(t["d_o"], dtype=np.float64).reshape(-1, wl.heads_q, d)
    dkm = np.asarray(g["dk_m"], dtype=np.float64)
    dvm = np.asarray(g["dv_m"], dtype=np.float64)
    km = np.asarray(t["k_m"], dtype=np.float64)
    has_b = wl.family != "causal"
    if has_b:
        dkb = np.asarray(g["dk_b"], dtype=np.float64).reshape(-1, Hkv, d)
        dvb = np.asarray(g["dv_b"], dtype=np.float64).reshape(-1, Hkv, d)
        kb = np.asarray(t["k_b"], dtype=np.float64).reshape(-1, Hkv, d)
    out = {"sum_dk": 0.0, "sum_dv": 0.0, "qdq_kdk": 0.0}
    for kh in range(Hkv):
        hs = slice(kh * G, (kh + 1) * G)
        sdk = dkm[:, kh].sum(0) + (dkb[:, kh].sum(0) if has_b else 0)
        scale_dk = np.abs(dkm[:, kh]).sum(0) + (np.abs(dkb[:, kh]).sum(0) if has_b else 0)
        out["sum_dk"] = max(out["sum_dk"], float((np.abs(sdk) / (scale_dk + 1e-30)).max()))
        sdv = dvm[:, kh].sum(0) + (dvb[:, kh].sum(0) if has_b else 0)
        sdo = do[:, hs].sum((0, 1))
        scale_dv = np.abs(dvm[:, kh]).sum(0) + (np.abs(dvb[:, kh]).sum(0) if has_b else 0) + np.abs(do[:, hs]).sum((0, 1))
        out["sum_dv"] = max(out["sum_dv"], float((np.abs(sdv - sdo) / (scale_dv + 1e-30)).max()))
        lhs_terms = (q[:, hs] * dq[:, hs]).sum(-1)
        rhs_terms = (km[:, kh] * dkm[:, kh]).sum(-1)
        if has_b:
            rhs_terms = np.concatenate([rhs_terms, (kb[:, kh] * dkb[:, kh]).sum(-1)])
        lhs, rhs = lhs_terms.sum(), rhs_terms.sum()
        den = np.abs(lhs_terms).sum() + np.abs(rhs_terms).sum() + 1e-30
        out["qdq_kdk"] = max(out["qdq_kdk"], float(abs(lhs - rhs) / den))
    return out


# --------------------------------------------------------------------------
# pin 5: the decomposition identity


def decomposition_error(wl, seed=0):
    rng = np.random.default_rng(seed)
    t = rand_inputs(wl, rng)
    o1, l1 = oracle.attention.forward(wl, t)
    o2, l2 = oracle.decomposed.forward(wl, t)
    return max(float(np.abs(o1 - o2).max()), float(np.abs(l1 - l2).max()))


def parse_golden(path):
    rows = []
    for line in open(path):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        rows.append(line.split())
    return rows


def golden_value(tok: str) -> float:
    tok = tok.strip()
    if tok == "-inf":
        return -math.inf
    if tok.startswith("log(") and tok.endswith(")"):
        return math.log(float(tok[4:-1]))
    return float(tok)
