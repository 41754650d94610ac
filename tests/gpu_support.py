"""Helpers for the GPU parity tests: a lazy input source that lets the
oracle read only the rows it needs from device tensors, tolerance checks, and
the seeded choice of sampled units."""

from __future__ import annotations

import numpy as np
import torch

import oracle

# Numeric tolerances (the stated bar for bf16 outputs against the fp64 oracle):
O_MAX_ABS = 2e-2
O_REL_RMS = 1e-2
LSE_MAX_ABS = 1e-3
GRAD_REL_RMS = 2e-2
INVARIANT_REL = 1e-2


class TorchSource:
    """oracle.attention input source over natural-layout device tensors."""

    def __init__(self, wl, tensors):
        self.wl = wl
        self.t = tensors
        self._main = {}

    def rows(self, name, ids):
        heads = self.wl.heads_q if name in ("q_b", "d_o") else self.wl.heads_kv
        x = self.t[name].reshape(-1, heads, self.wl.head_dim)
        idx = torch.as_tensor(np.asarray(ids, dtype=np.int64), device=x.device)
        return x.index_select(0, idx).float().cpu().double().numpy()

    def main(self, name, kh):
        key = (name, kh)
        if key not in self._main:
            self._main[key] = self.t[name][:, kh].contiguous().float().cpu().double().numpy()
        return self._main[key]


def rel_rms(got, want):
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    den = np.sqrt((want ** 2).mean())
    return float(np.sqrt(((got - want) ** 2).mean()) / max(den, 1e-30))


def check_o(got, want, what="o"):
    ma = float(np.abs(np.asarray(got, np.float64) - want).max())
    rr = rel_rms(got, want)
    assert ma <= O_MAX_ABS and rr <= O_REL_RMS, f"{what}: max-abs {ma:.3e} rel-rms {rr:.3e}"
    return ma, rr


def check_lse(got, want, what="lse"):
    ma = float(np.abs(np.asarray(got, np.float64) - want).max())
    assert ma <= LSE_MAX_ABS, f"{what}: max-abs {ma:.3e}"
    return ma


def check_grad(got, want, what):
    rr = rel_rms(got, want)
    assert rr <= GRAD_REL_RMS, f"{what}: rel-rms {rr:.3e}"
    return rr


def sample_units(wl, n, seed=1234):
    """Seeded anchor units: each sequence's first and last unit, the first
    and last unit of a few zigzag chunks, and uniform draws."""
    rng = np.random.default_rng(seed + wl.seed)
    nu = oracle.keysets.num_units(wl)
    pos = np.array([oracle.keysets.unit_position(wl, u) for u in range(nu)]) if wl.family == "block" else None
    picks = set()
    for (s, c, a, b, _) in oracle.zigzag.chunk_table(wl.cu_seqlens, wl.cp):
        if wl.family == "block":
            inside = np.nonzero((pos >= a) & (pos < b))[0]
            cand = [int(inside[0]), int(inside[-1])] if len(inside) else []
        else:
            cand = [a, b - 1]
        if c in (0, 2 * wl.cp - 1) or rng.random() < 0.25:
            picks.update(cand)
    picks = sorted(picks)
    if len(picks) > n // 2:
        picks = sorted(rng.choice(picks, n // 2, replace=False).tolist())
    rest = rng.choice(nu, size=min(nu, n - len(picks)), replace=False)
    return sorted(set(picks) | set(int(x) for x in rest))


def invariant_errors_torch(wl, t, g, chunk=1 << 18):
    """The three exact gradient identities on full device gradients, summed
    in fp64 over row chunks (no full-size fp64 copies): per kv head, the sum
    of dK over all keys = 0, the sum of dV = the sum of dO over the group's
    queries, sum <q, dq> = sum <k, dk>; each as |lhs - rhs| / sum|terms|."""
    Hkv, G, d = wl.heads_kv, wl.heads_q // wl.heads_kv, wl.head_dim
    dev = t["q_b"].device
    z = lambda *shape: torch.zeros(shape, dtype=torch.float64, device=dev)

    def rows(x, heads):
        return x.reshape(-1, heads, d)

    # query side: per q head, sum_i <q_i, dq_i> and its |terms|, sum_i dO_i, sum |dO_i|
    q, dq, do = rows(t["q_b"], wl.heads_q), rows(g["dq_b"], wl.heads_q), rows(t["d_o"], wl.heads_q)
    qdq, qdq_abs, sdo, sdo_abs = z(wl.heads_q), z(wl.heads_q), z(wl.heads_q, d), z(wl.heads_q, d)
    for i in range(0, q.shape[0], chunk):
        a = (q[i:i + chunk].float() * dq[i:i + chunk].float()).sum(-1).double()
        qdq += a.sum(0)
        qdq_abs += a.abs().sum(0)
        x = do[i:i + chunk].double()
        sdo += x.sum(0)
        sdo_abs += x.abs().sum(0)
    # key side: per kv head, sums of dK, |dK|, dV, |dV|, <k, dk>, |<k, dk>|
    sdk, adk, sdv, adv, kdk, kdk_abs = z(Hkv, d), z(Hkv, d), z(Hkv, d), z(Hkv, d), z(Hkv), z(Hkv)
    pairs = [(t["k_m"], g["dk_m"], g["dv_m"])]
    if wl.family != "causal":
        pairs.append((t["k_b"], g["dk_b"], g["dv_b"]))
    for k, gk, gv in pairs:
        k, gk, gv = rows(k, Hkv), rows(gk, Hkv), rows(gv, Hkv)
        for i in range(0, k.shape[0], chunk):
            x, y = gk[i:i + chunk].double(), gv[i:i + chunk].double()
            sdk += x.sum(0)
            adk += x.abs().sum(0)
            sdv += y.sum(0)
            adv += y.abs().sum(0)
            a = (k[i:i + chunk].float() * gk[i:i + chunk].float()).sum(-1).double()
            kdk += a.sum(0)
            kdk_abs += a.abs().sum(0)
    out = {"sum_dk": 0.0, "sum_dv": 0.0, "qdq_kdk": 0.0}
    for kh in range(Hkv):
        hs = slice(kh * G, (kh + 1) * G)
        out["sum_dk"] = max(out["sum_dk"], float((sdk[kh].abs() / adk[kh].clamp_min(1e-30)).max()))
        gd = sdo[hs].sum(0)
        out["sum_dv"] = max(out["sum_dv"], float(((sdv[kh] - gd).abs() /
                                                    (adv[kh] + sdo_abs[hs].sum(0)).clamp_min(1e-30)).max()))
        lhs, rhs = qdq[hs].sum(), kdk[kh]
        den = qdq_abs[hs].sum() + kdk_abs[kh]
        out["qdq_kdk"] = max(out["qdq_kdk"], float((lhs - rhs).abs() / den))
    return out
