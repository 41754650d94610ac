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


def invariant_errors_torch(wl, t, g):
    """The three exact gradient identities on full device gradients (fp64):
    per kv head, sum of dK over all keys = 0, sum of dV = sum of dO over the
    group's queries, sum <q, dq> = sum <k, dk>; each as |lhs - rhs| / sum|terms|."""
    Hkv, G, d = wl.heads_kv, wl.heads_q // wl.heads_kv, wl.head_dim
    f = lambda x: x.double()
    q = f(t["q_b"]).reshape(-1, wl.heads_q, d)
    do = f(t["d_o"]).reshape(-1, wl.heads_q, d)
    dq = f(g["dq_b"]).reshape(-1, wl.heads_q, d)
    km, dkm, dvm = f(t["k_m"]), f(g["dk_m"]), f(g["dv_m"])
    has_b = wl.family != "causal"
    if has_b:
        kb = f(t["k_b"]).reshape(-1, Hkv, d)
        dkb = f(g["dk_b"]).reshape(-1, Hkv, d)
        dvb = f(g["dv_b"]).reshape(-1, Hkv, d)
    out = {"sum_dk": 0.0, "sum_dv": 0.0, "qdq_kdk": 0.0}
    for kh in range(Hkv):
        hs = slice(kh * G, (kh + 1) * G)
        sdk = dkm[:, kh].sum(0) + (dkb[:, kh].sum(0) if has_b else 0)
        adk = dkm[:, kh].abs().sum(0) + (dkb[:, kh].abs().sum(0) if has_b else 0)
        out["sum_dk"] = max(out["sum_dk"], float((sdk.abs() / adk.clamp_min(1e-30)).max()))
        sdv = dvm[:, kh].sum(0) + (dvb[:, kh].sum(0) if has_b else 0)
        sdo = do[:, hs].sum((0, 1))
        adv = dvm[:, kh].abs().sum(0) + (dvb[:, kh].abs().sum(0) if has_b else 0) + do[:, hs].abs().sum((0, 1))
        out["sum_dv"] = max(out["sum_dv"], float(((sdv - sdo).abs() / adv.clamp_min(1e-30)).max()))
        lt = (q[:, hs] * dq[:, hs]).sum(-1)
        rt = (km[:, kh] * dkm[:, kh]).sum(-1)
        rb = (kb[:, kh] * dkb[:, kh]).sum(-1) if has_b else torch.zeros(1, dtype=torch.float64, device=q.device)
        lhs, rhs = lt.sum(), rt.sum() + rb.sum()
        den = lt.abs().sum() + rt.abs().sum() + rb.abs().sum()
        out["qdq_kdk"] = max(out["qdq_kdk"], float((lhs - rhs).abs() / den))
    return out
