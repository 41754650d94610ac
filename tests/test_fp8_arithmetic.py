"""The 8-bit forward's error bars against what e4m3 arithmetic itself does
(CPU, no GPU): the kernel's roundings — q, k and v to e4m3 with one scale per
tensor (amax / 448), P = 2^(s - m) against a reference max taken from a row's
first 128 keys and rounded to e4m3, fp32-like row sums of the unrounded P —
are emulated in fp64 with torch's float8_e4m3fn and compared with the oracle.
The bars the GPU test uses (O rel-RMS <= 0.1, max-abs <= 0.35; lse max-abs <=
0.25, RMS <= 0.03) must hold for this emulation with room to spare, and the
emulation's O error must be of the size the unit roundoff 2^-4 predicts."""

import math

import numpy as np
import pytest
import torch

import oracle
from branch_attention_speculative_gb300 import workloads as W
from tests import test_gpu_fp8 as F

if not hasattr(torch, "float8_e4m3fn"):
    pytest.skip("torch without float8_e4m3fn", allow_module_level=True)


def _e4m3(x):
    amax = float(np.abs(x).max())
    s = amax / 448.0 if amax > 0 else 1.0
    return torch.from_numpy(x / s).to(torch.float8_e4m3fn).to(torch.float64).numpy() * s


def _emulate(wl, t):
    """o, lse of the main part in the kernel's arithmetic (causal family: no
    branch keys, so this is the whole result)."""
    T, Hq, Hkv, d = wl.tokens, wl.heads_q, wl.heads_kv, wl.head_dim
    G = Hq // Hkv
    q8 = _e4m3(t["q_b"]).reshape(T, Hq, d)
    k8 = _e4m3(t["k_m"])
    v8 = _e4m3(t["v_m"])
    o = np.zeros((T, Hq, d))
    lse = np.zeros((T, Hq))
    cu = np.asarray(wl.cu_seqlens)
    for s in range(len(cu) - 1):
        a, b = int(cu[s]), int(cu[s + 1])
        for h in range(Hq):
            kh = h // G
            S = wl.scale * (q8[a:b, h] @ k8[a:b, kh].T)
            mask = np.tril(np.ones((b - a, b - a), bool))
            S = np.where(mask, S, -np.inf)
            mref = S[:, :128].max(axis=1, keepdims=True)
            P = np.exp(S - mref)
            l = P.sum(axis=1, keepdims=True)
            P8 = torch.from_numpy(P).to(torch.float8_e4m3fn).to(torch.float64).numpy()
            o[a:b, h] = (P8 @ v8[a:b, kh]) / l
            lse[a:b, h] = (mref + np.log(l))[:, 0]
    return o.reshape(1, T, Hq, d), lse.reshape(1, T, Hq)


def test_e4m3_emulation_meets_the_8bit_bars():
    wl = W.small("causal", [1024, 512], heads_q=4, heads_kv=2, head_dim=128, cp=2, seed=21)
    t = W.make_tensors(wl, device="cpu", gen_device="cpu")
    host = {k: v.float().double().numpy() for k, v in t.items() if v is not None}
    ro, rl = oracle.attention.forward(wl, host)
    eo, el = _emulate(wl, host)
    rr = float(np.sqrt(((eo - ro) ** 2).mean() / (ro ** 2).mean()))
    # three roundings at unit roundoff 2^-4 (about 3.6% RMS each) reach O
    assert 0.02 < rr < 0.5 * F.F8_O_REL_RMS + 0.03, rr
    assert np.abs(eo - ro).max() <= F.F8_O_MAX_ABS
    e = np.abs(el - rl)
    assert e.max() <= F.F8_LSE_MAX_ABS and math.sqrt((e ** 2).mean()) <= F.F8_LSE_RMS
