"""The dK/dV kernel's packed bf16x2 arithmetic against the gradient bar
(CPU, no GPU).  The kernel forms P^T two elements at a time: the exponent
s * scale * log2(e) - lse * log2(e) in fp32, rounded to bf16, then 2^x rounded
to bf16; and dS^T = P^T (dP^T - Delta) as the fp32 difference rounded to bf16
times P^T in bf16, rounded to bf16.  Those roundings are emulated in fp64 with
torch's bfloat16 on one causal head and the resulting dK and dV are compared
with the exact fp64 gradients of the same bf16 inputs: the error must sit
well inside the GPU tests' bar (rel-RMS <= 2e-2) and be of the size a few
bf16 roundings (unit roundoff 2^-8) predict."""

import numpy as np
import torch

import oracle
from tests.gpu_support import GRAD_REL_RMS, rel_rms

LOG2E = 1.0 / np.log(2.0)


def _bf16(x):
    return torch.from_numpy(np.ascontiguousarray(x)).to(torch.bfloat16).to(torch.float64).numpy()


def _f32(x):
    return np.asarray(x, dtype=np.float32).astype(np.float64)


def _emulate_kv(q, k, v, do, mask, scale, o, lse):
    """dK, dV with the kernel's roundings (fp32 accumulations, bf16 operands)."""
    s = _f32(q @ k.T)                                   # S from the MMA, fp32
    nl = _f32(-lse * LOG2E)                             # the row record's -lse*log2e
    x = _bf16(_f32(s * _f32(scale * LOG2E) + nl[:, None]))
    p = np.where(mask, _bf16(np.exp2(x)), 0.0)          # ex2 in bf16x2, masked
    dp = _f32(do @ v.T)                                 # dP from the MMA, fp32
    delta = _f32((do * o).sum(axis=1))                  # the row record's Delta
    ds = np.where(mask, _bf16(p * _bf16(_f32(dp - delta[:, None]))), 0.0)
    dv = p.T @ do                                       # dV += P^T dO (fp32 accumulation)
    dk = scale * (ds.T @ q)                             # dK += dS^T Q, scaled at the end
    return dk, dv


def test_packed_bf16_arithmetic_meets_the_gradient_bar():
    rng = np.random.default_rng(31)
    n, d = 640, 128
    q, k, v, do = (_bf16(rng.standard_normal((n, d))) for _ in range(4))
    scale = 1.0 / np.sqrt(d)
    mask = np.tril(np.ones((n, n), dtype=bool))
    o, lse = oracle.attention.masked_attention_fwd(q, k, v, mask, scale)
    _, dk_ref, dv_ref = oracle.attention.masked_attention_bwd(q, k, v, mask, scale, o, lse, do)
    dk, dv = _emulate_kv(q, k, v, do, mask, scale, o, lse)
    rk, rv = rel_rms(dk, dk_ref), rel_rms(dv, dv_ref)
    # a few roundings at 2^-8 relative: well below the bar, and not zero
    assert 1e-4 < rv < 0.5 * GRAD_REL_RMS, rv
    assert 1e-4 < rk < 0.5 * GRAD_REL_RMS, rk
