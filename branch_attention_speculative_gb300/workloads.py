"""Seeded synthetic workloads for branch attention.

This module only draws inputs: sequence lengths, branch anchors and the
Q/K/V/dO tensors.  It holds none of the attention arithmetic, so both the CPU
oracle (through the tests) and the CUDA path can be fed from it.

Shapes follow the pages' draft families ("Online Draft Co-Training for
Speculative Decoding in Large-Scale, Long-Context RL Post-Training"):

* EAGLE-3 Training-Time Test (TTT, §3.2 of the report; the paperlens
  walkthrough "Wall 1"): a branch of depth D grows at every main position.
  Natural layouts: q_b [D, T, Hq, d], k_b / v_b [D, T, Hkv, d].
* DFlash / DSpark block branches (same walkthrough, "Wall 1"): each anchor
  owns B branch tokens.  Natural layouts: q_b [NA, B, Hq, d],
  k_b / v_b [NA, B, Hkv, d], anchors in the order of the ``anchors`` array.
* Plain causal main queries (no branch keys): q_b [1, T, Hq, d].

Main keys and values are always k_m / v_m [T, Hkv, d]; dO has q_b's shape.
Every tensor is drawn as fp32 N(0, 1) and rounded to bf16.
"""

from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np

FAMILY_TTT = "ttt"
FAMILY_BLOCK = "block"
FAMILY_CAUSAL = "causal"


@dataclasses.dataclass
class Workload:
    name: str
    family: str
    cu_seqlens: np.ndarray  # int64 [S + 1], packed main-token offsets
    heads_q: int
    heads_kv: int
    head_dim: int
    cp: int  # virtual context-parallel degree C (zigzag with 2C chunks)
    depth: int = 0  # TTT depth D
    block: int = 0  # block size B (DFlash / DSpark)
    anchors: Optional[np.ndarray] = None  # int64 [S * A] absolute packed positions
    seed: int = 0

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.head_dim)

    @property
    def num_seqs(self) -> int:
        return len(self.cu_seqlens) - 1

    @property
    def tokens(self) -> int:
        return int(self.cu_seqlens[-1])

    @property
    def num_anchors(self) -> int:
        return 0 if self.anchors is None else len(self.anchors)

    @property
    def anchors_per_seq(self) -> int:
        return self.num_anchors // max(self.num_seqs, 1) if self.anchors is not None else 0

    @property
    def steps(self) -> int:
        """Leading dimension of q_b / k_b / v_b (D for TTT, 1 otherwise)."""
        return self.depth if self.family == FAMILY_TTT else 1

    @property
    def rows_per_step(self) -> int:
        """Branch rows per step and head: T (TTT, causal) or NA * B (block)."""
        if self.family == FAMILY_BLOCK:
            return self.num_anchors * self.block
        return self.tokens

    def q_shape(self):
        if self.family == FAMILY_BLOCK:
            return (self.num_anchors, self.block, self.heads_q, self.head_dim)
        return (self.steps, self.tokens, self.heads_q, self.head_dim)

    def kb_shape(self):
        if self.family == FAMILY_BLOCK:
            return (self.num_anchors, self.block, self.heads_kv, self.head_dim)
        if self.family == FAMILY_TTT:
            return (self.depth, self.tokens, self.heads_kv, self.head_dim)
        return (0, self.tokens, self.heads_kv, self.head_dim)

    def km_shape(self):
        return (self.tokens, self.heads_kv, self.head_dim)

    def branch_rows(self) -> int:
        """Query-head rows: every (branch query, q-head) pair."""
        return int(np.prod(self.q_shape()[:-1]))

    def describe(self) -> dict:
        d = {
            "workload": self.name,
            "family": self.family,
            "seqlens": [int(x) for x in np.diff(self.cu_seqlens)],
            "heads_q": self.heads_q,
            "heads_kv": self.heads_kv,
            "head_dim": self.head_dim,
            "cp": self.cp,
        }
        if self.family == FAMILY_TTT:
            d["ttt_depth"] = self.depth
        if self.family == FAMILY_BLOCK:
            d["block"] = self.block
            d["anchors_per_seq"] = self.anchors_per_seq
        d["seed"] = self.seed
        return d


# --------------------------------------------------------------------------
# lengths and anchors


def draw_seqlens(rng: np.random.Generator, n: int, lo: int, hi: int, total: int,
                 multiple: int) -> np.ndarray:
    """n lengths drawn uniformly in [lo, hi], rescaled to sum to ``total``,
    rounded to ``multiple`` (the last one takes the remainder); redrawn until
    every length lies in [lo, hi]."""
    for _ in range(10000):
        x = rng.uniform(lo, hi, size=n)
        x = x / x.sum() * total
        lens = np.round(x / multiple).astype(np.int64) * multiple
        lens[-1] = total - lens[:-1].sum()
        if lens.min() >= lo and lens.max() <= hi and lens[-1] % multiple == 0:
            return lens
    raise RuntimeError("could not draw sequence lengths")


def sample_anchors(rng: np.random.Generator, cu_seqlens: np.ndarray, per_seq: int) -> np.ndarray:
    """``per_seq`` anchor positions per sequence, uniformly without
    replacement from the sequence's tokens, sorted ascending (absolute packed
    positions)."""
    out = []
    for s in range(len(cu_seqlens) - 1):
        a, b = int(cu_seqlens[s]), int(cu_seqlens[s + 1])
        if per_seq > b - a:
            raise ValueError("more anchors than tokens")
        pos = rng.choice(b - a, size=per_seq, replace=False)
        out.append(np.sort(pos) + a)
    return np.concatenate(out).astype(np.int64) if out else np.zeros(0, np.int64)


def cu_from_lens(lens) -> np.ndarray:
    return np.concatenate([[0], np.cumsum(np.asarray(lens, dtype=np.int64))]).astype(np.int64)


# --------------------------------------------------------------------------
# the five measured shapes


def config(k: int) -> Workload:
    """Workload k = 1..5 (seed k - 1)."""
    seed = k - 1
    rng = np.random.default_rng(seed)
    if k == 1:
        return Workload("eagle3_ttt_d3_L256_tiny", FAMILY_TTT, cu_from_lens([256]), 2, 1, 64,
                        cp=2, depth=3, seed=seed)
    if k == 2:
        lens = draw_seqlens(rng, 4, 4096, 12288, 32768, multiple=8)
        return Workload("eagle3_ttt_d7_varlen_4x32k", FAMILY_TTT, cu_from_lens(lens), 32, 8, 128,
                        cp=4, depth=7, seed=seed)
    if k == 3:
        cu = cu_from_lens([32768, 32768])
        anchors = sample_anchors(rng, cu, 2048)
        return Workload("dflash_block16_2x32k", FAMILY_BLOCK, cu, 32, 8, 128, cp=8, block=16,
                        anchors=anchors, seed=seed)
    if k == 4:
        cu = cu_from_lens([131072])
        anchors = sample_anchors(rng, cu, 8192)
        return Workload("dspark_block8_128k", FAMILY_BLOCK, cu, 32, 8, 128, cp=8, block=8,
                        anchors=anchors, seed=seed)
    if k == 5:
        return Workload("eagle3_ttt_d7_256k", FAMILY_TTT, cu_from_lens([262144]), 32, 8, 128,
                        cp=8, depth=7, seed=seed)
    raise ValueError(k)


def small(family: str, lens, heads_q: int = 4, heads_kv: int = 2, head_dim: int = 64, cp: int = 2,
          depth: int = 3, block: int = 4, anchors_per_seq: int = 5, seed: int = 0,
          name: Optional[str] = None) -> Workload:
    """A small workload of the given family (test sizes)."""
    rng = np.random.default_rng(1000 + seed)
    cu = cu_from_lens(lens)
    anchors = None
    if family == FAMILY_BLOCK:
        anchors = sample_anchors(rng, cu, anchors_per_seq)
    return Workload(name or f"{family}_{'_'.join(str(x) for x in lens)}", family, cu, heads_q,
                    heads_kv, head_dim, cp=cp, depth=depth if family == FAMILY_TTT else 0,
                    block=block if family == FAMILY_BLOCK else 0, anchors=anchors, seed=seed)


# --------------------------------------------------------------------------
# tensors

TENSOR_ORDER = ("q_b", "k_m", "v_m", "k_b", "v_b", "d_o")


def tensor_shapes(wl: Workload) -> dict:
    return {
        "q_b": wl.q_shape(),
        "k_m": wl.km_shape(),
        "v_m": wl.km_shape(),
        "k_b": wl.kb_shape(),
        "v_b": wl.kb_shape(),
        "d_o": wl.q_shape(),
    }


def make_tensors(wl: Workload, device="cpu", gen_device: Optional[str] = None) -> dict:
    """Draw q_b, k_m, v_m, k_b, v_b, d_o (in that order) as fp32 N(0,1) from
    one torch generator seeded with ``wl.seed`` on ``gen_device``, rounded to
    bf16 and placed on ``device``.  Tensors with a leading step/anchor
    dimension are drawn one leading slice at a time, which bounds the fp32
    temporary.  The values depend on ``gen_device`` (the CPU and CUDA
    generators differ); by default small workloads are drawn on the CPU."""
    import torch

    shapes = tensor_shapes(wl)
    total = sum(int(np.prod(s)) for s in shapes.values())
    if gen_device is None:
        gen_device = "cpu" if total <= (1 << 26) else str(device)
    g = torch.Generator(device=gen_device)
    g.manual_seed(int(wl.seed))
    out = {}
    for name in TENSOR_ORDER:
        shp = shapes[name]
        t = torch.empty(shp, dtype=torch.bfloat16, device=device)
        if len(shp) == 4 and shp[0] > 0:
            for i in range(shp[0]):
                x = torch.randn(shp[1:], generator=g, device=gen_device, dtype=torch.float32)
                t[i].copy_(x.to(torch.bfloat16))
                del x
        elif int(np.prod(shp)) > 0:
            x = torch.randn(shp, generator=g, device=gen_device, dtype=torch.float32)
            t.copy_(x.to(torch.bfloat16))
            del x
        out[name] = t
    return out
