"""Packed zigzag chunking, virtual-rank ownership, ring schedule and Eq. 3.

Source: "Online Draft Co-Training ..." — rainbus page, prerequisites on
context parallelism (zigzag sharding gives every rank a head chunk and a tail
chunk of the sequence so causal work is balanced; packed variable-length
sequences carry no padding; ring attention circulates K/V between ranks while
queries stay put) and the five-step method, step 2 (the main sequence is
packed into zigzag chunks, each of the C ranks holds N/C tokens, each ring
step sends the local K/V on to the other C - 1 ranks); Figure 1(a) (the causal
prefix is zigzag-sharded, branch-local keys stay local); core method, the
forward CP volume V = 2(C-1)N/C * d_kv * b per rank (Eq. 3), independent of the
number and depth of branches.

Readings: each sequence of length L is cut into 2C equal chunks of L/(2C)
tokens (L must be a multiple of 2C); virtual rank r owns chunks r and
2C-1-r of every sequence; a rank's shard lists, sequence by sequence, chunk r
then chunk 2C-1-r; the packed order is the concatenation of the shards of
ranks 0..C-1.  A branch lives on the rank that owns its anchor position.  At
ring step s (0..C-1) rank r attends the main K/V shard of rank (r - s) mod C.
In Eq. 3, d_kv is the per-token K (or V) width Hkv * d and the leading 2
counts K and V.
"""

from __future__ import annotations

import numpy as np


def chunk_table(cu_seqlens, C: int):
    """List of (seq, chunk c, start, end, owner rank) in natural positions."""
    out = []
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    for s in range(len(cu) - 1):
        a, b = int(cu[s]), int(cu[s + 1])
        L = b - a
        if L % (2 * C) != 0:
            raise ValueError(f"sequence {s} length {L} is not a multiple of 2C = {2 * C}")
        n = L // (2 * C)
        for c in range(2 * C):
            out.append((s, c, a + c * n, a + (c + 1) * n, chunk_owner(c, C)))
    return out


def chunk_owner(c: int, C: int) -> int:
    return c if c < C else 2 * C - 1 - c


def rank_chunks(r: int, C: int):
    """The two chunk indices held by virtual rank r, in shard order."""
    return (r, 2 * C - 1 - r)


def token_chunk(cu_seqlens, C: int):
    """Per natural token: (chunk index within its sequence, owner rank)."""
    T = int(cu_seqlens[-1])
    chunk = np.zeros(T, dtype=np.int64)
    owner = np.zeros(T, dtype=np.int64)
    for (_, c, a, b, r) in chunk_table(cu_seqlens, C):
        chunk[a:b] = c
        owner[a:b] = r
    return chunk, owner


def packed_token_order(cu_seqlens, C: int) -> np.ndarray:
    """perm[packed index] = natural token index (rank-major zigzag shards)."""
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    order = []
    for r in range(C):
        for s in range(len(cu) - 1):
            a, b = int(cu[s]), int(cu[s + 1])
            n = (b - a) // (2 * C)
            for c in rank_chunks(r, C):
                order.extend(range(a + c * n, a + (c + 1) * n))
    return np.asarray(order, dtype=np.int64)


def rank_token_ranges(cu_seqlens, C: int, r: int):
    """Natural-position ranges [a, b) of the main tokens held by rank r."""
    return [(a, b) for (_, c, a, b, owner) in chunk_table(cu_seqlens, C) if owner == r]


def packed_anchor_order(cu_seqlens, C: int, anchors) -> np.ndarray:
    """perm[packed anchor] = natural anchor index: anchors follow their
    position's place in the packed token order."""
    perm = packed_token_order(cu_seqlens, C)
    inv = np.empty_like(perm)
    inv[perm] = np.arange(len(perm))
    key = inv[np.asarray(anchors, dtype=np.int64)]
    return np.argsort(key, kind="stable")


def ring_source(r: int, s: int, C: int) -> int:
    """Rank whose main K/V shard rank r attends at ring step s."""
    return (r - s) % C


def comm_volume_fwd(cu_seqlens, C: int, heads_kv: int, head_dim: int, elem_bytes: int):
    """Bytes of main K and V each rank receives over the C - 1 forward ring
    steps, counted from the schedule: sum over s = 1..C-1 of the shard held by
    rank (r - s) mod C.  Branch keys never move (they stay rank-local)."""
    shard = np.zeros(C, dtype=np.int64)
    for (_, _, a, b, owner) in chunk_table(cu_seqlens, C):
        shard[owner] += b - a
    vol = np.zeros(C, dtype=np.int64)
    for r in range(C):
        for s in range(1, C):
            vol[r] += 2 * shard[ring_source(r, s, C)] * heads_kv * head_dim * elem_bytes
    return vol
