"""Host-side checks of libba.so (no GPU launch): the exported C ABI, the
planner's zigzag tables against the oracle's, useful-pair counts, Eq. 3, and
descriptor validation."""

import ctypes
import re
import os

import numpy as np
import pytest

import oracle
from branch_attention_speculative_gb300 import build as B
from branch_attention_speculative_gb300 import workloads as W

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def api():
    B.build()
    from branch_attention_speculative_gb300 import api as A
    return A


def header_symbols():
    txt = open(os.path.join(ROOT, "include", "ba.h")).read()
    txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
    return sorted(set(re.findall(r"\b(ba_[a-z0-9_]+)\s*\(", txt)))


def test_library_exports_every_header_symbol(api):
    lib = ctypes.CDLL(api.LIB_PATH)
    syms = header_symbols()
    assert len(syms) >= 12
    for s in syms:
        assert hasattr(lib, s), s
    assert sorted(api.exported_symbols()) == syms
    assert api.version().endswith("sm_103a")


def _cases():
    return [W.config(1), W.config(2), W.config(3),
            W.small("ttt", [16, 32, 48], cp=4, depth=2),
            W.small("block", [64, 32], cp=2, block=4, anchors_per_seq=9, seed=3),
            W.small("causal", [24, 8], cp=2)]


@pytest.mark.parametrize("wl", _cases(), ids=lambda w: w.name)
def test_zigzag_tables_match_oracle(api, wl):
    p = api.Plan.from_workload(wl)
    perm = oracle.zigzag.packed_token_order(wl.cu_seqlens, wl.cp)
    assert np.array_equal(p.table("token_perm"), perm)
    _, owner = oracle.zigzag.token_chunk(wl.cu_seqlens, wl.cp)
    assert np.array_equal(p.table("token_rank"), owner)
    if wl.family == "block":
        ap = oracle.zigzag.packed_anchor_order(wl.cu_seqlens, wl.cp, wl.anchors)
        assert np.array_equal(p.table("anchor_perm"), ap)
        lim = np.repeat(np.asarray(wl.anchors)[ap], wl.block)
    else:
        lim = perm
    assert np.array_equal(p.table("row_limit"), lim)


def test_anchor_tables_match_hand_worked_golden(api):
    from tests import oracle_pins as P
    rows = P.parse_golden(os.path.join(ROOT, "tests", "golden", "zigzag_anchors_c2.txt"))
    for r in rows:
        ints = lambda tok: np.array([int(x) for x in tok.split(";")], dtype=np.int32)
        cu, anchors, order, lim = ints(r[1]), ints(r[2]), ints(r[3]), ints(r[4])
        S = len(cu) - 1
        p = api.Plan("block", cu, 2, 1, 64, 2, block_size=3, anchors=anchors)
        assert len(anchors) % S == 0
        assert np.array_equal(p.table("anchor_perm"), order)
        assert np.array_equal(p.table("row_limit"), np.repeat(lim, 3))


@pytest.mark.parametrize("wl", _cases(), ids=lambda w: w.name)
def test_useful_pairs_and_eq3_match_oracle(api, wl):
    p = api.Plan.from_workload(wl)
    inf = p.info()
    if wl.tokens <= 4096:
        assert inf["main_pairs"] + inf["branch_pairs"] == oracle.attention.useful_pairs(wl)
    vol = oracle.zigzag.comm_volume_fwd(wl.cu_seqlens, wl.cp, wl.heads_kv, wl.head_dim, 2)
    assert np.array_equal(p.comm_volume(), vol)
    assert inf["fwd_flops"] == 4 * wl.head_dim * (inf["main_pairs"] + inf["branch_pairs"])


@pytest.mark.parametrize("k", [1, 2, 3, 4, 5])
def test_measured_shape_plans_validate(api, k):
    api.Plan.from_workload(W.config(k)).validate()


@pytest.mark.parametrize("wl", _cases(), ids=lambda w: w.name)
def test_small_plans_validate(api, wl):
    api.Plan.from_workload(wl).validate()


def test_comm_volume_does_not_depend_on_branches(api):
    # Eq. 3: the same main sequence with and without branches moves the same bytes
    lens = [64, 128]
    vols = []
    for fam, kw in (("causal", {}), ("ttt", {"depth": 5}), ("block", {"block": 8, "anchors_per_seq": 7})):
        wl = W.small(fam, lens, cp=4, **kw)
        vols.append(api.Plan.from_workload(wl).comm_volume())
    assert all(np.array_equal(v, vols[0]) for v in vols)


def test_config5_pairs_closed_form(api):
    wl = W.config(5)
    inf = api.Plan.from_workload(wl).info()
    T = wl.tokens
    assert inf["main_pairs"] == 32 * 7 * (T * (T + 1) // 2)
    assert inf["branch_pairs"] == 32 * (7 * 8 // 2) * T


@pytest.mark.parametrize("bad", [
    dict(cp=3),                       # 256 not a multiple of 6
    dict(heads_q=3, heads_kv=2),      # not a GQA group
    dict(head_dim=0),
    dict(depth=0),
    dict(depth=17),
])
def test_bad_descriptors_rejected(api, bad):
    kw = dict(family="ttt", cu_seqlens=[0, 256], heads_q=2, heads_kv=1, head_dim=64, cp=2, ttt_depth=3)
    if "depth" in bad:
        kw["ttt_depth"] = bad.pop("depth")
    kw.update(bad)
    with pytest.raises(api.BaError) as e:
        api.Plan(**kw)
    assert e.value.code == -1


def test_unsupported_head_dim(api):
    with pytest.raises(api.BaError) as e:
        api.Plan("ttt", [0, 256], 2, 1, 96, 2, ttt_depth=3)
    assert e.value.code == -2


@pytest.mark.parametrize("anchors", [[5, 5, 9], [9, 5, 1], [0, 3, 64]])
def test_bad_anchors_rejected(api, anchors):
    with pytest.raises(api.BaError) as e:
        api.Plan("block", [0, 64], 2, 1, 64, 2, block_size=4, anchors=anchors)
    assert e.value.code == -1


def test_null_and_misaligned_pointers_rejected_before_launch(api):
    lib = api.lib()
    p = api.Plan("ttt", [0, 64], 2, 1, 64, 2, ttt_depth=2)
    rc = lib.ba_forward(p._h, None, None, None, None, None, None, None, None, 0, None)
    assert rc == -1
    rc = lib.ba_forward(p._h, *([ctypes.c_void_p(0x1001)] * 7), ctypes.c_void_p(0x1000), 1 << 30, None)
    assert rc == -1
    # aligned pointers but no workspace
    rc = lib.ba_forward(p._h, *([ctypes.c_void_p(0x1000)] * 7), None, 0, None)
    assert rc == -6
    assert lib.ba_lse_merge(4, 96, None, None, None, None, None, None, None) == -1


def test_step_and_8bit_arguments_rejected_before_launch(api):
    """The per-step TTT calls and the 8-bit forward check their arguments before
    anything is enqueued (fake, aligned, never dereferenced pointers)."""
    lib = api.lib()
    ptr = ctypes.c_void_p(0x1000)
    ttt = api.Plan("ttt", [0, 64], 2, 1, 64, 2, ttt_depth=2)
    for step in (-1, 2, 7):  # slots are 0 .. depth - 1
        assert lib.ba_forward_step(ttt._h, step, *([ptr] * 7), ptr, 1 << 30, None) == -1
        assert lib.ba_backward_step(ttt._h, step, *([ptr] * 14), 1 << 30, None) == -1
    block = api.Plan("block", [0, 64], 2, 1, 64, 2, block_size=4, anchors=[3, 40])
    assert lib.ba_forward_step(block._h, 0, *([ptr] * 7), ptr, 1 << 30, None) == -1
    assert lib.ba_backward_step(block._h, 0, *([ptr] * 14), 1 << 30, None) == -1
    # a valid step with a null input, a misaligned output, no workspace
    assert lib.ba_forward_step(ttt._h, 1, None, *([ptr] * 6), ptr, 1 << 30, None) == -1
    assert lib.ba_forward_step(ttt._h, 1, *([ptr] * 5), ctypes.c_void_p(0x1004), ptr, ptr, 1 << 30, None) == -1
    assert lib.ba_forward_step(ttt._h, 1, *([ptr] * 7), None, 0, None) == -6
    # the 8-bit forward is built for head_dim 128 only
    assert lib.ba_forward_fp8(ttt._h, *([ptr] * 7), ptr, 1 << 40, None) == -2


# ---------------------------------------------------------------- the main-attention schedule
#
# The kernels see the main part only through the planner's tile tables.  These
# checks rebuild, from those tables alone, which (query row, main key) pairs
# the forward and the backward visit, and compare the result with the
# oracle's main-key mask: every visible pair exactly once, nothing else.


def _schedule_cases():
    return [W.config(1),
            W.small("ttt", [200, 56, 320], heads_q=4, heads_kv=2, head_dim=64, cp=2, depth=3, seed=1),
            W.small("ttt", [1280, 768], heads_q=8, heads_kv=2, head_dim=128, cp=2, depth=2, seed=7),
            W.small("ttt", [16, 32, 48], cp=4, depth=2),
            W.small("block", [1536, 512], heads_q=8, heads_kv=2, head_dim=128, cp=2, block=16, anchors_per_seq=40,
                    seed=8),
            W.small("block", [96, 32, 160], heads_q=4, heads_kv=2, head_dim=64, cp=4, block=3, anchors_per_seq=7,
                    seed=4),
            W.small("causal", [136, 8, 256], heads_q=4, heads_kv=4, head_dim=64, cp=2, seed=5)]


def _stream_rows(wl):
    return wl.num_anchors * wl.block if wl.family == "block" else wl.tokens


def _expected_cover(wl):
    n = _stream_rows(wl)
    return oracle.keysets.main_mask(wl, np.arange(n), np.arange(wl.tokens)).astype(np.int32)


def _tile_rows(tile, row_limit):
    row0, nrows, nrow0 = int(tile[0]), int(tile[1]), int(tile[8])
    lim = row_limit[row0:row0 + nrows]
    assert tile[4] == lim.min() and tile[5] == lim.max()
    return nrow0 + np.arange(nrows), lim


def _forward_cover(wl, lim, fq, fs):
    """(row, key) visit counts of the forward tables; asserts the per-segment rules."""
    cover = np.zeros((_stream_rows(wl), wl.tokens), dtype=np.int32)
    for tile in fq:
        rows, rl = _tile_rows(tile, lim)
        assert 0 < len(rows) <= 128
        for k0, nkeys, pos0, diag in fs[tile[2]:tile[2] + tile[3]]:
            keys = pos0 + np.arange(nkeys)
            vis = keys[None, :] <= rl[:, None]
            if diag:
                assert vis.any()  # fully masked (tile, segment) pairs are dropped
            else:
                assert vis.all()  # an unmasked segment is below every row limit
            cover[rows[:, None], keys[None, :]] += vis
    return cover


def _backward_cover(wl, lim, bq, bkv, br):
    """(row, key) visit counts of the backward tables."""
    cover = np.zeros((_stream_rows(wl), wl.tokens), dtype=np.int32)
    for k0, nkeys, pos0, qr0, nqr in bkv[:, :5]:
        assert 0 <= nkeys <= 128
        if nkeys == 0:  # a filler that completes a cluster owns no keys
            continue
        keys = pos0 + np.arange(nkeys)
        for t0, t1, diag, _ in br[qr0:qr0 + nqr]:
            for t in range(t0, t1):
                rows, rl = _tile_rows(bq[t], lim)
                assert 0 < len(rows) <= 128
                vis = keys[None, :] <= rl[:, None]
                if not diag:
                    assert vis.all()
                cover[rows[:, None], keys[None, :]] += vis
    return cover


def _fwd_tables(p):
    return p.table("row_limit"), p.table("fwd_qtiles").reshape(-1, 10), p.table("fwd_segs").reshape(-1, 4)


def _bwd_tables(p):
    return (p.table("row_limit"), p.table("bwd_qtiles").reshape(-1, 10), p.table("bwd_kvtiles").reshape(-1, 8),
            p.table("bwd_qranges").reshape(-1, 4))


@pytest.mark.parametrize("wl", _schedule_cases(), ids=lambda w: w.name)
def test_forward_schedule_covers_each_visible_pair_once(api, wl):
    p = api.Plan.from_workload(wl)
    assert np.array_equal(_forward_cover(wl, *_fwd_tables(p)), _expected_cover(wl))


@pytest.mark.parametrize("wl", _schedule_cases(), ids=lambda w: w.name)
def test_backward_schedule_covers_each_visible_pair_once(api, wl):
    p = api.Plan.from_workload(wl)
    assert np.array_equal(_backward_cover(wl, *_bwd_tables(p)), _expected_cover(wl))


def _schedule_check_fails(fn):
    try:
        return not fn()
    except AssertionError:
        return True


def test_schedule_checks_catch_planted_mistakes(api):
    """Each planted table mistake (in a copy of the tables, on the host) makes
    the coverage checks fail, so they would catch it in the planner."""
    wl = W.small("ttt", [1280, 768], heads_q=8, heads_kv=2, head_dim=128, cp=2, depth=2, seed=7)
    p = api.Plan.from_workload(wl)
    want = _expected_cover(wl)
    lim, fq, fs = _fwd_tables(p)
    ok = lambda lim_, fq_, fs_: np.array_equal(_forward_cover(wl, lim_, fq_, fs_), want)
    assert ok(lim, fq, fs)
    # a segment dropped from a tile's list
    fq2 = fq.copy()
    t = int(np.argmax(fq2[:, 3]))
    fq2[t, 3] -= 1
    assert _schedule_check_fails(lambda: ok(lim, fq2, fs))
    # a diagonal segment marked unmasked
    fs2 = fs.copy()
    fs2[np.nonzero(fs2[:, 3])[0][0], 3] = 0
    assert _schedule_check_fails(lambda: ok(lim, fq, fs2))
    # a segment shifted by one key
    fs3 = fs.copy()
    fs3[0, 2] += 1
    assert _schedule_check_fails(lambda: ok(lim, fq, fs3))
    lim, bq, bkv, br = _bwd_tables(p)
    okb = lambda bkv_, br_: np.array_equal(_backward_cover(wl, lim, bq, bkv_, br_), want)
    assert okb(bkv, br)
    # a key tile that loses its last query range
    bkv2 = bkv.copy()
    t = int(np.argmax(bkv2[:, 4]))
    bkv2[t, 4] -= 1
    assert _schedule_check_fails(lambda: okb(bkv2, br))
    # a key tile one key short
    bkv3 = bkv.copy()
    bkv3[np.nonzero(bkv3[:, 1])[0][0], 1] -= 1
    assert _schedule_check_fails(lambda: okb(bkv3, br))
