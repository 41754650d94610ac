// Host planner for branch attention.
//
// Zigzag layout ("Online Draft Co-Training ...", rainbus page, CP
// prerequisites and method step 2; Figure 1(a)): every sequence of length L
// is cut into 2C chunks of L/(2C) tokens; virtual rank r holds chunks r and
// 2C-1-r of every sequence, in that order, sequence by sequence, and the
// packed order concatenates the shards of ranks 0..C-1.  A branch lives on
// the rank that owns its anchor position (same page, Figure 1(a): branch-local
// keys stay local).  Ring order: at step s rank r attends the main K/V shard of
// rank (r - s) mod C (ai.info summary, "Methodology in Plain English": K/V
// circulate while queries stay put); the backward replays the ring (rainbus
// page, method step 5), so the key shard of rank r meets the queries of rank
// (r + s) mod C at step s.  Eq. 3 (rainbus page, core method): the forward
// volume per rank is 2(C-1)(T/C) d_kv b, whatever the branches.
//
// On one GPU the ranks are virtual: the planner turns the schedule into tile
// lists.  A forward query tile lists the key segments it visits in ring order
// (chunk pairs above the diagonal are dropped, pairs below are unmasked, the
// diagonal pair is cut at the tile's largest row limit); a backward key tile
// lists the query-tile ranges that the ring replay brings to it (unmasked
// chunks first in a canonical order, the diagonal chunk last).  Tiles are
// handed out longest first.
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstring>
#include <limits>
#include <new>

#include "plan.h"

namespace {

std::atomic<uint64_t> g_next_plan_id{1};

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

int owner_of_chunk(int c, int C) { return c < C ? c : 2 * C - 1 - c; }

template <class T>
size_t table_span(const std::vector<T>& v) { return align256(std::max<size_t>(v.size() * sizeof(T), 16)); }

template <class T>
void put(std::vector<unsigned char>& img, size_t off, const std::vector<T>& v) {
  if (!v.empty()) std::memcpy(img.data() + off, v.data(), v.size() * sizeof(T));
}

}  // namespace

int ba_build_plan(const ba_plan_desc* d, ba_plan* p) {
  if (!d || !p) return BA_ERR_INVALID_ARG;
  const int fam = d->family;
  if (fam != BA_FAMILY_TTT && fam != BA_FAMILY_BLOCK && fam != BA_FAMILY_CAUSAL) return BA_ERR_INVALID_ARG;
  if (d->num_seqs < 1 || !d->cu_seqlens) return BA_ERR_INVALID_ARG;
  if (d->heads_q < 1 || d->heads_kv < 1 || d->heads_q % d->heads_kv != 0) return BA_ERR_INVALID_ARG;
  if (d->head_dim < 1) return BA_ERR_INVALID_ARG;
  if (d->head_dim != 64 && d->head_dim != 128) return BA_ERR_UNSUPPORTED;
  if (!(d->softmax_scale > 0.f) || !std::isfinite(d->softmax_scale)) return BA_ERR_INVALID_ARG;
  const int C = d->cp_degree;
  if (C < 1 || C > 64) return BA_ERR_INVALID_ARG;
  const int S = d->num_seqs;
  if (d->cu_seqlens[0] != 0) return BA_ERR_INVALID_ARG;
  for (int s = 0; s < S; ++s) {
    const int64_t len = int64_t(d->cu_seqlens[s + 1]) - d->cu_seqlens[s];
    if (len <= 0 || len % (2 * C) != 0) return BA_ERR_INVALID_ARG;
  }
  const int64_t T = d->cu_seqlens[S];
  int D = 1, B = 1, A = 0;
  if (fam == BA_FAMILY_TTT) {
    D = d->ttt_depth;
    if (D < 1 || D > 16) return BA_ERR_INVALID_ARG;
  }
  if (fam == BA_FAMILY_BLOCK) {
    B = d->block_size;
    A = d->anchors_per_seq;
    if (B < 1 || B > 64 || A < 1 || !d->anchors) return BA_ERR_INVALID_ARG;
    for (int s = 0; s < S; ++s) {
      for (int i = 0; i < A; ++i) {
        const int32_t a = d->anchors[int64_t(s) * A + i];
        if (a < d->cu_seqlens[s] || a >= d->cu_seqlens[s + 1]) return BA_ERR_INVALID_ARG;
        if (i > 0 && a <= d->anchors[int64_t(s) * A + i - 1]) return BA_ERR_INVALID_ARG;
      }
    }
  }
  const int64_t NA = fam == BA_FAMILY_BLOCK ? int64_t(S) * A : 0;
  const int64_t rows = fam == BA_FAMILY_BLOCK ? NA * B : T;
  if (rows > std::numeric_limits<int32_t>::max() / 2) return BA_ERR_INVALID_ARG;

  p->id = g_next_plan_id.fetch_add(1);
  p->cu.assign(d->cu_seqlens, d->cu_seqlens + S + 1);
  if (fam == BA_FAMILY_BLOCK) p->anchors.assign(d->anchors, d->anchors + NA);
  p->C = C;
  p->S = S;
  p->NA = NA;
  BaShape& sh = p->shape;
  sh.family = fam;
  sh.Hq = d->heads_q;
  sh.Hkv = d->heads_kv;
  sh.G = d->heads_q / d->heads_kv;
  sh.d = d->head_dim;
  sh.steps = fam == BA_FAMILY_TTT ? D : 1;
  sh.B = fam == BA_FAMILY_BLOCK ? B : 1;
  sh.nbk = fam == BA_FAMILY_TTT ? D : (fam == BA_FAMILY_BLOCK ? B : 0);
  sh.step0 = 0;
  sh.T = T;
  sh.rows = rows;
  sh.units = fam == BA_FAMILY_BLOCK ? NA : T;
  sh.scale = d->softmax_scale;
  sh.scale_log2 = float(double(d->softmax_scale) * 1.4426950408889634);

  // ---- chunks and the packed token order
  const int nch = 2 * C;
  p->chunks.assign(size_t(S) * nch, BaChunk{});
  for (int s = 0; s < S; ++s) {
    const int32_t len = (p->cu[s + 1] - p->cu[s]) / nch;
    for (int c = 0; c < nch; ++c) {
      BaChunk& ch = p->chunks[size_t(s) * nch + c];
      ch.seq = s;
      ch.c = c;
      ch.rank = owner_of_chunk(c, C);
      ch.nat0 = p->cu[s] + c * len;
      ch.len = len;
    }
  }
  std::vector<int32_t> chunk_order;  // global chunk ids in packed order
  chunk_order.reserve(p->chunks.size());
  {
    int32_t pk = 0;
    for (int r = 0; r < C; ++r)
      for (int s = 0; s < S; ++s)
        for (int c : {r, nch - 1 - r}) {
          BaChunk& ch = p->chunks[size_t(s) * nch + c];
          ch.pk0 = pk;
          pk += ch.len;
          chunk_order.push_back(s * nch + c);
        }
  }
  p->tok_perm.assign(T, 0);
  p->tok_rank.assign(T, 0);
  std::vector<int32_t> inv_tok(T);
  for (const BaChunk& ch : p->chunks)
    for (int32_t i = 0; i < ch.len; ++i) {
      p->tok_perm[ch.pk0 + i] = ch.nat0 + i;
      inv_tok[ch.nat0 + i] = ch.pk0 + i;
      p->tok_rank[ch.nat0 + i] = ch.rank;
    }

  // ---- packed query rows and their key limits
  p->row_lim.assign(rows, 0);
  if (fam != BA_FAMILY_BLOCK) {
    for (BaChunk& ch : p->chunks) {
      ch.row0 = ch.pk0;
      ch.nrows = ch.len;
    }
    for (int64_t r = 0; r < T; ++r) p->row_lim[r] = p->tok_perm[r];
  } else {
    p->anc_perm.resize(NA);
    for (int64_t a = 0; a < NA; ++a) p->anc_perm[a] = int32_t(a);
    std::stable_sort(p->anc_perm.begin(), p->anc_perm.end(), [&](int32_t x, int32_t y) {
      return inv_tok[p->anchors[x]] < inv_tok[p->anchors[y]];
    });
    for (BaChunk& ch : p->chunks) { ch.row0 = -1; ch.nrows = 0; }
    // chunk of a natural position: sequence by cu, then offset / len
    auto chunk_of = [&](int32_t pos) -> BaChunk& {
      const int s = int(std::upper_bound(p->cu.begin(), p->cu.end(), pos) - p->cu.begin()) - 1;
      const int32_t len = (p->cu[s + 1] - p->cu[s]) / nch;
      return p->chunks[size_t(s) * nch + (pos - p->cu[s]) / len];
    };
    for (int64_t ap = 0; ap < NA; ++ap) {
      const int32_t pos = p->anchors[p->anc_perm[ap]];
      BaChunk& ch = chunk_of(pos);
      if (ch.row0 < 0) ch.row0 = int32_t(ap * B);
      ch.nrows += B;
      for (int u = 0; u < B; ++u) p->row_lim[ap * B + u] = pos;
    }
    // empty chunks: place them at the row where they would start
    int32_t next = 0;
    for (int32_t gid : chunk_order) {
      BaChunk& ch = p->chunks[gid];
      if (ch.row0 < 0) ch.row0 = next;
      next = ch.row0 + ch.nrows;
    }
  }

  // natural row -> limit (TTT / causal: the row's own position; block: its anchor)
  p->nat_lim.assign(rows, 0);
  if (fam != BA_FAMILY_BLOCK) {
    for (int64_t r = 0; r < T; ++r) p->nat_lim[r] = int32_t(r);
  } else {
    for (int64_t a = 0; a < NA; ++a)
      for (int u = 0; u < B; ++u) p->nat_lim[a * B + u] = p->anchors[a];
  }
  auto natural_row = [&](int32_t r) -> int32_t {
    return fam == BA_FAMILY_BLOCK ? p->anc_perm[r / B] * B + r % B : p->tok_perm[r];
  };

  // ---- useful pairs
  p->main_pairs = 0;
  for (const BaChunk& ch : p->chunks) {
    const int32_t start = p->cu[ch.seq];
    for (int32_t r = ch.row0; r < ch.row0 + ch.nrows; ++r) p->main_pairs += int64_t(p->row_lim[r]) - start + 1;
  }
  p->main_pairs *= int64_t(sh.Hq) * sh.steps;
  if (fam == BA_FAMILY_TTT) p->branch_pairs = int64_t(D) * (D + 1) / 2 * T * sh.Hq;
  else if (fam == BA_FAMILY_BLOCK) p->branch_pairs = NA * B * B * sh.Hq;
  else p->branch_pairs = 0;

  // ---- forward query tiles and their key segments (ring order)
  auto make_qtiles = [&](int BM, std::vector<BaQTile>& out, std::vector<int32_t>* first, std::vector<int32_t>* count) {
    out.clear();
    if (first) first->assign(p->chunks.size(), 0);
    if (count) count->assign(p->chunks.size(), 0);
    for (int32_t gid : chunk_order) {
      const BaChunk& ch = p->chunks[gid];
      if (first) (*first)[gid] = int32_t(out.size());
      for (int32_t r0 = ch.row0; r0 < ch.row0 + ch.nrows; r0 += BM) {
        BaQTile t{};
        t.row0 = r0;
        t.nrows = std::min(BM, ch.row0 + ch.nrows - r0);
        t.lim_min = p->row_lim[r0];
        t.lim_max = p->row_lim[r0 + t.nrows - 1];
        t.chunk = gid;
        t.nrow0 = natural_row(r0);
        out.push_back(t);
      }
      if (count) (*count)[gid] = int32_t(out.size()) - (*first)[gid];
    }
  };
  make_qtiles(BA_FWD_BM, p->fq, nullptr, nullptr);
  p->fseg.clear();
  p->fwd_blocks = 0;
  for (BaQTile& t : p->fq) {
    const BaChunk& qch = p->chunks[t.chunk];
    t.seg0 = int32_t(p->fseg.size());
    t.work = 0;
    for (int step = 0; step < C; ++step) {
      const int src = ((qch.rank - step) % C + C) % C;
      for (int kc : {src, nch - 1 - src}) {
        const BaChunk& kch = p->chunks[size_t(qch.seq) * nch + kc];
        BaKvSeg sg{};
        if (kc < qch.c) {
          sg = BaKvSeg{kch.pk0, kch.len, kch.nat0, 0};
        } else if (kc == qch.c) {
          const int32_t nk = t.lim_max - kch.nat0 + 1;
          sg = BaKvSeg{kch.pk0, nk, kch.nat0, t.lim_min < kch.nat0 + nk - 1 ? 1 : 0};
        } else {
          continue;
        }
        p->fseg.push_back(sg);
        t.work += (sg.nkeys + BA_FWD_BN - 1) / BA_FWD_BN;
      }
    }
    t.nseg = int32_t(p->fseg.size()) - t.seg0;
    p->fwd_blocks += t.work;
  }
  p->forder.resize(p->fq.size());
  for (size_t i = 0; i < p->fq.size(); ++i) p->forder[i] = int32_t(i);
  std::stable_sort(p->forder.begin(), p->forder.end(),
                   [&](int32_t x, int32_t y) { return p->fq[x].work > p->fq[y].work; });

  // ---- backward key tiles and the query ranges that see them (ring replay)
  std::vector<int32_t> bfirst, bcount;
  make_qtiles(BA_BWD_BM, p->bq, &bfirst, &bcount);
  p->bkv.clear();
  p->bqr.clear();
  std::vector<int32_t> gwork;  // per group of BA_BWD_CS key tiles
  for (int32_t gid : chunk_order) {
    const BaChunk& kch = p->chunks[gid];
    const int32_t ntiles = (kch.len + BA_BWD_BN - 1) / BA_BWD_BN;
    for (int32_t g0 = 0; g0 < ntiles; g0 += BA_BWD_CS) {
      // The query chunks a key tile meets are those the ring replay brings to
      // it (rank (r + s) mod C at step s): every later chunk of the sequence,
      // unmasked, and its own chunk, cut by the causal limit.  They are listed
      // unmasked chunks first, in descending chunk order — a prefix shared by
      // every key tile of the sequence — and the diagonal chunk last.  The
      // tiles of a group share one list: on the diagonal chunk it starts at the
      // first query tile that sees the group's first (lowest) key, so it holds
      // every query tile any member sees; the per-row limits mask the rest.
      // Only the summation order of dK / dV depends on the order.
      const int32_t gpos0 = kch.nat0 + g0 * BA_BWD_BN;
      const int32_t qr0 = int32_t(p->bqr.size());
      int32_t work = 0;
      for (int qc = nch - 1; qc >= kch.c; --qc) {
        const int32_t qg = kch.seq * nch + qc;
        int32_t t0 = bfirst[qg], t1 = bfirst[qg] + bcount[qg];
        int diag = 0;
        if (qc == kch.c) {
          while (t0 < t1 && p->bq[t0].lim_max < gpos0) ++t0;
          diag = 1;
        }
        if (t0 >= t1) continue;
        p->bqr.push_back(BaQRange{t0, t1, diag, 0});
        work += t1 - t0;
      }
      const int32_t nqr = int32_t(p->bqr.size()) - qr0;
      for (int32_t m = 0; m < BA_BWD_CS; ++m) {
        const int32_t t = g0 + m;
        BaKvTile kt{};
        if (t < ntiles) {
          kt.k0 = kch.pk0 + t * BA_BWD_BN;
          kt.nkeys = std::min(BA_BWD_BN, kch.len - t * BA_BWD_BN);
          kt.pos0 = kch.nat0 + t * BA_BWD_BN;
        } else {  // filler: no keys; loads point at the chunk's first tile
          kt.k0 = kch.pk0;
          kt.nkeys = 0;
          kt.pos0 = kch.nat0;
        }
        kt.chunk = gid;
        kt.qr0 = qr0;
        kt.nqr = nqr;
        kt.work = work;
        // kept even when no query sees it: its dK / dV must still be written (as zeros)
        p->bkv.push_back(kt);
      }
      gwork.push_back(work);
    }
  }
  // groups longest first; the members of a group stay consecutive
  std::vector<int32_t> gorder(gwork.size());
  for (size_t g = 0; g < gwork.size(); ++g) gorder[g] = int32_t(g);
  std::stable_sort(gorder.begin(), gorder.end(), [&](int32_t x, int32_t y) { return gwork[x] > gwork[y]; });
  p->border.clear();
  for (int32_t g : gorder)
    for (int32_t m = 0; m < BA_BWD_CS; ++m) p->border.push_back(g * BA_BWD_CS + m);

  // ---- Eq. 3 volume from the schedule
  std::vector<int64_t> shard(C, 0);
  for (const BaChunk& ch : p->chunks) shard[ch.rank] += ch.len;
  p->comm.assign(C, 0);
  for (int r = 0; r < C; ++r)
    for (int step = 1; step < C; ++step)
      p->comm[r] += 2 * shard[((r - step) % C + C) % C] * sh.Hkv * sh.d * 2;

  // ---- workspace layout
  BaWorkspaceLayout& w = p->ws;
  size_t off = 0;
  w.status = off;
  off += 256;
  w.tables = off;
  size_t t = 0;
  w.t_row_lim = t; t += table_span(p->row_lim);
  w.t_nat_lim = t; t += table_span(p->nat_lim);
  w.t_tok_perm = t; t += table_span(p->tok_perm);
  w.t_anc_perm = t; t += table_span(p->anc_perm);
  w.t_fq = t; t += table_span(p->fq);
  w.t_fseg = t; t += table_span(p->fseg);
  w.t_forder = t; t += table_span(p->forder);
  w.t_bq = t; t += table_span(p->bq);
  w.t_bkv = t; t += table_span(p->bkv);
  w.t_bqr = t; t += table_span(p->bqr);
  w.t_border = t; t += table_span(p->border);
  w.table_bytes = t;
  off += t;
  const size_t qrows = size_t(sh.steps) * size_t(rows) * size_t(sh.Hq);
  const size_t dd = size_t(sh.d);
  // The kernels read the caller's natural-layout tensors directly and finish
  // every output row in their epilogues, so the workspace holds only the
  // backward's row records.
  w.rowrec = off;
  off = align256(off + qrows * 16);
  w.total = off;
  size_t g = align256(w.total);
  w.f8_amax = g; g += 256;
  w.f8_q = g; g = align256(g + qrows * dd);
  w.f8_k = g; g = align256(g + size_t(T) * sh.Hkv * dd);
  w.f8_vt = g; g = align256(g + size_t(T) * sh.Hkv * dd);
  w.total_fp8 = g;
  p->fp8_ok = sh.d == 128 && T % 16 == 0;
  for (const BaChunk& ch : p->chunks)
    if (ch.nat0 % 16 != 0) p->fp8_ok = false;

  // ---- host image of the table region
  try {
    p->image.assign(w.table_bytes, 0);
  } catch (const std::bad_alloc&) {
    return BA_ERR_HOST_ALLOC;
  }
  put(p->image, w.t_row_lim, p->row_lim);
  put(p->image, w.t_nat_lim, p->nat_lim);
  put(p->image, w.t_tok_perm, p->tok_perm);
  put(p->image, w.t_anc_perm, p->anc_perm);
  put(p->image, w.t_fq, p->fq);
  put(p->image, w.t_fseg, p->fseg);
  put(p->image, w.t_forder, p->forder);
  put(p->image, w.t_bq, p->bq);
  put(p->image, w.t_bkv, p->bkv);
  put(p->image, w.t_bqr, p->bqr);
  put(p->image, w.t_border, p->border);
  return BA_OK;
}

int ba_validate_plan(const ba_plan* p) {
  const BaShape& sh = p->shape;
  const int64_t rows = sh.rows, T = sh.T;
  auto bad = [] { return BA_ERR_INVALID_ARG; };
  if (int64_t(p->row_lim.size()) != rows || int64_t(p->tok_perm.size()) != T) return bad();
  std::vector<char> seen(T, 0);
  for (int32_t v : p->tok_perm) {
    if (v < 0 || v >= T || seen[v]) return bad();
    seen[v] = 1;
  }
  if (sh.family == BA_FAMILY_BLOCK) {
    std::vector<char> sa(p->NA, 0);
    if (int64_t(p->anc_perm.size()) != p->NA) return bad();
    for (int32_t v : p->anc_perm) {
      if (v < 0 || v >= p->NA || sa[v]) return bad();
      sa[v] = 1;
    }
  }
  for (int32_t v : p->row_lim)
    if (v < 0 || v >= T) return bad();
  if (int64_t(p->nat_lim.size()) != rows) return bad();
  auto natural_row = [&](int32_t r) -> int64_t {
    return sh.family == BA_FAMILY_BLOCK ? int64_t(p->anc_perm[r / sh.B]) * sh.B + r % sh.B : p->tok_perm[r];
  };
  auto check_tile = [&](const BaQTile& t, int bm) {
    if (!(t.row0 >= 0 && t.nrows >= 1 && t.nrows <= bm && int64_t(t.row0) + t.nrows <= rows &&
          t.lim_min <= t.lim_max && p->row_lim[t.row0] == t.lim_min && p->row_lim[t.row0 + t.nrows - 1] == t.lim_max))
      return false;
    // rows are contiguous in the natural layout and keep their limits there
    for (int32_t i = 0; i < t.nrows; ++i) {
      const int64_t nr = natural_row(t.row0 + i);
      if (nr != int64_t(t.nrow0) + i || p->nat_lim[nr] != p->row_lim[t.row0 + i]) return false;
    }
    return true;
  };
  for (const BaQTile& t : p->fq) {
    if (!check_tile(t, BA_FWD_BM) || t.seg0 < 0 || t.nseg < 1 || int64_t(t.seg0) + t.nseg > int64_t(p->fseg.size()))
      return bad();
    for (int i = 0; i < t.nseg; ++i) {
      const BaKvSeg& g = p->fseg[t.seg0 + i];
      if (g.k0 < 0 || g.nkeys < 1 || int64_t(g.k0) + g.nkeys > T) return bad();
      // positions inside a segment are contiguous and map back through the permutation
      if (p->tok_perm[g.k0] != g.pos0 || p->tok_perm[g.k0 + g.nkeys - 1] != g.pos0 + g.nkeys - 1) return bad();
      if (!g.diag && g.pos0 + g.nkeys - 1 > t.lim_min) return bad();
    }
  }
  for (const BaQTile& t : p->bq)
    if (!check_tile(t, BA_BWD_BM)) return bad();
  if (p->bkv.size() % BA_BWD_CS != 0) return bad();
  for (size_t i = 0; i < p->bkv.size(); ++i) {
    const BaKvTile& k = p->bkv[i];
    const BaKvTile& lead = p->bkv[i - i % BA_BWD_CS];
    // a group shares its chunk and its query ranges; only members after the
    // first may be empty fillers, and a filler is followed only by fillers
    if (k.chunk != lead.chunk || k.qr0 != lead.qr0 || k.nqr != lead.nqr) return bad();
    if (i % BA_BWD_CS == 0 ? k.nkeys < 1 : (k.nkeys > 0 && p->bkv[i - 1].nkeys == 0)) return bad();
    if (k.k0 < 0 || k.nkeys < 0 || k.nkeys > BA_BWD_BN || int64_t(k.k0) + std::max(k.nkeys, 1) > T) return bad();
    if (p->tok_perm[k.k0] != k.pos0) return bad();
    if (k.nkeys > 0 && p->tok_perm[k.k0 + k.nkeys - 1] != k.pos0 + k.nkeys - 1) return bad();
    if (k.qr0 < 0 || k.nqr < 0 || int64_t(k.qr0) + k.nqr > int64_t(p->bqr.size())) return bad();
    for (int i = 0; i < k.nqr; ++i) {
      const BaQRange& r = p->bqr[k.qr0 + i];
      if (r.t0 < 0 || r.t1 <= r.t0 || r.t1 > int64_t(p->bq.size())) return bad();
      for (int32_t q = r.t0; q < r.t1; ++q)
        if (!r.diag && p->bq[q].lim_min < k.pos0 + k.nkeys - 1) return bad();
    }
  }
  {
    std::vector<char> cov(T, 0);
    for (const BaKvTile& k : p->bkv)
      for (int32_t i = 0; i < k.nkeys; ++i) {
        if (cov[k.k0 + i]) return bad();
        cov[k.k0 + i] = 1;
      }
    for (char c : cov)
      if (!c) return bad();
  }
  auto is_perm = [](const std::vector<int32_t>& v, size_t n) {
    if (v.size() != n) return false;
    std::vector<char> s(n, 0);
    for (int32_t x : v) {
      if (x < 0 || size_t(x) >= n || s[x]) return false;
      s[x] = 1;
    }
    return true;
  };
  if (!is_perm(p->forder, p->fq.size()) || !is_perm(p->border, p->bkv.size())) return bad();
  // the launch order keeps the members of a group together and in order
  for (size_t i = 0; i < p->border.size(); ++i)
    if (p->border[i] != p->border[i - i % BA_BWD_CS] + int32_t(i % BA_BWD_CS) ||
        p->border[i - i % BA_BWD_CS] % BA_BWD_CS != 0)
      return bad();
  return BA_OK;
}
