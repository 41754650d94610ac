// Internal types shared by the host planner and the kernels (not part of the C ABI).
#pragma once

#include <stdint.h>

#include "../../include/ba.h"

// Tile sizes of the main-attention kernels.  The planner cuts the query rows
// and main keys of every zigzag chunk into tiles of these sizes.
#define BA_FWD_BM 128   // query rows per forward tile
#define BA_FWD_BN 64    // keys per forward key block (work estimate only)
#define BA_BWD_BM 128   // query rows per backward query tile
#define BA_BWD_BN 128   // keys per backward key tile
#define BA_BWD_CS 2     // key tiles per thread-block cluster of the dK/dV kernel:
                        // the tiles of a cluster come from one chunk and meet
                        // the same query tiles in the same order; the cluster
                        // only makes them run side by side, so each CTA's own
                        // loads of a Q / dO tile follow the first one into L2

// Device status word values (first word of the workspace).
#define BA_DEV_OK 0u
#define BA_DEV_TIMEOUT 1u
#define BA_DEV_BOUNDS 2u

// A run of <= BM consecutive packed query rows inside one zigzag chunk.  The
// same tiling serves every query stream (step j and head h).  A chunk is a
// contiguous range of natural positions (and of natural anchors), so the
// tile's rows are also contiguous in the natural layout, from nrow0: kernels
// address the caller's natural tensors directly (the zigzag pack is folded
// into their load coordinates).
struct BaQTile {
  int32_t row0;     // first packed row (per stream); indexes the row_lim table
  int32_t nrows;    // rows in the tile (<= BM)
  int32_t seg0;     // first key segment (forward) / unused (backward)
  int32_t nseg;     // key segments, in ring order
  int32_t lim_min;  // smallest row limit (natural position of the last visible main key)
  int32_t lim_max;  // largest row limit
  int32_t work;     // key blocks visited (forward) — used for longest-first order
  int32_t chunk;    // global chunk index (sequence * 2C + c)
  int32_t nrow0;    // natural row (per stream) of row0; rows are contiguous
  int32_t pad;
};

// A run of packed main keys inside one chunk that a query tile attends.
struct BaKvSeg {
  int32_t k0;      // first packed key
  int32_t nkeys;   // keys in the segment
  int32_t pos0;    // natural position of k0 (positions are contiguous inside a
                   // chunk): the key rows the kernels load
  int32_t diag;    // 1: the per-row causal limit cuts into the segment
};

// Backward: a run of <= BN packed main keys inside one chunk.  Key tiles come
// in groups of BA_BWD_CS consecutive tiles of one chunk (consecutive in the
// table, and in the launch order) that share one list of query ranges; a
// group at the end of a chunk is filled up with empty tiles (nkeys = 0) that
// take part in the group's loads but own no keys.
struct BaKvTile {
  int32_t k0, nkeys, pos0;
  int32_t qr0, nqr;   // query-tile ranges that see this key tile, ring-replay order
  int32_t work;       // query tiles visited (per stream)
  int32_t chunk, pad;
};

// Backward: query tiles [t0, t1) of one chunk that see a key tile.
struct BaQRange {
  int32_t t0, t1, diag, pad;
};

// Shape of a plan as the kernels see it.
struct BaShape {
  int32_t family;     // ba_family
  int32_t Hq, Hkv, G; // G = Hq / Hkv
  int32_t d;
  int32_t steps;      // D for TTT, 1 otherwise (leading dim of q_b)
  int32_t B;          // block size (BLOCK), 1 otherwise
  int32_t nbk;        // branch key slots a unit's queries read: D (TTT), B (BLOCK),
                      // 0 (CAUSAL); step + 1 in a single-step TTT call
  int32_t step0;      // TTT: slot of the call's first query step (0 for the
                      // whole plan; the step in a single-step call)
  int64_t T;          // main tokens
  int64_t rows;       // packed rows per stream: T (TTT/CAUSAL) or NA * B (BLOCK)
  int64_t units;      // anchor units: T (TTT/CAUSAL) or NA (BLOCK)
  float scale;
  float scale_log2;   // scale * log2(e)
};

// Device tables (inside the workspace).
struct BaTables {
  const int32_t* row_lim;   // [rows]   packed row -> last visible main position
  const int32_t* nat_lim;   // [rows]   natural row -> last visible main position
  const int32_t* tok_perm;  // [T]   packed token -> natural token
  const int32_t* anc_perm;  // [NA]  packed anchor -> natural anchor (BLOCK)
  const BaQTile* fq;        // forward query tiles
  const BaKvSeg* fseg;      // forward key segments
  const int32_t* forder;    // forward tiles, longest first
  const BaQTile* bq;        // backward query tiles
  const BaKvTile* bkv;      // backward key tiles
  const BaQRange* bqr;      // backward query ranges
  const int32_t* border;    // backward key tiles, longest first
  int32_t n_fq, n_fseg, n_bq, n_bkv, n_bqr, pad;
  unsigned int* status;     // device status word
};
