// Host planner: zigzag chunk map, row limits, main-attention tile lists and
// the workspace layout of one branch-attention problem.
#pragma once

#include <stddef.h>
#include <stdint.h>

#include <vector>

#include "ba_internal.h"

// Byte offsets of everything the library keeps in the caller's workspace.
struct BaWorkspaceLayout {
  size_t status;                  // device status word (256 B)
  size_t tables;                  // start of the uploaded table image
  size_t table_bytes;             // size of the table image
  size_t t_row_lim, t_nat_lim, t_tok_perm, t_anc_perm, t_fq, t_fseg, t_forder, t_bq, t_bkv, t_bqr, t_border;
  size_t rowrec;                  // backward scratch: row records (16 B), natural order
  size_t total;
  // 8-bit forward (after `total`, so it overlaps neither scratch region):
  // amax[3], e4m3 copies of q and k_m, the transposed e4m3 V^T [Hkv][d][T]
  size_t f8_amax, f8_q, f8_k, f8_vt;
  size_t total_fp8;
};

// Chunk c of sequence s: natural start, packed start, length, owner rank.
struct BaChunk {
  int32_t seq, c, rank;
  int32_t nat0;   // natural position of the first token
  int32_t pk0;    // packed index of the first token
  int32_t len;    // tokens
  int32_t row0;   // first packed query row of the chunk (per stream)
  int32_t nrows;  // packed query rows whose anchor lies in the chunk
};

struct ba_plan {
  uint64_t id;
  std::vector<int32_t> cu;       // [S+1]
  std::vector<int32_t> anchors;  // [NA] (BLOCK)
  BaShape shape;
  int32_t C;
  int32_t S;
  int64_t NA;

  std::vector<BaChunk> chunks;   // indexed seq * 2C + c
  std::vector<int32_t> row_lim, nat_lim, tok_perm, anc_perm, tok_rank;
  std::vector<BaQTile> fq;
  std::vector<BaKvSeg> fseg;
  std::vector<int32_t> forder;
  std::vector<BaQTile> bq;
  std::vector<BaKvTile> bkv;
  std::vector<BaQRange> bqr;
  std::vector<int32_t> border;
  std::vector<int64_t> comm;     // Eq. 3 bytes per rank

  int64_t main_pairs = 0, branch_pairs = 0, fwd_blocks = 0;
  // the 8-bit forward's V^T loads start at chunk starts: they must be
  // multiples of 16 tokens (TMA inner coordinate), and head_dim must be 128
  bool fp8_ok = false;

  BaWorkspaceLayout ws;
  std::vector<unsigned char> image;  // host copy of the table region

  // optional per-kernel timing (events are opaque cudaEvent_t handles)
  bool prof_on = false;
  std::vector<void*> prof_events;                  // pool, pairs (start, stop)
  size_t prof_used = 0;                            // pairs recorded since the last read
  std::vector<int> prof_kernel;                    // kernel id of each recorded pair
  double prof_ms[16] = {0};
  int64_t prof_launches[16] = {0};

  ~ba_plan();
};

// Builds the plan; returns a ba_status.
int ba_build_plan(const ba_plan_desc* desc, ba_plan* p);

// Checks every index the kernels will follow against the buffer it points
// into (host only); returns BA_OK or BA_ERR_INVALID_ARG.
int ba_validate_plan(const ba_plan* p);
