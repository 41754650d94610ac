// One query row's branch keys, for the epilogues of the main-attention
// kernels that finish the row themselves.
//
// "Online Draft Co-Training ...", ai.info summary, Key Contributions 1 and
// "Methodology in Plain English"; paperlens walkthrough, Wall 1: besides its
// causal main prefix, a branch query attends only the few keys of its own
// branch, which live on its anchor's rank —
//   TTT   — the step-j query at position p sees branch keys (p, i), i <= j;
//   BLOCK — each of the B queries of an anchor sees all B keys of its block.
// Keys are read straight from the caller's natural-layout k_b / v_b: TTT
// slot i of position p is row i * T + p, block key t of anchor a is row
// a * B + t.  The rows of one main-attention tile are consecutive positions
// (or anchors), so the CTAs that share a tile find these rows in L2.
#pragma once

#include "device.cuh"

// branch keys of a query of global TTT step `jg` (or of a block query)
__device__ __forceinline__ int branch_key_count(const BaShape& sh, int jg) {
  return sh.family == BA_FAMILY_TTT ? jg + 1 : (sh.family == BA_FAMILY_BLOCK ? sh.B : 0);
}

// anchor unit of natural query row nr: its position (TTT) or anchor (BLOCK)
__device__ __forceinline__ int64_t branch_unit_of_row(const BaShape& sh, int64_t nr) {
  return sh.family == BA_FAMILY_BLOCK ? nr / sh.B : nr;
}

// row of branch key t of unit u in the [slot][Hkv][d] branch tensors
__device__ __forceinline__ int64_t branch_key_row(const BaShape& sh, int64_t u, int t) {
  return sh.family == BA_FAMILY_TTT ? int64_t(t) * sh.T + u : u * sh.B + t;
}

// <a, b> over 8 bf16 pairs held in two 16-byte words, fp32
__device__ __forceinline__ float dot8_bf16(uint4 a, uint4 b) {
  const float2 a0 = unpack_bf16(a.x), a1 = unpack_bf16(a.y), a2 = unpack_bf16(a.z), a3 = unpack_bf16(a.w);
  const float2 b0 = unpack_bf16(b.x), b1 = unpack_bf16(b.y), b2 = unpack_bf16(b.z), b3 = unpack_bf16(b.w);
  float s = a0.x * b0.x;
  s = fmaf(a0.y, b0.y, s);
  s = fmaf(a1.x, b1.x, s);
  s = fmaf(a1.y, b1.y, s);
  s = fmaf(a2.x, b2.x, s);
  s = fmaf(a2.y, b2.y, s);
  s = fmaf(a3.x, b3.x, s);
  return fmaf(a3.y, b3.y, s);
}

// acc[0..7] += w * (8 bf16 values in one 16-byte word)
__device__ __forceinline__ void axpy8_bf16(float* acc, float w, uint4 v) {
  const float2 v0 = unpack_bf16(v.x), v1 = unpack_bf16(v.y), v2 = unpack_bf16(v.z), v3 = unpack_bf16(v.w);
  acc[0] = fmaf(w, v0.x, acc[0]);
  acc[1] = fmaf(w, v0.y, acc[1]);
  acc[2] = fmaf(w, v1.x, acc[2]);
  acc[3] = fmaf(w, v1.y, acc[3]);
  acc[4] = fmaf(w, v2.x, acc[4]);
  acc[5] = fmaf(w, v2.y, acc[5]);
  acc[6] = fmaf(w, v3.x, acc[6]);
  acc[7] = fmaf(w, v3.y, acc[7]);
}

// Largest number of branch keys one query can have: block size B <= 64, TTT
// depth D <= 16 (the planner's limits).
#define BA_MAX_BRANCH_KEYS 64
