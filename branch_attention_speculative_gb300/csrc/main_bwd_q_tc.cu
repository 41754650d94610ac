// K6 (dQ part) — gradient of the main-sequence queries on the tcgen05 tensor
// cores, query-stationary.
//
// "Online Draft Co-Training ...", rainbus page, method step 5: the backward
// replays the ring.  For dQ the replay has the forward's shape: one CTA keeps a
// 128-row query tile of one query stream (TTT step j, q head h) and walks the
// key segments the planner lists for it in ring order.  P is recomputed from
// the merged lse (exact for both key sets, since the merged result is the
// single softmax over their union), so no running max is needed:
//   dP = dO V^T         M=128 queries, N=128 keys, K=d        -> TMEM
//   S  = Q K^T          same                                  -> TMEM (2 buffers)
//   (threads)  P = exp2(S * scale*log2e - lse*log2e) with the causal / ragged
//              mask, dS = P (dP - Delta), written back as bf16 into the S
//              buffer it came from
//   dQ += dS K          M=128 queries, N=d, K=128 keys; dS read from TMEM as
//                       the A operand, K an MN-major shared operand -> TMEM
// dQ stays in TMEM for the whole tile and is written once (no atomics, no
// read-modify-write) as bf16 into dq_b; the branch kernel, which stages each
// anchor's branch keys once for all of its rows, adds the branch part.
// TMEM: S0 [0,128), S1 [128,256), dP [256,384), dQ [384,512).  Inside an S
// buffer the warp of key half h reads fp32 columns [64h, 64h+64) and writes
// dS (bf16 pairs) back into [64h, 64h+32): no warp writes a column another
// warp still has to read.  The MMA warp issues dP(i+1), S(i+1), dQ(i) in that
// order: S(i+1) reuses the buffer dQ(i-1) read, and dP(i+1) covers the wait
// for dQ(i-1) to finish, so the tensor cores never drain between blocks.
// K sits in a three-stage ring (it is read by S and, a block later, by dQ), V
// in a two-stage ring.
// Warps: 0-7 compute (warp w: TMEM lane quarter w % 4 = query rows, keys
// 64 (w / 4) .. of each block; two warps per SM sub-partition hide each other's
// latencies), 8 TMA, 9 MMA + TMEM.
// head_dim 64 and 128: the kernel is templated on d (tiles of d / 64
// 128-byte swizzled blocks; dQ takes d TMEM columns).
// Every query row of the plan lies in exactly one tile and every tile writes
// all of its rows (the main part zero for a tile without key blocks).
#include <cudaTypedefs.h>
#include <math.h>

#include <mutex>

#include "kernels.h"
#include "tc.cuh"

namespace {

constexpr int QBM = 128;  // query rows per tile (BA_FWD_BM)
constexpr int KBN = 128;  // keys per block
constexpr int NTHREADS = 320;  // 8 compute warps, 1 TMA warp, 1 MMA warp
constexpr int NK = 3;          // K ring stages
constexpr int NV = 2;          // V ring stages

template <int D>
struct DqSmem {
  static constexpr int CB = D / 64;              // 64-column (128-byte) blocks per row
  static constexpr uint32_t TILE = 128u * 128u;  // [128 rows][64 columns] bf16, swizzled
  static constexpr uint32_t q = 0;               // CB blocks
  static constexpr uint32_t go = q + CB * TILE;  // CB blocks
  static constexpr uint32_t k = go + CB * TILE;       // [NK stages][CB blocks]
  static constexpr uint32_t v = k + NK * CB * TILE;   // [NV stages][CB blocks]
  static constexpr uint32_t bars = v + NV * CB * TILE;
  static constexpr uint32_t bytes = bars + 256;
  static constexpr uint32_t alloc = bytes + 1024;
};

enum {
  B_QFULL = 0,
  B_KFULL = 1,                // [NK]
  B_KEMPTY = B_KFULL + NK,    // [NK]
  B_VFULL = B_KEMPTY + NK,    // [NV]
  B_VEMPTY = B_VFULL + NV,    // [NV]
  B_SFULL = B_VEMPTY + NV,    // [2] dP and S of a block are in TMEM
  B_DSFULL = B_SFULL + 2,     // [2] dS of a block is in TMEM (per buffer, so the
                              // threads can finish a block before the MMA warp
                              // has waited for the previous one)
  B_SFREE = B_DSFULL + 2,     // [2] dQ of the block is done: the buffer is free
  B_DPEMPTY = B_SFREE + 2,    // the threads have loaded dP
  B_COUNT = B_DPEMPTY + 1
};
static_assert(8 * B_COUNT + 16 <= 256, "barrier area");

struct BlockIter {
  const BaKvSeg* seg;
  int si, send, kb;
  BaKvSeg cur;
  __device__ void init(const BaKvSeg* s, int s0, int n) {
    seg = s;
    si = s0;
    send = s0 + n;
    kb = 0;
    if (si < send) cur = seg[si];
  }
  __device__ bool valid() const { return si < send; }
  __device__ void next() {
    kb += KBN;
    if (kb >= cur.nkeys) {
      kb = 0;
      ++si;
      if (si < send) cur = seg[si];
    }
  }
};

template <int D>
__global__ void __launch_bounds__(NTHREADS, 1)
    main_bwd_q_tc_kernel(const BaBwdArgs a, const __grid_constant__ CUtensorMap tmq,
                         const __grid_constant__ CUtensorMap tmdo, const __grid_constant__ CUtensorMap tmk,
                         const __grid_constant__ CUtensorMap tmv) {
  using L = DqSmem<D>;
  constexpr int CB = L::CB;
  extern __shared__ unsigned char smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  unsigned char* gbase = smem_raw + (sbase - raw);
  const uint32_t bar0 = sbase + L::bars;
  auto bar = [&](int i) { return bar0 + 8u * uint32_t(i); };
  volatile int* abort_flag = reinterpret_cast<volatile int*>(gbase + L::bars + 8 * B_COUNT);
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(gbase + L::bars + 8 * B_COUNT + 8);

  const BaShape& sh = a.sh;
  const BaTables& tb = a.tb;
  const int nstreams = sh.steps * sh.Hq;
  const int si = int(blockIdx.x % nstreams);
  const int oi = int(blockIdx.x / nstreams);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (oi >= tb.n_fq) {
    if (tid == 0) ba_set_status(tb.status, BA_DEV_BOUNDS);
    return;
  }
  if (*reinterpret_cast<volatile unsigned int*>(tb.status) != 0u) return;
  const BaQTile tile = tb.fq[tb.forder[oi]];
  const int kvh = si / (sh.steps * sh.G);
  const int rem = si % (sh.steps * sh.G);
  const int j = rem / sh.G;
  const int h = kvh * sh.G + rem % sh.G;

  if (tid == 0) {
    *abort_flag = 0;
    mbar_init(bar(B_QFULL), 1);
    for (int s = 0; s < NK; ++s) {
      mbar_init(bar(B_KFULL + s), 1);
      mbar_init(bar(B_KEMPTY + s), 1);
    }
    for (int s = 0; s < NV; ++s) {
      mbar_init(bar(B_VFULL + s), 1);
      mbar_init(bar(B_VEMPTY + s), 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(B_SFULL + s), 1);
      mbar_init(bar(B_DSFULL + s), 8);
      mbar_init(bar(B_SFREE + s), 1);
    }
    mbar_init(bar(B_DPEMPTY), 8);
    fence_mbar_init();
  }
  if (warp == 9) {
    tmem_alloc(smem_u32(const_cast<uint32_t*>(tmem_slot)), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t tS = tmem, tDP = tmem + 256, tDQ = tmem + 384;

  if (warp == 8) {
    // ------------------------------------------------------------ TMA producer
    if (elect_one()) {
      tma_prefetch_desc(&tmq);
      tma_prefetch_desc(&tmdo);
      tma_prefetch_desc(&tmk);
      tma_prefetch_desc(&tmv);
      const int qrow = int(int64_t(j) * sh.rows + tile.nrow0);
      mbar_expect_tx(bar(B_QFULL), 2 * CB * L::TILE);
      for (int cb = 0; cb < CB; ++cb) {
        tma_load_3d(sbase + L::q + cb * L::TILE, &tmq, bar(B_QFULL), cb * 64, h, qrow);
        tma_load_3d(sbase + L::go + cb * L::TILE, &tmdo, bar(B_QFULL), cb * 64, h, qrow);
      }
      BlockIter it;
      it.init(tb.fseg, tile.seg0, tile.nseg);
      for (int i = 0; it.valid(); ++i, it.next()) {
        const int ks = i % NK, vs = i % NV;
        const int key = it.cur.pos0 + it.kb;  // natural key row
        if (!mbar_wait(bar(B_VEMPTY + vs), ((i / NV) & 1) ^ 1, tb.status, abort_flag)) break;
        mbar_expect_tx(bar(B_VFULL + vs), CB * L::TILE);
        for (int cb = 0; cb < CB; ++cb)
          tma_load_3d(sbase + L::v + (vs * CB + cb) * L::TILE, &tmv, bar(B_VFULL + vs), cb * 64, kvh, key);
        if (!mbar_wait(bar(B_KEMPTY + ks), ((i / NK) & 1) ^ 1, tb.status, abort_flag)) break;
        mbar_expect_tx(bar(B_KFULL + ks), CB * L::TILE);
        for (int cb = 0; cb < CB; ++cb)
          tma_load_3d(sbase + L::k + (ks * CB + cb) * L::TILE, &tmk, bar(B_KFULL + ks), cb * 64, kvh, key);
      }
    }
  } else if (warp == 9) {
    // ------------------------------------------------------------ MMA issuer
    if (elect_one()) {
      constexpr uint32_t id_s = idesc_bf16_f32(128, KBN, false, false);  // S, dP
      constexpr uint32_t id_q = idesc_bf16_f32(128, D, false, true);     // dQ (K as MN-major B)
      // operand descriptors, built once: every MMA below adds a constant offset
      const uint64_t dq0 = smem_desc_sw128(sbase + L::q, 16, 1024), dg0 = smem_desc_sw128(sbase + L::go, 16, 1024);
      const uint64_t dk0 = smem_desc_sw128(sbase + L::k, 16, 1024), dv0 = smem_desc_sw128(sbase + L::v, 16, 1024);
      const uint64_t dkm = smem_desc_sw128(sbase + L::k, L::TILE, 1024);
      auto issue_dp = [&](int i) -> bool {
        const int vs = i % NV;
        if (!mbar_wait(bar(B_VFULL + vs), (i / NV) & 1, tb.status, abort_flag)) return false;
        if (!mbar_wait(bar(B_DPEMPTY), (i & 1) ^ 1, tb.status, abort_flag)) return false;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * L::TILE + (kk & 3) * 32;
          tc_mma(tDP, desc_add(dg0, off), desc_add(dv0, vs * CB * L::TILE + off), id_s, kk > 0);
        }
        tc_commit(bar(B_VEMPTY + vs));
        return true;
      };
      auto issue_s = [&](int i) -> bool {
        const int ks = i % NK, sb = i & 1;
        if (!mbar_wait(bar(B_KFULL + ks), (i / NK) & 1, tb.status, abort_flag)) return false;
        if (!mbar_wait(bar(B_SFREE + sb), ((i >> 1) & 1) ^ 1, tb.status, abort_flag)) return false;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * L::TILE + (kk & 3) * 32;
          tc_mma(tS + sb * KBN, desc_add(dq0, off), desc_add(dk0, ks * CB * L::TILE + off), id_s, kk > 0);
        }
        tc_commit(bar(B_SFULL + sb));  // also covers dP(i), issued before
        return true;
      };
      auto issue_dq = [&](int i) -> bool {
        const int ks = i % NK, sb = i & 1;
        if (!mbar_wait(bar(B_DSFULL + sb), (i >> 1) & 1, tb.status, abort_flag)) return false;
        tc_fence_after();
        const uint64_t dks = desc_add(dkm, ks * CB * L::TILE);
#pragma unroll
        for (int kk = 0; kk < KBN / 16; ++kk)
          tc_mma_tmem_a(tDQ, tS + sb * KBN + (kk >> 2) * 64 + (kk & 3) * 8, desc_add(dks, kk * 2048), id_q,
                        (i > 0 || kk > 0) ? 1u : 0u);
        tc_commit(bar(B_SFREE + sb));
        tc_commit(bar(B_KEMPTY + ks));
        return true;
      };
      bool ok = mbar_wait(bar(B_QFULL), 0, tb.status, abort_flag);
      int n = 0;  // blocks, counted the way the other roles walk them
      {
        BlockIter it;
        for (it.init(tb.fseg, tile.seg0, tile.nseg); it.valid(); it.next()) ++n;
      }
      if (ok && n > 0) ok = issue_dp(0) && issue_s(0);
      for (int i = 0; ok && i < n; ++i) {
        if (i + 1 < n && !(issue_dp(i + 1) && issue_s(i + 1))) break;
        if (!issue_dq(i)) break;
      }
    }
  } else {
    // ------------------------------------------------------------ compute
    // warp w: TMEM lane quarter w % 4 (query rows 32 (w % 4) ..), keys
    // 64 (w / 4) .. 64 (w / 4) + 63 of each 128-key block
    const int quarter = warp & 3, half = warp >> 2;
    const int r = quarter * 32 + lane;
    const uint32_t lane_off = uint32_t(quarter * 32) << 16;
    const bool rok = r < tile.nrows;
    float nl2 = 0.f, delta = 0.f;  // -lse*log2e, Delta
    int lim = -1;
    if (rok) {
      const float4 rec = a.rowrec[(int64_t(j) * sh.Hq + h) * sh.rows + tile.nrow0 + r];
      nl2 = rec.x;
      delta = rec.y;
      lim = __float_as_int(rec.z);
    }
    BlockIter it;
    it.init(tb.fseg, tile.seg0, tile.nseg);
    int i = 0;
    bool ok = true;
    for (; it.valid(); ++i, it.next()) {
      const int sb = i & 1;
      const uint32_t ph = (i >> 1) & 1;
      const int nvalid = it.cur.nkeys - it.kb;
      const int climit = !rok ? 0 : (it.cur.diag ? min(nvalid, lim - (it.cur.pos0 + it.kb) + 1) : nvalid);
      if (!mbar_wait_warp(bar(B_SFULL + sb), ph, tb.status, abort_flag)) { ok = false; break; }
      tc_fence_after();
      // this warp's 64 keys: both S and dP chunks loaded before one wait
      float s[64], dp[64];
      tmem_ld32(tS + lane_off + sb * KBN + half * 64, s);
      tmem_ld32(tS + lane_off + sb * KBN + half * 64 + 32, s + 32);
      tmem_ld32(tDP + lane_off + half * 64, dp);
      tmem_ld32(tDP + lane_off + half * 64 + 32, dp + 32);
      tmem_wait_ld();
      // dP is in registers: its TMEM buffer can be refilled now
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_DPEMPTY));
      // dS = P (dP - Delta) in 32-key groups, each packed (keys 2c and 2c + 1
      // of this half in column c) and stored into the first 32 of this warp's
      // 64 columns of the S buffer while the next group is computed
#pragma unroll
      for (int g = 0; g < 2; ++g) {
        if (climit >= KBN) {  // full block (the common case): no mask
#pragma unroll
          for (int e = 32 * g; e < 32 * g + 32; ++e)
            s[e] = ex2_approx(fmaf(s[e], sh.scale_log2, nl2)) * (dp[e] - delta);
        } else {
#pragma unroll
          for (int e = 32 * g; e < 32 * g + 32; ++e) {
            const int c = half * 64 + e;
            const float p = ex2_approx(fmaf(s[e], sh.scale_log2, nl2));
            s[e] = (c < climit ? p : 0.f) * (dp[e] - delta);
          }
        }
        uint32_t w[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) w[e] = pack_bf16(s[32 * g + 2 * e], s[32 * g + 2 * e + 1]);
        tmem_st16(tS + lane_off + sb * KBN + half * 64 + g * 16, w);
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_DSFULL + sb));
    }
    // epilogue: dQ (main part, scaled) -> bf16 dq row, written once; each warp
    // writes d-columns (d / 2) (w / 4) .. of its 32 rows (zeros when the tile
    // has no key blocks).  The branch kernel adds each row's branch part.
    constexpr int HD = D / 2;
    const bool have = ok && i > 0 &&
                      mbar_wait_warp(bar(B_SFREE + ((i - 1) & 1)), ((i - 1) >> 1) & 1, tb.status, abort_flag);
    if (have || (ok && i == 0)) {
      if (have) tc_fence_after();
      const int64_t qrow = (int64_t(j) * sh.rows + tile.nrow0 + r) * sh.Hq + h;
      uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.dq) + qrow * D + half * HD);
#pragma unroll
      for (int c = 0; c < HD / 32; ++c) {
        float o[32];
        if (have) {
          tmem_ld32(tDQ + lane_off + half * HD + c * 32, o);
          tmem_wait_ld();
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] = 0.f;
        }
        if (rok) {
#pragma unroll
          for (int q = 0; q < 4; ++q)
            dst[c * 4 + q] = make_uint4(
                pack_bf16(sh.scale * o[8 * q], sh.scale * o[8 * q + 1]),
                pack_bf16(sh.scale * o[8 * q + 2], sh.scale * o[8 * q + 3]),
                pack_bf16(sh.scale * o[8 * q + 4], sh.scale * o[8 * q + 5]),
                pack_bf16(sh.scale * o[8 * q + 6], sh.scale * o[8 * q + 7]));
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  // after a failed wait, give MMAs and copies already in flight time to land
  // before TMEM is released
  if (*abort_flag) {
    const long long t0 = clock64();
    while (clock64() - t0 < (1ll << 21)) {
    }
  }
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_once;

cudaError_t encoder() {
  std::call_once(g_once, [] {
    cudaDriverEntryPointQueryResult q;
    void* fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  return g_encode ? cudaSuccess : cudaErrorNotSupported;
}

cudaError_t map3d(CUtensorMap* m, const void* base, int d, int heads, int64_t rows) {
  const cuuint64_t dims[3] = {cuuint64_t(d), cuuint64_t(heads), cuuint64_t(rows)};
  const cuuint64_t strides[2] = {cuuint64_t(d) * 2, cuuint64_t(heads) * d * 2};
  const cuuint32_t box[3] = {64, 1, 128};
  const cuuint32_t es[3] = {1, 1, 1};
  const CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
                              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

template <int D>
cudaError_t launch_q(const BaBwdArgs& a, int64_t grid, cudaStream_t st) {
  const int64_t qrows = int64_t(a.sh.steps) * a.sh.rows;
  CUtensorMap mq, mdo, mk, mv;
  cudaError_t e;
  if ((e = map3d(&mq, a.q, D, a.sh.Hq, qrows)) != cudaSuccess) return e;
  if ((e = map3d(&mdo, a.d_o, D, a.sh.Hq, qrows)) != cudaSuccess) return e;
  if ((e = map3d(&mk, a.km, D, a.sh.Hkv, a.sh.T)) != cudaSuccess) return e;
  if ((e = map3d(&mv, a.vm, D, a.sh.Hkv, a.sh.T)) != cudaSuccess) return e;
  const int smem = int(DqSmem<D>::alloc);
  if ((e = cudaFuncSetAttribute(main_bwd_q_tc_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem)) !=
      cudaSuccess)
    return e;
  main_bwd_q_tc_kernel<D><<<unsigned(grid), NTHREADS, smem, st>>>(a, mq, mdo, mk, mv);
  return cudaGetLastError();
}

}  // namespace

cudaError_t ba_launch_main_bwd_q_tc(const BaBwdArgs& a, cudaStream_t st) {
  const int64_t grid = int64_t(a.tb.n_fq) * a.sh.steps * a.sh.Hq;
  if (grid == 0) return cudaSuccess;
  if (grid > 0x7fffffffLL || (a.sh.d != 128 && a.sh.d != 64)) return cudaErrorInvalidConfiguration;
  cudaError_t e = encoder();
  if (e != cudaSuccess) return e;
  return a.sh.d == 128 ? launch_q<128>(a, grid, st) : launch_q<64>(a, grid, st);
}
