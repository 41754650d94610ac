// K2 — causal main-sequence attention forward on the 5th-generation tensor
// cores (tcgen05, TMEM accumulators, TMA-fed 128B-swizzled tiles).
//
// "Online Draft Co-Training ...", ai.info summary, "Methodology in Plain
// English": the main part is ordinary causal context-parallel attention —
// zigzag-ring attention where K/V circulate, queries stay put, and partial
// results are merged with the log-sum-exp rule between ring steps.  On one GPU
// a query tile walks the key segments the planner lists for it in ring order
// (step s: the chunks of rank (r - s) mod C below or on its own chunk); the
// online softmax carried from one key block to the next is exactly that merge.
//
// One CTA = one 128-row query tile of one query stream (TTT step j, q head h)
// against blocks of 128 keys of kv head h / G.  Warp roles:
//   warps 0-3  softmax: thread t owns row t (TMEM lane t).  Reads S from TMEM,
//              masks the ragged block end and the per-row causal limit on the
//              diagonal chunk, keeps the row max / sum, writes P (bf16, two
//              per 32-bit column) back into the first 64 columns of the same
//              S buffer, rescales O in TMEM only when the row max grew by more
//              than 2^8 (the values of P stay below 256), and finally
//              finishes its row: the rank-local branch part over the row's
//              few branch keys (read from k_b / v_b), the Eq. 2 merge with the
//              main part O / l, and the bf16 output row and its lse.
//   warp 4     TMA producer: Q once, then K and V blocks into three-stage rings.
//   warp 5     owns TMEM; one thread issues S = Q K^T into one of three TMEM
//              S buffers.
//   warp 6     one thread issues O += P V with P read from TMEM as the A
//              operand.  Two issuing threads: an MMA instruction is accepted
//              only as fast as the tensor cores take it, so a single thread
//              that also waits on the softmax between groups lets the queue
//              run dry; each thread's commits track its own GEMMs.
// TMEM: S buffers at columns [0,128), [128,256), [256,384); O = [384, 384 + d).
// An S buffer is busy from its QK^T GEMM until the PV GEMM of the same block
// has read P out of it, so with three of them the next block's QK^T is always
// queued on the tensor cores behind the current PV while the softmax runs.
// Every wait is bounded (BA_WAIT_CYCLES); a timeout records BA_DEV_TIMEOUT,
// every role leaves its loop, and TMEM is released before the CTA exits.
//
// 8-bit variant (F8 = true; rainbus page, limitations and future work, item
// (4): fp8 training of the decomposition).  Q, K and V^T arrive as e4m3
// copies with per-tensor scales (s_q, s_k, s_v = amax / 448, made by the
// quantisation kernels); QK^T and PV run as kind::f8f6f4 MMAs with K = 32,
// S is fp32 in TMEM, the softmax folds s_q s_k into its scale and keeps the
// row max, sum and lse in fp32, P (at most 2^8 by the lazy rescale) is stored
// as e4m3, four per TMEM column, and the epilogue multiplies O by s_v.  A d =
// 128 row of 8-bit values is one 128-byte swizzled block; V is read from its
// transposed copy [Hkv][d][T], so the PV GEMM's B operand is K-major (keys
// along the 128-byte rows) like every other operand.
#include <cudaTypedefs.h>
#include <cuda_fp8.h>
#include <math.h>

#include <mutex>

#include "branch_row.cuh"
#include "kernels.h"
#include "tc.cuh"

namespace {

constexpr int TBM = 128;  // query rows per tile
constexpr int TBN = 128;  // keys per block
constexpr int NTHREADS = 224;  // 4 softmax warps, 1 TMA warp, 2 MMA-issuing warps
constexpr int NKV = 3;    // K / V ring stages
constexpr int NSB = 3;    // S (and P) buffers in TMEM

template <int D, bool F8>
struct FwdSmem {
  static constexpr int EB = F8 ? 1 : 2;                   // bytes per element
  static constexpr int CB = D * EB / 128;                 // 128-byte blocks per row
  static constexpr int ELB = 128 / EB;                    // elements per block row
  static constexpr uint32_t TILE = 128u * 128u;           // one 128-row x 128-byte swizzled block
  static constexpr uint32_t q = 0;
  static constexpr uint32_t k = q + CB * TILE;            // [NKV stages][CB blocks]
  static constexpr uint32_t v = k + NKV * CB * TILE;      // [NKV stages][CB blocks]
  static constexpr uint32_t bars = v + NKV * CB * TILE;
  static constexpr uint32_t bytes = bars + 256;
  static constexpr uint32_t alloc = bytes + 1024;         // slack for 1024-byte alignment
};

// barrier slots (8 bytes each) after FwdSmem::bars
enum {
  B_QFULL = 0,
  B_KFULL = 1,                // [NKV]
  B_KEMPTY = B_KFULL + NKV,   // [NKV]
  B_VFULL = B_KEMPTY + NKV,   // [NKV]
  B_VEMPTY = B_VFULL + NKV,   // [NKV]
  B_SFULL = B_VEMPTY + NKV,   // [NSB] S of a block is in TMEM
  B_PFULL = B_SFULL + NSB,    // [NSB] P of a block is in TMEM (per buffer, so the
                              // softmax can run a block ahead of the MMA warp's wait)
  B_SFREE = B_PFULL + NSB,    // [NSB] the block's PV GEMM is done: O is up to date
                              // and the S / P buffer is free
  B_COUNT = B_SFREE + NSB
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
    kb += TBN;
    if (kb >= cur.nkeys) {
      kb = 0;
      ++si;
      if (si < send) cur = seg[si];
    }
  }
};

// One row's 128 scores of a block out of TMEM (four 32-column loads, one
// wait), with keys at or past `climit` set to -inf when the block is masked.
__device__ __forceinline__ void load_scores(float (&s)[TBN], uint32_t taddr, bool masked, int climit) {
#pragma unroll
  for (int c = 0; c < TBN / 32; ++c) tmem_ld32(taddr + c * 32, s + c * 32);
  tmem_wait_ld();
  if (masked) {
#pragma unroll
    for (int c = 0; c < TBN; ++c)
      if (c >= climit) s[c] = -INFINITY;
  }
}

// Four fp32 values as e4m3, packed low byte first (the element order of a
// K-major 8-bit operand along a TMEM column).
__device__ __forceinline__ uint32_t pack_e4m3x4(float a, float b, float c, float d) {
  const uint32_t lo = __nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
  const uint32_t hi = __nv_cvt_float2_to_fp8x2(make_float2(c, d), __NV_SATFINITE, __NV_E4M3);
  return lo | (hi << 16);
}

// (a0 * b + c, a1 * b + c) in one packed fp32x2 FMA, rounded to f16x2
// (a0 in the low half).
__device__ __forceinline__ uint32_t fma_f32x2(float a0, float a1, float b, float c) {
  uint32_t h;
  asm("{\n .reg .b64 a, bb, cc, d;\n .reg .f32 d0, d1;\n"
      " mov.b64 a, {%1, %2};\n mov.b64 bb, {%3, %3};\n mov.b64 cc, {%4, %4};\n"
      " fma.rn.f32x2 d, a, bb, cc;\n mov.b64 {d0, d1}, d;\n"
      " cvt.rn.f16x2.f32 %0, d1, d0;\n}\n"
      : "=r"(h)
      : "f"(a0), "f"(a1), "f"(b), "f"(c));
  return h;
}

// 2^x for both halves of an f16x2 (one MUFU instruction for the pair).
__device__ __forceinline__ __half2 ex2_f16x2(uint32_t x) {
  uint32_t y;
  asm("ex2.approx.f16x2 %0, %1;\n" : "=r"(y) : "r"(x));
  __half2_raw r;
  r.x = static_cast<unsigned short>(y & 0xffffu);
  r.y = static_cast<unsigned short>(y >> 16);
  return __half2(r);
}

// Per-tensor fp8 scale from an amax (amax / 448, or 1 for an all-zero tensor).
__device__ __forceinline__ float f8_scale(float amax) { return amax > 0.f ? amax * (1.0f / 448.0f) : 1.0f; }

template <int D, bool F8>
__global__ void __launch_bounds__(NTHREADS, 1)
    main_fwd_tc_kernel(const BaFwdArgs a, const __grid_constant__ CUtensorMap tmq,
                       const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv) {
  using L = FwdSmem<D, F8>;
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
  // an earlier CTA already failed: leave before touching barriers or TMEM
  if (*reinterpret_cast<volatile unsigned int*>(tb.status) != 0u) return;
  const BaQTile tile = tb.fq[tb.forder[oi]];
  const int kvh = si / (sh.steps * sh.G);
  const int rem = si % (sh.steps * sh.G);
  const int j = rem / sh.G;
  const int h = kvh * sh.G + rem % sh.G;

  if (tid == 0) {
    *abort_flag = 0;
    mbar_init(bar(B_QFULL), 1);
    for (int s = 0; s < NKV; ++s) {
      mbar_init(bar(B_KFULL + s), 1);
      mbar_init(bar(B_KEMPTY + s), 1);
      mbar_init(bar(B_VFULL + s), 1);
      mbar_init(bar(B_VEMPTY + s), 1);
    }
    for (int s = 0; s < NSB; ++s) {
      mbar_init(bar(B_SFULL + s), 1);
      mbar_init(bar(B_PFULL + s), 4);
      mbar_init(bar(B_SFREE + s), 1);
    }
    fence_mbar_init();
  }
  if (warp == 5) {
    tmem_alloc(smem_u32(const_cast<uint32_t*>(tmem_slot)), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t tS = tmem, tO = tmem + NSB * TBN;

  if (warp == 4) {
    // ------------------------------------------------------------ TMA producer
    if (elect_one()) {
      tma_prefetch_desc(&tmq);
      tma_prefetch_desc(&tmk);
      tma_prefetch_desc(&tmv);
      mbar_expect_tx(bar(B_QFULL), CB * L::TILE);
      for (int cb = 0; cb < CB; ++cb)
        tma_load_3d(sbase + L::q + cb * L::TILE, &tmq, bar(B_QFULL), cb * L::ELB, h, int(j * sh.rows + tile.nrow0));
      BlockIter it;
      it.init(tb.fseg, tile.seg0, tile.nseg);
      for (int i = 0; it.valid(); ++i, it.next()) {
        const int st = i % NKV;
        const uint32_t ph = (i / NKV) & 1;
        const int key = it.cur.pos0 + it.kb;  // natural key row
        if (!mbar_wait(bar(B_KEMPTY + st), ph ^ 1, tb.status, abort_flag)) break;
        mbar_expect_tx(bar(B_KFULL + st), CB * L::TILE);
        for (int cb = 0; cb < CB; ++cb)
          tma_load_3d(sbase + L::k + (st * CB + cb) * L::TILE, &tmk, bar(B_KFULL + st), cb * L::ELB, kvh, key);
        if (!mbar_wait(bar(B_VEMPTY + st), ph ^ 1, tb.status, abort_flag)) break;
        mbar_expect_tx(bar(B_VFULL + st), CB * L::TILE);
        if constexpr (F8) {
          // V^T block: d rows of 128 keys (key a multiple of 16: the plan checks
          // that every chunk starts on a 16-token boundary)
          tma_load_3d(sbase + L::v + st * L::TILE, &tmv, bar(B_VFULL + st), key, 0, kvh);
        } else {
          for (int cb = 0; cb < CB; ++cb)
            tma_load_3d(sbase + L::v + (st * CB + cb) * L::TILE, &tmv, bar(B_VFULL + st), cb * 64, kvh, key);
        }
      }
    }
  } else if (warp == 5 || warp == 6) {
    // ------------------------------------------------------------ MMA issuers
    if (elect_one()) {
      constexpr uint32_t idesc_qk =
          F8 ? idesc_e4m3_f32(128, TBN, false, false) : idesc_bf16_f32(128, TBN, false, false);
      // 8-bit: V^T makes B K-major; 16-bit: V is an MN-major B
      constexpr uint32_t idesc_pv = F8 ? idesc_e4m3_f32(128, D, false, false) : idesc_bf16_f32(128, D, false, true);
      // operand descriptors, built once: every MMA below adds a constant offset
      const uint64_t dq0 = smem_desc_sw128(sbase + L::q, 16, 1024), dk0 = smem_desc_sw128(sbase + L::k, 16, 1024);
      const uint64_t dvm = smem_desc_sw128(sbase + L::v, F8 ? 16 : L::TILE, 1024);
      auto issue_pv = [&](int i) -> bool {
        const int pb = i % NSB, vs = i % NKV;
        if (!mbar_wait(bar(B_PFULL + pb), (i / NSB) & 1, tb.status, abort_flag)) return false;
        if (!mbar_wait(bar(B_VFULL + vs), (i / NKV) & 1, tb.status, abort_flag)) return false;
        tc_fence_after();
        const uint64_t dvs = desc_add(dvm, vs * CB * L::TILE);
        if constexpr (F8) {
          // P: 32 keys per K step = 8 TMEM columns; V^T: 32 keys = 32 bytes along its rows
#pragma unroll
          for (int kk = 0; kk < TBN / 32; ++kk)
            tc_mma_f8_tmem_a(tO, tS + pb * TBN + kk * 8, desc_add(dvs, kk * 32), idesc_pv, (i > 0 || kk > 0) ? 1u : 0u);
        } else {
#pragma unroll
          for (int kk = 0; kk < TBN / 16; ++kk)
            tc_mma_tmem_a(tO, tS + pb * TBN + kk * 8, desc_add(dvs, kk * 2048), idesc_pv, (i > 0 || kk > 0) ? 1u : 0u);
        }
        tc_commit(bar(B_SFREE + pb));
        tc_commit(bar(B_VEMPTY + vs));
        return true;
      };
      bool ok = mbar_wait(bar(B_QFULL), 0, tb.status, abort_flag);
      BlockIter it;
      it.init(tb.fseg, tile.seg0, tile.nseg);
      int i = 0;
      if (warp == 5) {
        for (; ok && it.valid(); ++i, it.next()) {
          const int ks = i % NKV, sb = i % NSB;
          if (!mbar_wait(bar(B_KFULL + ks), (i / NKV) & 1, tb.status, abort_flag)) { ok = false; break; }
          if (!mbar_wait(bar(B_SFREE + sb), ((i / NSB) & 1) ^ 1, tb.status, abort_flag)) { ok = false; break; }
          tc_fence_after();
          const uint64_t dks = desc_add(dk0, ks * CB * L::TILE);
          if constexpr (F8) {
            // a K = 32 step is 32 bytes along the single 128-byte block
#pragma unroll
            for (int kk = 0; kk < D / 32; ++kk)
              tc_mma_f8(tS + sb * TBN, desc_add(dq0, kk * 32), desc_add(dks, kk * 32), idesc_qk, kk > 0 ? 1u : 0u);
          } else {
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
              const uint32_t off = (kk >> 2) * L::TILE + (kk & 3) * 32;
              tc_mma(tS + sb * TBN, desc_add(dq0, off), desc_add(dks, off), idesc_qk, kk > 0 ? 1u : 0u);
            }
          }
          tc_commit(bar(B_SFULL + sb));
          tc_commit(bar(B_KEMPTY + ks));
        }
      } else {
        for (; it.valid(); ++i, it.next())
          if (!issue_pv(i)) break;
      }
    }
  } else {
    // ------------------------------------------------------------ softmax (rows)
    const int r = tid;  // TMEM lane == query row
    const int lim = r < tile.nrows ? tb.row_lim[tile.row0 + r] : -1;
    const uint32_t lane_off = uint32_t(warp * 32) << 16;
    float m_used = -INFINITY, l = 0.f;
    // scores come out of the MMA in units of the operands: the 8-bit path
    // folds the two quantisation scales into the softmax scale
    const float sl2 = F8 ? sh.scale_log2 * f8_scale(a.f8amax[0]) * f8_scale(a.f8amax[1]) : sh.scale_log2;
    // P of one 32-key group into its columns of the S buffer it came from:
    // bf16 two per column (16 columns), e4m3 four per column (8 columns)
    auto store_p = [&](const float* pv, uint32_t taddr_group0, int g) {
      if constexpr (F8) {
        uint32_t w[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) w[e] = pack_e4m3x4(pv[4 * e], pv[4 * e + 1], pv[4 * e + 2], pv[4 * e + 3]);
        tmem_st8(taddr_group0 + g * 8, w);
      } else {
        uint32_t w[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) w[e] = pack_bf16(pv[2 * e], pv[2 * e + 1]);
        tmem_st16(taddr_group0 + g * 16, w);
      }
    };
    BlockIter it;
    it.init(tb.fseg, tile.seg0, tile.nseg);
    int i = 0;
    bool ok = true;
    for (; it.valid(); ++i, it.next()) {
      const int sb = i % NSB;
      const uint32_t ph = (i / NSB) & 1;
      if (!mbar_wait_warp(bar(B_SFULL + sb), ph, tb.status, abort_flag)) { ok = false; break; }
      tc_fence_after();
      float s[TBN];
      const int nvalid = it.cur.nkeys - it.kb;
      const bool masked = it.cur.diag || nvalid < TBN;
      const int climit = it.cur.diag ? min(nvalid, lim - (it.cur.pos0 + it.kb) + 1) : nvalid;
      // S out of TMEM; mask: ragged end of the segment, causal limit on the
      // diagonal chunk
      load_scores(s, tS + lane_off + sb * TBN, masked, climit);
      // Once every row of the warp has a reference max, the exponentials are
      // taken against it without looking for the block max first: the block's
      // row sum bounds each of its P values, so a sum within 2^8 shows that no
      // row max grew by more than 2^8 and the result is exactly the one the
      // max-first path gives.  Otherwise (a row's first keys, or a rare grow)
      // the scores are reloaded and the block is done max-first.
      bool fast = __all_sync(0xffffffffu, m_used != -INFINITY);
      if (F8 && fast) {
        // 8-bit path: P is stored as e4m3 (3 mantissa bits), so it is computed
        // in packed halves — two exponents per fp32x2 FMA, one f16x2 ex2 and
        // one e4m3x2 conversion per pair, and an f16x2 tree for the block's
        // row sum (relative error below 2^-8, against e4m3's 2^-4).  A grown
        // max shows as a sum above 2^8 (or an f16 overflow to inf) and takes
        // the fp32 max-first path below.
        __half2 h[TBN / 2];
#pragma unroll
        for (int c = 0; c < TBN / 2; ++c)
          h[c] = ex2_f16x2(fma_f32x2(s[2 * c], s[2 * c + 1], sl2, -m_used));
        __half2 t[TBN / 4];
#pragma unroll
        for (int c = 0; c < TBN / 4; ++c) t[c] = __hadd2(h[2 * c], h[2 * c + 1]);
#pragma unroll
        for (int w = TBN / 8; w >= 1; w >>= 1) {
#pragma unroll
          for (int c = 0; c < w; ++c) t[c] = __hadd2(t[c], t[c + w]);
        }
        const float2 tf = __half22float2(t[0]);
        const float rs = tf.x + tf.y;
        if (__any_sync(0xffffffffu, !(rs <= 256.f))) {
          fast = false;
        } else {
          l += rs;
#pragma unroll
          for (int g = 0; g < TBN / 32; ++g) {
            uint32_t w[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              const uint32_t lo = __nv_cvt_halfraw2_to_fp8x2(__half2_raw(h[16 * g + 2 * e]), __NV_SATFINITE, __NV_E4M3);
              const uint32_t hi =
                  __nv_cvt_halfraw2_to_fp8x2(__half2_raw(h[16 * g + 2 * e + 1]), __NV_SATFINITE, __NV_E4M3);
              w[e] = lo | (hi << 16);
            }
            tmem_st8(tS + lane_off + sb * TBN + g * 8, w);
          }
        }
      } else if (fast) {
        float rsp[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int c = 0; c < TBN; ++c) {
          s[c] = ex2_approx(fmaf(s[c], sl2, -m_used));
          rsp[c & 7] += s[c];
        }
        const float rs = ((rsp[0] + rsp[1]) + (rsp[2] + rsp[3])) + ((rsp[4] + rsp[5]) + (rsp[6] + rsp[7]));
        if (__any_sync(0xffffffffu, rs > 256.f)) {
          fast = false;
          load_scores(s, tS + lane_off + sb * TBN, masked, climit);
        } else {
          l += rs;
#pragma unroll
          for (int g = 0; g < TBN / 32; ++g) {
            store_p(s + 32 * g, tS + lane_off + sb * TBN, g);
          }
        }
      }
      if (!fast) {
        // row max as 8 independent chains (a single chain is 128 dependent steps)
        float mxp[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) mxp[k] = s[k];
#pragma unroll
        for (int c = 8; c < TBN; ++c) mxp[c & 7] = fmaxf(mxp[c & 7], s[c]);
#pragma unroll
        for (int k = 0; k < 4; ++k) mxp[k] = fmaxf(mxp[k], mxp[k + 4]);
        const float mx = fmaxf(fmaxf(mxp[0], mxp[1]), fmaxf(mxp[2], mxp[3]));
        const float m_blk = mx * sl2;
        const bool grow = m_blk > m_used + 8.f;
        const float m_next = grow ? m_blk : m_used;
        const float base = m_next == -INFINITY ? 0.f : m_next;
        // rescale O (warp-uniform TMEM access) when any row's max grew; PV of
        // the previous block must have landed first
        if (i >= 1 && __any_sync(0xffffffffu, grow)) {
          const int pb = (i - 1) % NSB;
          if (!mbar_wait_warp(bar(B_SFREE + pb), ((i - 1) / NSB) & 1, tb.status, abort_flag)) { ok = false; break; }
          tc_fence_after();
          const float cfac = grow ? ex2_approx(m_used - base) : 1.f;
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            float o[32];
            tmem_ld32(tO + lane_off + c * 32, o);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] *= cfac;
            tmem_st32(tO + lane_off + c * 32, o);
          }
          tmem_wait_st();
          l *= cfac;
        } else if (grow) {
          l *= ex2_approx(m_used - base);  // i == 0: O not written yet
        }
        m_used = m_next;
        // P = exp2(S - base) in 32-key groups, each packed (keys 2c and 2c + 1
        // in column c) and stored into this row's lane of the S buffer while
        // the next group's exponentials run; only this thread reads or writes
        // the lane
        float rsp[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int g = 0; g < TBN / 32; ++g) {
#pragma unroll
          for (int c = 32 * g; c < 32 * g + 32; ++c) {
            s[c] = ex2_approx(fmaf(s[c], sl2, -base));
            rsp[c & 7] += s[c];
          }
          store_p(s + 32 * g, tS + lane_off + sb * TBN, g);
        }
        l += ((rsp[0] + rsp[1]) + (rsp[2] + rsp[3])) + ((rsp[4] + rsp[5]) + (rsp[6] + rsp[7]));
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_PFULL + sb));
    }
    // epilogue: the row is finished here.  Its branch part (the few keys of
    // its own branch, read from k_b / v_b) is computed by the row's thread,
    // then merged with the main part O / l, l_m by Eq. 2 (rainbus page, core
    // method): l = log(e^l_m + e^l_b) shifted by the larger of the two,
    // O = (e^(l_m - l) O_m + e^(l_b - l) O_b) / (e^(l_m - l) + e^(l_b - l)); an
    // empty part contributes nothing.  o (bf16) and lse are written in natural
    // order.
    if (ok && i > 0 && mbar_wait_warp(bar(B_SFREE + (i - 1) % NSB), ((i - 1) / NSB) & 1, tb.status, abort_flag)) {
      tc_fence_after();
      const bool write = r < tile.nrows;
      const int64_t nr = tile.nrow0 + r;
      const int64_t qrow = (int64_t(j) * sh.rows + nr) * sh.Hq + h;
      const float lm = l > 0.f ? (m_used + log2f(l)) * BA_LN2 : -INFINITY;
      // branch scores in base 2, their max and sum (online)
      const int nk = write ? branch_key_count(sh, sh.step0 + j) : 0;
      const int64_t u = branch_unit_of_row(sh, nr);
      const auto* kbp = static_cast<const __nv_bfloat16*>(a.kb);
      const auto* vbp = static_cast<const __nv_bfloat16*>(a.vb);
      float sc[BA_MAX_BRANCH_KEYS];
      float mb = -INFINITY, lsb = 0.f;
      if (nk > 0) {
        uint4 qv[D / 8];
        const uint4* qp = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(a.q) + qrow * D);
#pragma unroll
        for (int c = 0; c < D / 8; ++c) qv[c] = qp[c];
        for (int t = 0; t < nk; ++t) {
          const uint4* kp = reinterpret_cast<const uint4*>(kbp + (branch_key_row(sh, u, t) * sh.Hkv + kvh) * D);
          float dot = 0.f;
#pragma unroll
          for (int c = 0; c < D / 8; ++c) dot += dot8_bf16(qv[c], kp[c]);
          const float s2 = dot * sh.scale_log2;
          sc[t] = s2;
          const float mn = fmaxf(mb, s2);
          lsb = lsb * ex2_approx(mb - mn) + ex2_approx(s2 - mn);
          mb = mn;
        }
      }
      const float lb = nk > 0 ? (mb + log2f(lsb)) * BA_LN2 : -INFINITY;
      const float top = fmaxf(lm, lb);
      float wm = 0.f, wb = 0.f, lout = -INFINITY;
      if (top != -INFINITY) {
        lout = top + logf(expf(lm - top) + expf(lb - top));
        wm = expf(lm - lout);
        wb = expf(lb - lout);
        const float den = 1.0f / (wm + wb);
        wm *= den;
        wb *= den;
      }
      // O_m = O (TMEM) * s_v / l; O_b = sum_t p_t v_t / sum_t p_t.  The whole
      // row sits in registers while the branch values are added key by key,
      // so each key costs one round of 16-byte loads of its v row.
      const float cm = l > 0.f ? wm * (F8 ? f8_scale(a.f8amax[2]) : 1.f) / l : 0.f;
      const float cb = nk > 0 ? wb / lsb : 0.f;
      float o[D];
#pragma unroll
      for (int c = 0; c < D / 32; ++c) tmem_ld32(tO + lane_off + c * 32, o + 32 * c);
      tmem_wait_ld();
      if (write) {
#pragma unroll
        for (int e = 0; e < D; ++e) o[e] = wm > 0.f ? cm * o[e] : 0.f;
        if (wb > 0.f) {
          for (int t = 0; t < nk; ++t) {
            const float p = ex2_approx(sc[t] - mb) * cb;
            const uint4* vp = reinterpret_cast<const uint4*>(vbp + (branch_key_row(sh, u, t) * sh.Hkv + kvh) * D);
            uint4 vv[D / 8];
#pragma unroll
            for (int q = 0; q < D / 8; ++q) vv[q] = vp[q];
#pragma unroll
            for (int q = 0; q < D / 8; ++q) axpy8_bf16(o + 8 * q, p, vv[q]);
          }
        }
        uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.o) + qrow * D);
#pragma unroll
        for (int q = 0; q < D / 8; ++q)
          dst[q] = make_uint4(pack_bf16(o[8 * q], o[8 * q + 1]), pack_bf16(o[8 * q + 2], o[8 * q + 3]),
                              pack_bf16(o[8 * q + 4], o[8 * q + 5]), pack_bf16(o[8 * q + 6], o[8 * q + 7]));
      }
      if (write) a.lse[qrow] = lout;
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
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

cudaError_t get_encoder() {
  std::call_once(g_encode_once, [] {
    cudaDriverEntryPointQueryResult q;
    void* fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  return g_encode ? cudaSuccess : cudaErrorNotSupported;
}

// 3-D view (d, heads, rows) of a row-major [rows][heads][d] tensor of 1- or
// 2-byte elements; box (128 bytes of d, 1, 128 rows).
cudaError_t make_map(CUtensorMap* m, const void* base, int esize, int d, int heads, int64_t rows) {
  const cuuint64_t dims[3] = {cuuint64_t(d), cuuint64_t(heads), cuuint64_t(rows)};
  const cuuint64_t strides[2] = {cuuint64_t(d) * esize, cuuint64_t(heads) * d * esize};
  const cuuint32_t box[3] = {cuuint32_t(128 / esize), 1, 128};
  const cuuint32_t es[3] = {1, 1, 1};
  const CUtensorMapDataType dt = esize == 1 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const CUresult r = g_encode(m, dt, 3, const_cast<void*>(base), dims, strides, box, es,
                              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// 3-D view (keys, d, kv heads) of the 8-bit V^T copy [Hkv][d][T]; box (128 keys, 128 d rows, 1).
cudaError_t make_map_vt(CUtensorMap* m, const void* base, int d, int heads, int64_t T) {
  const cuuint64_t dims[3] = {cuuint64_t(T), cuuint64_t(d), cuuint64_t(heads)};
  const cuuint64_t strides[2] = {cuuint64_t(T), cuuint64_t(T) * d};
  const cuuint32_t box[3] = {128, 128, 1};
  const cuuint32_t es[3] = {1, 1, 1};
  const CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides, box, es,
                              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

template <int D, bool F8>
cudaError_t launch(const BaFwdArgs& a, cudaStream_t st) {
  CUtensorMap mq, mk, mv;
  cudaError_t e;
  const int es = F8 ? 1 : 2;
  const int64_t qrows = int64_t(a.sh.steps) * a.sh.rows;
  if ((e = make_map(&mq, F8 ? a.q8 : a.q, es, D, a.sh.Hq, qrows)) != cudaSuccess) return e;
  if ((e = make_map(&mk, F8 ? a.k8 : a.km, es, D, a.sh.Hkv, a.sh.T)) != cudaSuccess) return e;
  if constexpr (F8) {
    if ((e = make_map_vt(&mv, a.vt8, D, a.sh.Hkv, a.sh.T)) != cudaSuccess) return e;
  } else {
    if ((e = make_map(&mv, a.vm, es, D, a.sh.Hkv, a.sh.T)) != cudaSuccess) return e;
  }
  const int64_t grid = int64_t(a.tb.n_fq) * a.sh.steps * a.sh.Hq;
  const int smem = int(FwdSmem<D, F8>::alloc);
  if ((e = cudaFuncSetAttribute(main_fwd_tc_kernel<D, F8>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem)) !=
      cudaSuccess)
    return e;
  main_fwd_tc_kernel<D, F8><<<unsigned(grid), NTHREADS, smem, st>>>(a, mq, mk, mv);
  return cudaGetLastError();
}

}  // namespace

cudaError_t ba_launch_main_fwd_tc(const BaFwdArgs& a, cudaStream_t st) {
  const int64_t grid = int64_t(a.tb.n_fq) * a.sh.steps * a.sh.Hq;
  if (grid == 0) return cudaSuccess;
  if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  cudaError_t e = get_encoder();
  if (e != cudaSuccess) return e;
  return a.sh.d == 128 ? launch<128, false>(a, st) : launch<64, false>(a, st);
}

cudaError_t ba_launch_main_fwd_fp8(const BaFwdArgs& a, cudaStream_t st) {
  const int64_t grid = int64_t(a.tb.n_fq) * a.sh.steps * a.sh.Hq;
  if (grid == 0) return cudaSuccess;
  if (grid > 0x7fffffffLL || a.sh.d != 128 || !a.q8 || !a.k8 || !a.vt8 || !a.f8amax)
    return cudaErrorInvalidConfiguration;
  cudaError_t e = get_encoder();
  if (e != cudaSuccess) return e;
  return launch<128, true>(a, st);
}
