// K6 (dK / dV part) — gradient of the main keys and values on the tcgen05
// tensor cores, key-stationary.
//
// "Online Draft Co-Training ...", rainbus page, method step 5 and core method:
// the backward replays the same ring and accumulates gradients locally, with
// no branch-dependent traffic.  One CTA owns a tile of 128 main keys (inside
// one zigzag chunk) of one kv head and meets, in ring-replay order, every
// 64-row query tile that sees it, for every query stream (TTT step j, q head h)
// of its group.  P is recomputed from the merged lse (exact for both key sets,
// because Eq. 2's merged result is the single softmax over their union).
//
// Per (query tile, key tile) pair, on the tensor cores (tiles of 128 queries,
// so every GEMM has N = 128):
//   S^T  = K Q^T        M=128 keys, N=128 queries, K=d        -> TMEM S^T buffer
//   dP^T = V dO^T       same                                  -> TMEM dP^T buffer
//   (threads)  P^T = exp2(S^T * scale*log2e - lse*log2e),  dS^T = P^T (dP^T - Delta),
//              in packed bf16x2 arithmetic, written over the buffer each came from
//   dV  += P^T dO       M=128 keys, N=d, K=128 queries; P^T read from TMEM,
//                       dO an MN-major shared operand
//   dK  += dS^T Q       same, dS^T from TMEM
// dK and dV stay in TMEM for the whole CTA and are written once, in natural
// order, at the end.  dQ is computed by the query-stationary kernel
// (main_bwd_q_tc.cu), which needs no atomics.
// Why 128 queries: one tcgen05.mma costs at least about 46 cycles whatever its
// N (about 55 with A in TMEM), so an N=64 MMA (32 cycles of tensor work) runs
// the tensor pipe at two thirds of its rate, while an N=128 one (64 cycles)
// runs it at the full rate.  The price is TMEM: S^T, dP^T, dK and dV take
// 128 columns each, so P^T and dS^T are written over the S^T and dP^T values
// they came from, and K stays in shared memory.
// TMEM columns: S^T / P^T [0,128), dP^T / dS^T [128,256), dK [256,256+d), dV
// after it.  Inside the S^T buffer the warp of query half h (queries
// 64h..64h+63) reads fp32 columns [64h, 64h+64) and writes P^T (bf16 pairs)
// into [64h, 64h+32), so no warp writes a column another warp still has to
// read; the same holds for dP^T / dS^T.
// Order of the GEMMs: the next pair's S^T overwrites P^T, so it waits for this
// pair's dV; the next dP^T waits for this pair's dK.  Two threads issue: one
// S^T then dV, the other dP^T then dK, so the tensor pipe sees dV(i), dK(i),
// S^T(i+1), dP^T(i+1), ...: each GEMM's wait is covered by the one before it
// (the threads compute P^T(i+1) while dP^T(i+1) runs, and dS^T(i+1) while
// dV(i+1) runs).
// Warp roles: warps 0-7 compute (warp w: TMEM lane quarter w % 4 = key rows,
// query columns 64 (w / 4) ..; two warps per SM sub-partition hide each
// other's latencies), warp 8 loads with TMA (Q, dO and the tile's 16-byte row
// records {-lse*log2e, Delta, key limit}) into a ring of stages, warp 9 (which
// owns TMEM) issues S^T and dV, warp 10 dP^T and dK.  Each thread's commits
// track its own GEMMs.  All waits are bounded.
// Clusters: BA_BWD_CS CTAs that own consecutive key tiles of one chunk (and
// one kv head) form a thread-block cluster, which only makes the hardware run
// them side by side.  They meet the same query tiles in the same order and
// each loads its own Q / dO stages with plain TMA, so they read the same
// tiles within a few pairs of each other and all but the first read of a tile
// hit in L2.  The CTAs do not wait for one another: tying each stage refill
// to the slowest member's release (a barrier arrival relayed to every member)
// measured 2.4 times slower than letting each CTA run free.
// head_dim 64 and 128: the kernel is templated on d; a 128-byte swizzled block
// holds 64 columns, so d = 128 tiles are two blocks wide and d = 64 tiles one.
#include <cudaTypedefs.h>
#include <math.h>

#include <mutex>

#include "kernels.h"
#include "tc.cuh"

namespace {

constexpr int KBN = 128;  // keys per CTA
constexpr int QBM = BA_BWD_BM;  // queries per tile (128)
constexpr int NTHREADS = 352;  // 8 compute warps, 1 TMA warp, 2 MMA-issuing warps
static_assert(QBM == 128, "the GEMM shapes below assume 128-query tiles");

constexpr int CS = BA_BWD_CS;

template <int D>
struct BwdSmem {
  static constexpr int CB = D / 64;            // 64-column (128-byte) blocks per row
  static constexpr int NQS = D == 128 ? 2 : 4; // query-tile pipeline stages
  static constexpr uint32_t KT = 128u * 128u;  // [128 keys][64 d] bf16 block
  static constexpr uint32_t QT = 128u * 128u;  // [128 queries][64 d] bf16 block
  static constexpr uint32_t META = QBM * 16;   // row records {-lse*log2e, Delta, limit, 0}
  static constexpr uint32_t k = 0;             // CB blocks
  static constexpr uint32_t v = k + CB * KT;
  static constexpr uint32_t q = v + CB * KT;   // [NQS stages][CB blocks]
  static constexpr uint32_t go = q + NQS * CB * QT;
  static constexpr uint32_t meta = go + NQS * CB * QT;  // [NQS stages]
  // the stage's -lse*log2e and Delta as two planes of 128 floats, so that a
  // thread reads four columns' values with one 16-byte load
  static constexpr uint32_t PLANES = 2 * QBM * 4;
  static constexpr uint32_t planes = meta + NQS * META;  // [NQS stages]
  static constexpr uint32_t bars = planes + NQS * PLANES;
  static constexpr uint32_t bytes = bars + 256;
  static constexpr uint32_t alloc = bytes + 1024;
};
static_assert(BwdSmem<128>::alloc <= 227u * 1024u && BwdSmem<64>::alloc <= 227u * 1024u, "shared memory");

enum {
  B_KV = 0,                    // K and V are in shared memory
  B_SFULL = 1,                 // S^T of a pair is in TMEM
  B_SFREE = 2,                 // dV of a pair has read P^T: the S^T buffer is free
  B_DPFULL = 3,                // dP^T of a pair is in TMEM
  B_DPFREE = 4,                // dK of a pair has read dS^T: the dP^T buffer is free
  B_PFULL = 5,                 // P^T is in TMEM (one arrival per compute warp)
  B_DSFULL = 6,                // dS^T is in TMEM (one arrival per compute warp)
  B_DONE = 7,                  // both issuers' last GEMMs have completed
  B_QFULL = 8,                 // [NQS]
  // B_QFREE = B_QFULL + NQS   // [NQS] the pair's dV and dK have read the stage
  // B_RFULL = B_QFULL + 2 NQS // [NQS] the stage's record planes are written
};
__host__ __device__ constexpr int b_count(int nqs) { return B_QFULL + 3 * nqs; }
static_assert(8 * b_count(4) + 16 <= 256, "barrier area");

// Iteration of one key tile over (phase, stream, query range, query tile).
// Phase 0 covers the unmasked ranges (every range but the last when the last
// is the diagonal one) for all streams, phase 1 the diagonal range for all
// streams.  Key tiles of one sequence share the phase-0 sweep (same ranges, same
// order), so CTAs that run at the same time read the same Q / dO tiles within a
// tile or two of each other and share them in L2; the diagonal parts, whose
// lengths differ, come last so they do not shift that sweep.
struct QIter {
  const BaQRange* qr;
  int first, nfull, nall, phase, rr, rrend, ti, sx, nstream;
  BaQRange cur;
  __device__ void init(const BaQRange* q, int f, int n, int ns) {
    qr = q;
    first = f;
    nall = n;
    nstream = ns;
    nfull = (n > 0 && qr[f + n - 1].diag) ? n - 1 : n;
    phase = 0;
    sx = 0;
    if (!start_phase()) {
      phase = 1;
      if (!start_phase()) phase = 2;
    }
  }
  // first range of the current phase for stream sx; false if the phase is empty
  __device__ bool start_phase() {
    rr = phase == 0 ? first : first + nfull;
    rrend = phase == 0 ? first + nfull : first + nall;
    if (rr >= rrend) return false;
    cur = qr[rr];
    ti = cur.t0;
    return true;
  }
  __device__ bool valid() const { return phase < 2; }
  __device__ void next() {
    if (++ti < cur.t1) return;
    if (++rr < rrend) {
      cur = qr[rr];
      ti = cur.t0;
      return;
    }
    if (++sx < nstream) {
      start_phase();
      return;
    }
    sx = 0;
    if (++phase < 2 && start_phase()) return;
    phase = 2;
  }
};

// Packed arithmetic of the compute warps.  P^T and dS^T are GEMM operands in
// bf16, so they are formed two at a time in bf16x2: one fp32x2 FMA for the
// exponent, rounded to bf16x2, one ex2.bf16x2 (two exponentials per MUFU
// instruction), and dS^T = P^T (dP^T - Delta) as one fp32x2 subtraction,
// rounded, times P^T in bf16x2.  The first element of each pair is in the low
// half, which is the column order of a packed TMEM operand.
__device__ __forceinline__ uint32_t fma2_bf16x2(float a0, float a1, float b, float c0, float c1) {
  uint32_t h;
  asm("{\n .reg .b64 a, bb, cc, d;\n .reg .f32 d0, d1;\n"
      " mov.b64 a, {%1, %2};\n mov.b64 bb, {%3, %3};\n mov.b64 cc, {%4, %5};\n"
      " fma.rn.f32x2 d, a, bb, cc;\n mov.b64 {d0, d1}, d;\n"
      " cvt.rn.bf16x2.f32 %0, d1, d0;\n}\n"
      : "=r"(h)
      : "f"(a0), "f"(a1), "f"(b), "f"(c0), "f"(c1));
  return h;
}
__device__ __forceinline__ uint32_t ex2_bf16x2(uint32_t x) {
  uint32_t y;
  asm("ex2.approx.ftz.bf16x2 %0, %1;\n" : "=r"(y) : "r"(x));
  return y;
}
__device__ __forceinline__ uint32_t sub2_bf16x2(float a0, float a1, float b0, float b1) {
  uint32_t h;
  asm("{\n .reg .b64 a, b, d;\n .reg .f32 d0, d1;\n"
      " mov.b64 a, {%1, %2};\n mov.b64 b, {%3, %4};\n"
      " sub.rn.f32x2 d, a, b;\n mov.b64 {d0, d1}, d;\n"
      " cvt.rn.bf16x2.f32 %0, d1, d0;\n}\n"
      : "=r"(h)
      : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
  return h;
}
__device__ __forceinline__ uint32_t mul_bf16x2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.bf16x2 %0, %1, %2;\n" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

template <int D>
__global__ void __launch_bounds__(NTHREADS, 1)
    main_bwd_kv_tc_kernel(const BaBwdArgs a, const __grid_constant__ CUtensorMap tmq,
                          const __grid_constant__ CUtensorMap tmdo, const __grid_constant__ CUtensorMap tmk,
                          const __grid_constant__ CUtensorMap tmv, const __grid_constant__ CUtensorMap tmrec) {
  using L = BwdSmem<D>;
  constexpr int CB = L::CB;
  constexpr int NQS = L::NQS;
  constexpr int B_QFREE = B_QFULL + NQS;
  constexpr int B_RFULL = B_QFULL + 2 * NQS;
  constexpr int B_COUNT = b_count(NQS);
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
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // blockIdx.x = (group * Hkv + kvh) * CS + rank in the cluster
  const int crank = int(blockIdx.x % CS);
  const int cid = int(blockIdx.x / CS);
  const int kvh = cid % sh.Hkv;
  const int gi = cid / sh.Hkv;
  if ((gi + 1) * CS > tb.n_bkv) {  // the same for every CTA of the cluster
    if (tid == 0) ba_set_status(tb.status, BA_DEV_BOUNDS);
    return;
  }
  const BaKvTile kt = tb.bkv[tb.border[gi * CS + crank]];
  const int nstream = sh.steps * sh.G;

  if (tid == 0) {
    *abort_flag = 0;
    mbar_init(bar(B_KV), 1);
    mbar_init(bar(B_SFULL), 1);
    mbar_init(bar(B_SFREE), 1);
    mbar_init(bar(B_DPFULL), 1);
    mbar_init(bar(B_DPFREE), 1);
    mbar_init(bar(B_PFULL), 8);
    mbar_init(bar(B_DSFULL), 8);
    mbar_init(bar(B_DONE), 2);
    for (int s = 0; s < NQS; ++s) {
      mbar_init(bar(B_QFULL + s), 1);
      mbar_init(bar(B_QFREE + s), 2);  // one commit from each issuer
      mbar_init(bar(B_RFULL + s), 1);
    }
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
  const uint32_t tS = tmem, tDP = tmem + 128, tDK = tmem + 256, tDV = tmem + 256 + D;
  const bool any = kt.nqr > 0;
  // pairs this CTA visits
  int npairs = 0;
  for (int r = kt.qr0; r < kt.qr0 + kt.nqr; ++r) npairs += (tb.bqr[r].t1 - tb.bqr[r].t0) * nstream;

  if (warp == 8) {
    // ------------------------------------------------------------ loads
    if (lane == 0) {
      tma_prefetch_desc(&tmq);
      tma_prefetch_desc(&tmdo);
      tma_prefetch_desc(&tmk);
      tma_prefetch_desc(&tmv);
      tma_prefetch_desc(&tmrec);
      if (any) {
        mbar_expect_tx(bar(B_KV), 2 * CB * L::KT);
        for (int cb = 0; cb < CB; ++cb) {
          tma_load_3d(sbase + L::k + cb * L::KT, &tmk, bar(B_KV), cb * 64, kvh, kt.pos0);
          tma_load_3d(sbase + L::v + cb * L::KT, &tmv, bar(B_KV), cb * 64, kvh, kt.pos0);
        }
      }
    }
    // Q / dO rows and the record row of pair state `q`
    auto coords = [&](const QIter& q, int& h, int& qrow, int& srow) {
      const BaQTile qt = tb.bq[q.ti];
      const int j = q.sx / sh.G;
      h = kvh * sh.G + q.sx % sh.G;
      qrow = int(int64_t(j) * sh.rows + qt.nrow0);
      srow = int((int64_t(j) * sh.Hq + h) * sh.rows + qt.nrow0);
    };
    QIter it;
    it.init(tb.bqr, kt.qr0, kt.nqr, nstream);
    int h = 0, qrow = 0, srow = 0;
    if (it.valid()) coords(it, h, qrow, srow);
    for (int i = 0; it.valid(); ++i) {
      const int st = i % NQS;
      const uint32_t fb = bar(B_QFULL + st);
      bool ok = true;
      if (lane == 0) {
        // pair i - NQS has left the stage
        ok = mbar_wait(bar(B_QFREE + st), ((i / NQS) & 1) ^ 1, tb.status, abort_flag);
        if (ok) {
          mbar_expect_tx(fb, 2 * CB * L::QT + L::META);
          // the stage's boxes: Q and dO in CB 64-column blocks each, the row records
          for (int cb = 0; cb < CB; ++cb) {
            tma_load_3d(sbase + L::q + (st * CB + cb) * L::QT, &tmq, fb, cb * 64, h, qrow);
            tma_load_3d(sbase + L::go + (st * CB + cb) * L::QT, &tmdo, fb, cb * 64, h, qrow);
          }
          tma_load_2d(sbase + L::meta + st * L::META, &tmrec, fb, 0, srow);
        }
      }
      if (!__shfl_sync(0xffffffffu, ok, 0)) break;
      // the next pair's table entry is read while this stage's loads fly
      it.next();
      if (it.valid()) coords(it, h, qrow, srow);
      // the records as planes: lane l moves columns 4l .. 4l + 3
      if (!mbar_wait_warp(fb, (i / NQS) & 1, tb.status, abort_flag)) break;
      const uint32_t rec = sbase + L::meta + st * L::META + 64 * lane;
      const float4 r0 = lds_f4(rec), r1 = lds_f4(rec + 16), r2 = lds_f4(rec + 32), r3 = lds_f4(rec + 48);
      float4* pl = reinterpret_cast<float4*>(gbase + L::planes + st * L::PLANES);
      pl[lane] = make_float4(r0.x, r1.x, r2.x, r3.x);
      pl[QBM / 4 + lane] = make_float4(r0.y, r1.y, r2.y, r3.y);
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_RFULL + st));
    }
  } else if (warp == 9 || warp == 10) {
    // ------------------------------------------------------------ issuers
    // warp 9: S^T = K Q^T, then dV += P^T dO;  warp 10: dP^T = V dO^T, then dK += dS^T Q
    if (elect_one() && any) {
      constexpr uint32_t id_s = idesc_bf16_f32(128, QBM, false, false);
      constexpr uint32_t id_kv = idesc_bf16_f32(128, D, false, true);
      const bool is_s = warp == 9;
      // operand descriptors, built once: every MMA below adds a constant offset
      const uint64_t da = smem_desc_sw128(sbase + (is_s ? L::k : L::v), 16, 1024);  // K or V (K-major A)
      const uint64_t db = smem_desc_sw128(sbase + (is_s ? L::q : L::go), 16, 1024);  // Q or dO (K-major B)
      // dV reads dO, dK reads Q, both as MN-major B operands (N = d)
      const uint64_t dm = smem_desc_sw128(sbase + (is_s ? L::go : L::q), L::QT, 1024);
      const uint32_t t_first = is_s ? tS : tDP;    // S^T / dP^T, then P^T / dS^T over it
      const uint32_t t_acc = is_s ? tDV : tDK;
      const int full_bar = is_s ? B_SFULL : B_DPFULL, free_bar = is_s ? B_SFREE : B_DPFREE;
      const int ready_bar = is_s ? B_PFULL : B_DSFULL;
      bool ok = mbar_wait(bar(B_KV), 0, tb.status, abort_flag);
      for (int i = 0; ok && i < npairs; ++i) {
        const int qs = i % NQS;
        if (!mbar_wait(bar(B_QFULL + qs), (i / NQS) & 1, tb.status, abort_flag)) break;
        // the buffer is free once pair i - 1's dV (dK) has read what the threads wrote over it
        if (i > 0 && !mbar_wait(bar(free_bar), (i - 1) & 1, tb.status, abort_flag)) break;
        tc_fence_after();
        const uint64_t dbs = desc_add(db, qs * CB * L::QT);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          tc_mma(t_first, desc_add(da, (kk >> 2) * L::KT + (kk & 3) * 32),
                 desc_add(dbs, (kk >> 2) * L::QT + (kk & 3) * 32), id_s, kk > 0);
        tc_commit(bar(full_bar));
        // P^T (dS^T) written by the threads
        if (!mbar_wait(bar(ready_bar), i & 1, tb.status, abort_flag)) break;
        tc_fence_after();
        const uint64_t dms = desc_add(dm, qs * CB * L::QT);
        // queries 16 kk .. 16 kk + 15 sit in query half kk / 4, columns 8 (kk % 4) ..
#pragma unroll
        for (int kk = 0; kk < QBM / 16; ++kk)
          tc_mma_tmem_a(t_acc, t_first + (kk >> 2) * 64 + (kk & 3) * 8, desc_add(dms, kk * 2048), id_kv,
                        (i > 0 || kk > 0) ? 1u : 0u);
        tc_commit(bar(free_bar));
        tc_commit(bar(B_QFREE + qs));
      }
      tc_commit(bar(B_DONE));
    }
  } else if (warp < 8) {
    // ------------------------------------------------------------ compute
    // warp w: TMEM lane quarter w % 4 (key rows 32 (w % 4) ..), query columns
    // 64 (w / 4) .. 64 (w / 4) + 63 of each 128-query tile
    const int quarter = warp & 3, half = warp >> 2;
    const int row = quarter * 32 + lane;
    const int col0 = half * 64;
    const uint32_t lane_off = uint32_t(quarter * 32) << 16;
    const bool kok = row < kt.nkeys;
    const int kpos = kt.pos0 + row;
    QIter it;
    it.init(tb.bqr, kt.qr0, kt.nqr, nstream);
    bool ok = true;
    int i = 0;
    for (; it.valid(); ++i, it.next()) {
      const int qs = i % NQS;
      const uint32_t ph = i & 1;
      const int nrows = tb.bq[it.ti].nrows;
      const bool diag = it.cur.diag != 0;
      // the row records of this tile (and their planes) are in shared memory
      if (!mbar_wait_warp(bar(B_RFULL + qs), (i / NQS) & 1, tb.status, abort_flag)) { ok = false; break; }
      if (!mbar_wait_warp(bar(B_SFULL), ph, tb.status, abort_flag)) { ok = false; break; }
      tc_fence_after();
      float p[64];
      tmem_ld32(tS + lane_off + col0, p);
      tmem_ld32(tS + lane_off + col0 + 32, p + 32);
      tmem_wait_ld();
      // row records {-lse*log2e, Delta, limit, 0}; queries past the tile are masked
      const uint32_t rec = sbase + L::meta + qs * L::META + 16 * col0;
      const uint32_t pln = sbase + L::planes + qs * L::PLANES + 4 * col0;  // -lse*log2e; Delta at + 4 QBM
      const int nq = nrows - col0;
      uint32_t pb[32];  // P^T, bf16 pairs
      if (!diag && kok && nq >= 64) {
        // full tile (the common case): no mask
#pragma unroll
        for (int c = 0; c < 64; c += 4) {
          const float4 n = lds_f4(pln + 4 * c);
          pb[c >> 1] = ex2_bf16x2(fma2_bf16x2(p[c], p[c + 1], sh.scale_log2, n.x, n.y));
          pb[(c >> 1) + 1] = ex2_bf16x2(fma2_bf16x2(p[c + 2], p[c + 3], sh.scale_log2, n.z, n.w));
        }
      } else {
#pragma unroll
        for (int c = 0; c < 64; c += 2) {
          const float4 r0 = lds_f4(rec + 16 * c), r1 = lds_f4(rec + 16 * (c + 1));
          const bool v0 = kok && c < nq && (!diag || kpos <= __float_as_int(r0.z));
          const bool v1 = kok && c + 1 < nq && (!diag || kpos <= __float_as_int(r1.z));
          const float e0 = ex2_approx(fmaf(p[c], sh.scale_log2, r0.x));
          const float e1 = ex2_approx(fmaf(p[c + 1], sh.scale_log2, r1.x));
          pb[c >> 1] = pack_bf16(v0 ? e0 : 0.f, v1 ? e1 : 0.f);
        }
      }
      // P^T over the first 32 of this warp's 64 columns of the S^T buffer
      tmem_st16(tS + lane_off + col0, pb);
      tmem_st16(tS + lane_off + col0 + 16, pb + 16);
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_PFULL));
      // dS^T = P^T (dP^T - Delta), over the first 32 of this warp's columns of
      // the dP^T buffer: columns 0..31 are loaded before 0..15 are written,
      // 32..63 before 16..31
      if (!mbar_wait_warp(bar(B_DPFULL), ph, tb.status, abort_flag)) { ok = false; break; }
      tc_fence_after();
#pragma unroll
      for (int g = 0; g < 2; ++g) {
        float dp[32];
        tmem_ld32(tDP + lane_off + col0 + 32 * g, dp);
        tmem_wait_ld();
        uint32_t w[16];
#pragma unroll
        for (int e = 0; e < 16; e += 2) {
          const float4 d4 = lds_f4(pln + 4 * QBM + 4 * (32 * g + 2 * e));
          w[e] = mul_bf16x2(pb[16 * g + e], sub2_bf16x2(dp[2 * e], dp[2 * e + 1], d4.x, d4.y));
          w[e + 1] = mul_bf16x2(pb[16 * g + e + 1], sub2_bf16x2(dp[2 * e + 2], dp[2 * e + 3], d4.z, d4.w));
        }
        tmem_st16(tDP + lane_off + col0 + 16 * g, w);
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_DSFULL));
    }
    // epilogue: dK (scaled) and dV of this key tile, natural order; each warp
    // writes d-columns (d / 2) (w / 4) .. (d / 2) (w / 4) + d / 2 - 1 of its 32 key rows
    auto* dkm = static_cast<__nv_bfloat16*>(a.dkm);
    auto* dvm = static_cast<__nv_bfloat16*>(a.dvm);
    const bool have = any && ok && i > 0 && mbar_wait_warp(bar(B_DONE), 0, tb.status, abort_flag);
    if (have) tc_fence_after();
    constexpr int HD = D / 2;
    const int64_t base = kok ? (int64_t(kt.pos0 + row) * sh.Hkv + kvh) * D + half * HD : 0;
#pragma unroll
    for (int c = 0; c < HD / 32; ++c) {
      float xk[32], xv[32];
      if (have) {
        tmem_ld32(tDK + lane_off + half * HD + c * 32, xk);
        tmem_ld32(tDV + lane_off + half * HD + c * 32, xv);
        tmem_wait_ld();
      } else {
#pragma unroll
        for (int e = 0; e < 32; ++e) xk[e] = xv[e] = 0.f;
      }
      if (kok && (have || !any) && a.dkm_acc) {
        // single-step call: add into the fp32 accumulators (this CTA owns the rows)
        float4* ak = reinterpret_cast<float4*>(a.dkm_acc + base + c * 32);
        float4* av = reinterpret_cast<float4*>(a.dvm_acc + base + c * 32);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const float4 k0 = ak[e], v0 = av[e];
          ak[e] = make_float4(k0.x + sh.scale * xk[4 * e], k0.y + sh.scale * xk[4 * e + 1],
                              k0.z + sh.scale * xk[4 * e + 2], k0.w + sh.scale * xk[4 * e + 3]);
          av[e] = make_float4(v0.x + xv[4 * e], v0.y + xv[4 * e + 1], v0.z + xv[4 * e + 2], v0.w + xv[4 * e + 3]);
        }
      } else if (kok && (have || !any)) {
        uint4* pk = reinterpret_cast<uint4*>(dkm + base + c * 32);
        uint4* pv = reinterpret_cast<uint4*>(dvm + base + c * 32);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          pk[e] = make_uint4(pack_bf16(sh.scale * xk[8 * e], sh.scale * xk[8 * e + 1]),
                             pack_bf16(sh.scale * xk[8 * e + 2], sh.scale * xk[8 * e + 3]),
                             pack_bf16(sh.scale * xk[8 * e + 4], sh.scale * xk[8 * e + 5]),
                             pack_bf16(sh.scale * xk[8 * e + 6], sh.scale * xk[8 * e + 7]));
          pv[e] = make_uint4(pack_bf16(xv[8 * e], xv[8 * e + 1]), pack_bf16(xv[8 * e + 2], xv[8 * e + 3]),
                             pack_bf16(xv[8 * e + 4], xv[8 * e + 5]), pack_bf16(xv[8 * e + 6], xv[8 * e + 7]));
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  // after a failed wait, give copies, MMAs and commits already in flight time
  // to land before TMEM is released and the CTA leaves
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

// 3-D view (d, heads, rows) of a row-major [rows][heads][d] tensor.
cudaError_t map3d(CUtensorMap* m, const void* base, CUtensorMapDataType dt, int esize, int d, int heads, int64_t rows,
                  uint32_t box0, uint32_t box2, CUtensorMapSwizzle sw) {
  const cuuint64_t dims[3] = {cuuint64_t(d), cuuint64_t(heads), cuuint64_t(rows)};
  const cuuint64_t strides[2] = {cuuint64_t(d) * esize, cuuint64_t(heads) * d * esize};
  const cuuint32_t box[3] = {box0, 1, box2};
  const cuuint32_t es[3] = {1, 1, 1};
  const CUresult r = g_encode(m, dt, 3, const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                              sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

template <int D>
cudaError_t launch_kv(const BaBwdArgs& a, int64_t grid, cudaStream_t st) {
  const int64_t qrows = int64_t(a.sh.steps) * a.sh.rows;
  CUtensorMap mq, mdo, mk, mv;
  const auto bf = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const auto sw = CU_TENSOR_MAP_SWIZZLE_128B;
  cudaError_t e;
  if ((e = map3d(&mq, a.q, bf, 2, D, a.sh.Hq, qrows, 64, QBM, sw)) != cudaSuccess) return e;
  if ((e = map3d(&mdo, a.d_o, bf, 2, D, a.sh.Hq, qrows, 64, QBM, sw)) != cudaSuccess) return e;
  if ((e = map3d(&mk, a.km, bf, 2, D, a.sh.Hkv, a.sh.T, 64, KBN, sw)) != cudaSuccess) return e;
  if ((e = map3d(&mv, a.vm, bf, 2, D, a.sh.Hkv, a.sh.T, 64, KBN, sw)) != cudaSuccess) return e;
  CUtensorMap mrec;
  {
    const cuuint64_t dims[2] = {4, cuuint64_t(qrows) * a.sh.Hq};
    const cuuint64_t strides[1] = {16};
    const cuuint32_t box[2] = {4, QBM};
    const cuuint32_t es[2] = {1, 1};
    if (g_encode(&mrec, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, a.rowrec, dims, strides, box, es,
                 CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                 CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  const int smem = int(BwdSmem<D>::alloc);
  if ((e = cudaFuncSetAttribute(main_bwd_kv_tc_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem)) !=
      cudaSuccess)
    return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(grid));
  cfg.blockDim = dim3(NTHREADS);
  cfg.dynamicSmemBytes = size_t(smem);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = CS;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if ((e = cudaLaunchKernelEx(&cfg, main_bwd_kv_tc_kernel<D>, a, mq, mdo, mk, mv, mrec)) != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace

cudaError_t ba_launch_main_bwd_kv_tc(const BaBwdArgs& a, cudaStream_t st) {
  const int64_t grid = int64_t(a.tb.n_bkv) * a.sh.Hkv;
  if (grid == 0) return cudaSuccess;
  if (grid > 0x7fffffffLL || grid % CS != 0 || (a.sh.d != 128 && a.sh.d != 64)) return cudaErrorInvalidConfiguration;
  cudaError_t e = encoder();
  if (e != cudaSuccess) return e;
  return a.sh.d == 128 ? launch_kv<128>(a, grid, st) : launch_kv<64>(a, grid, st);
}
