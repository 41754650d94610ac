// K2 (legacy tensor path) — causal main-sequence attention forward with
// mma.sync m16n8k16 bf16.  Correctness path and the baseline the tcgen05
// kernel is measured against.
//
// "Online Draft Co-Training ...", ai.info summary, "Methodology in Plain
// English": the main part behaves like ordinary causal context parallelism —
// zigzag-ring attention where K/V circulate and queries stay put, partials
// merged with the log-sum-exp trick between ring steps.  On one GPU a query
// tile walks the key segments the planner lists for it in ring order
// (step s: chunks of rank (r - s) mod C), and the online softmax carried across
// the segments is exactly that between-step merge.
//
// CTA: 128 query rows of one query stream (step j, head h) x blocks of 64
// keys; 8 warps, 16 rows each.  K/V blocks are double-buffered with cp.async.
// Output: O_m (fp32, normalised) and l_m (natural log) in packed order.
#include <math.h>

#include "device.cuh"
#include "kernels.h"

namespace {

constexpr int FBM = 128;
constexpr int FBN = 64;

template <int D>
__global__ void __launch_bounds__(256, 1) main_fwd_mma_kernel(BaFwdArgs a) {
  constexpr int LD = D + 8;
  constexpr int CH = D / 8;  // 16-byte chunks per row
  extern __shared__ __align__(16) unsigned char smem_raw[];
  __nv_bfloat16* Qs = reinterpret_cast<__nv_bfloat16*>(smem_raw);
  __nv_bfloat16* Ks = Qs + FBM * LD;
  __nv_bfloat16* Vs = Ks + 2 * FBN * LD;

  const BaShape& sh = a.sh;
  const BaTables& tb = a.tb;
  const int nstreams = sh.steps * sh.Hq;
  const int si = int(blockIdx.x % nstreams);
  const int oi = int(blockIdx.x / nstreams);
  if (oi >= tb.n_fq) { ba_set_status(tb.status, BA_DEV_BOUNDS); return; }
  const BaQTile tile = tb.fq[tb.forder[oi]];
  const int kvh = si / (sh.steps * sh.G);
  const int rem = si % (sh.steps * sh.G);
  const int j = rem / sh.G;
  const int h = kvh * sh.G + rem % sh.G;

  const auto* qg = static_cast<const __nv_bfloat16*>(a.q);
  const auto* kmg = static_cast<const __nv_bfloat16*>(a.km);
  const auto* vmg = static_cast<const __nv_bfloat16*>(a.vm);
  const int64_t qstride = int64_t(sh.Hq) * D;
  const __nv_bfloat16* qbase = qg + (int64_t(j) * sh.rows * sh.Hq + h) * D;
  const int64_t kstride = int64_t(sh.Hkv) * D;
  const __nv_bfloat16* kbase = kmg + int64_t(kvh) * D;
  const __nv_bfloat16* vbase = vmg + int64_t(kvh) * D;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, t4 = lane & 3;

  // Q tile -> smem (rows past the tile read as zero)
  for (int c = tid; c < FBM * CH; c += 256) {
    const int r = c / CH, col = (c % CH) * 8;
    const bool ok = r < tile.nrows;
    const __nv_bfloat16* src = qbase + int64_t(tile.nrow0 + (ok ? r : 0)) * qstride + col;
    cp_async16(smem_u32(Qs + r * LD + col), src, ok ? 16 : 0);
  }
  cp_async_commit();

  auto load_kv = [&](const BaKvSeg& sg, int kb, int buf) {
    __nv_bfloat16* kd = Ks + buf * FBN * LD;
    __nv_bfloat16* vd = Vs + buf * FBN * LD;
    for (int c = tid; c < FBN * CH; c += 256) {
      const int r = c / CH, col = (c % CH) * 8;
      const bool ok = kb + r < sg.nkeys;
      const int64_t key = int64_t(sg.pos0) + (ok ? kb + r : 0);
      cp_async16(smem_u32(kd + r * LD + col), kbase + key * kstride + col, ok ? 16 : 0);
      cp_async16(smem_u32(vd + r * LD + col), vbase + key * kstride + col, ok ? 16 : 0);
    }
  };

  const int rA = warp * 16 + g, rB = rA + 8;
  const int limA = rA < tile.nrows ? tb.row_lim[tile.row0 + rA] : -1;
  const int limB = rB < tile.nrows ? tb.row_lim[tile.row0 + rB] : -1;

  float acc[D / 8][4];
#pragma unroll
  for (int i = 0; i < D / 8; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
  float mA = -INFINITY, mB = -INFINITY, lA = 0.f, lB = 0.f;
  uint32_t qf[D / 16][4];

  int seg = tile.seg0;
  const int segend = tile.seg0 + tile.nseg;
  if (seg >= segend) return;
  BaKvSeg sg = tb.fseg[seg];
  int kb = 0, buf = 0;
  load_kv(sg, kb, buf);
  cp_async_commit();
  for (int it = 0;; ++it) {
    int nseg = seg, nkb = kb + FBN;
    if (nkb >= sg.nkeys) { ++nseg; nkb = 0; }
    const bool has_next = nseg < segend;
    BaKvSeg nsg = sg;
    if (has_next) {
      nsg = tb.fseg[nseg];
      load_kv(nsg, nkb, buf ^ 1);
    }
    cp_async_commit();
    cp_async_wait<1>();
    __syncthreads();
    if (it == 0) {
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk)
        ldsm_x4(smem_u32(Qs + (warp * 16 + (lane & 15)) * LD + kk * 16 + (lane >> 4) * 8), qf[kk][0], qf[kk][1],
                qf[kk][2], qf[kk][3]);
    }
    const __nv_bfloat16* kt = Ks + buf * FBN * LD;
    const __nv_bfloat16* vt = Vs + buf * FBN * LD;

    // S = Q K^T (16 x 64 per warp)
    float s[8][4];
#pragma unroll
    for (int i = 0; i < 8; ++i) s[i][0] = s[i][1] = s[i][2] = s[i][3] = 0.f;
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
#pragma unroll
      for (int np = 0; np < 4; ++np) {
        uint32_t b0, b1, b2, b3;
        ldsm_x4(smem_u32(kt + (np * 16 + (lane & 7) + (lane >> 4) * 8) * LD + kk * 16 + ((lane >> 3) & 1) * 8), b0,
                b1, b2, b3);
        mma_bf16(s[2 * np], qf[kk], b0, b1);
        mma_bf16(s[2 * np + 1], qf[kk], b2, b3);
      }
    }
    // scale, mask (ragged block end; per-row causal limit on the diagonal)
    const bool ragged = kb + FBN > sg.nkeys;
#pragma unroll
    for (int nt = 0; nt < 8; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int col = nt * 8 + 2 * t4 + (e & 1);
        float v = s[nt][e] * sh.scale_log2;
        if (ragged || sg.diag) {
          const int koff = kb + col;
          const int lim = (e >> 1) ? limB : limA;
          const bool ok = koff < sg.nkeys && (!sg.diag || sg.pos0 + koff <= lim);
          if (!ok) v = -INFINITY;
        }
        s[nt][e] = v;
      }
    // online softmax (base 2)
    float xA = -INFINITY, xB = -INFINITY;
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
      xA = fmaxf(xA, fmaxf(s[nt][0], s[nt][1]));
      xB = fmaxf(xB, fmaxf(s[nt][2], s[nt][3]));
    }
    xA = fmaxf(xA, __shfl_xor_sync(0xffffffffu, xA, 1));
    xA = fmaxf(xA, __shfl_xor_sync(0xffffffffu, xA, 2));
    xB = fmaxf(xB, __shfl_xor_sync(0xffffffffu, xB, 1));
    xB = fmaxf(xB, __shfl_xor_sync(0xffffffffu, xB, 2));
    const float nA = fmaxf(mA, xA), nB = fmaxf(mB, xB);
    const float bA = nA == -INFINITY ? 0.f : nA, bB = nB == -INFINITY ? 0.f : nB;
    const float cA = exp2f(mA - bA), cB = exp2f(mB - bB);
    mA = nA;
    mB = nB;
    float sA = 0.f, sB = 0.f;
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
      s[nt][0] = exp2f(s[nt][0] - bA);
      s[nt][1] = exp2f(s[nt][1] - bA);
      s[nt][2] = exp2f(s[nt][2] - bB);
      s[nt][3] = exp2f(s[nt][3] - bB);
      sA += s[nt][0] + s[nt][1];
      sB += s[nt][2] + s[nt][3];
    }
    lA = lA * cA + sA;
    lB = lB * cB + sB;
#pragma unroll
    for (int i = 0; i < D / 8; ++i) {
      acc[i][0] *= cA;
      acc[i][1] *= cA;
      acc[i][2] *= cB;
      acc[i][3] *= cB;
    }
    // O += P V
#pragma unroll
    for (int kq = 0; kq < 4; ++kq) {
      uint32_t pa[4];
      pa[0] = pack_bf16(s[2 * kq][0], s[2 * kq][1]);
      pa[1] = pack_bf16(s[2 * kq][2], s[2 * kq][3]);
      pa[2] = pack_bf16(s[2 * kq + 1][0], s[2 * kq + 1][1]);
      pa[3] = pack_bf16(s[2 * kq + 1][2], s[2 * kq + 1][3]);
#pragma unroll
      for (int dp = 0; dp < D / 16; ++dp) {
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(smem_u32(vt + (kq * 16 + (lane & 7) + ((lane >> 3) & 1) * 8) * LD + dp * 16 + (lane >> 4) * 8), b0,
                  b1, b2, b3);
        mma_bf16(acc[2 * dp], pa, b0, b1);
        mma_bf16(acc[2 * dp + 1], pa, b2, b3);
      }
    }
    __syncthreads();
    if (!has_next) break;
    seg = nseg;
    kb = nkb;
    sg = nsg;
    buf ^= 1;
  }

  lA += __shfl_xor_sync(0xffffffffu, lA, 1);
  lA += __shfl_xor_sync(0xffffffffu, lA, 2);
  lB += __shfl_xor_sync(0xffffffffu, lB, 1);
  lB += __shfl_xor_sync(0xffffffffu, lB, 2);
  const int64_t rowbase = int64_t(j) * sh.rows + tile.nrow0;
  if (rA < tile.nrows) {
    const int64_t qrow = (rowbase + rA) * sh.Hq + h;
    const float inv = lA > 0.f ? 1.f / lA : 0.f;
#pragma unroll
    for (int dt = 0; dt < D / 8; ++dt)
      *reinterpret_cast<float2*>(a.om + qrow * D + dt * 8 + 2 * t4) = make_float2(acc[dt][0] * inv, acc[dt][1] * inv);
    if (t4 == 0) a.lm[qrow] = lA > 0.f ? (mA + log2f(lA)) * BA_LN2 : -INFINITY;
  }
  if (rB < tile.nrows) {
    const int64_t qrow = (rowbase + rB) * sh.Hq + h;
    const float inv = lB > 0.f ? 1.f / lB : 0.f;
#pragma unroll
    for (int dt = 0; dt < D / 8; ++dt)
      *reinterpret_cast<float2*>(a.om + qrow * D + dt * 8 + 2 * t4) = make_float2(acc[dt][2] * inv, acc[dt][3] * inv);
    if (t4 == 0) a.lm[qrow] = lB > 0.f ? (mB + log2f(lB)) * BA_LN2 : -INFINITY;
  }
}

}  // namespace

cudaError_t ba_launch_main_fwd(const BaFwdArgs& a, cudaStream_t st) {
  const int64_t grid = int64_t(a.tb.n_fq) * a.sh.steps * a.sh.Hq;
  if (grid == 0) return cudaSuccess;
  if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  if (a.sh.d == 128) {
    const int smem = (FBM + 4 * FBN) * (128 + 8) * 2;
    if (cudaError_t e = set_dynamic_smem(main_fwd_mma_kernel<128>, size_t(smem)); e != cudaSuccess) return e;
    main_fwd_mma_kernel<128><<<unsigned(grid), 256, smem, st>>>(a);
  } else {
    const int smem = (FBM + 4 * FBN) * (64 + 8) * 2;
    if (cudaError_t e = set_dynamic_smem(main_fwd_mma_kernel<64>, size_t(smem)); e != cudaSuccess) return e;
    main_fwd_mma_kernel<64><<<unsigned(grid), 256, smem, st>>>(a);
  }
  return cudaGetLastError();
}
