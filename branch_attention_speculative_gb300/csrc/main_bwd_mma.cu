// K6 (legacy tensor path) — causal main-sequence attention backward with
// mma.sync m16n8k16 bf16, key-stationary.
//
// "Online Draft Co-Training ...", rainbus page, method step 5 and core method:
// the backward replays the same ring and accumulates gradients locally.  On
// one GPU a key tile (128 keys of one kv head, inside one zigzag chunk) meets
// the query tiles of rank (r + s) mod C at replay step s, in the order the
// planner lists them, for every query stream (step j, q head) of its group.
// P is recomputed from the merged lse: the merged result is the single softmax
// over main and branch keys, so P_ij = exp(scale q_i.k_j - l_i) is already the
// full-softmax probability and dS = P * (dP - Delta) splits by key set.
//
// CTA: 8 warps over a 128-key tile, warp w owns keys 16w..16w+15: it computes
// S^T and dP^T for its keys against a 64-row query tile, accumulates dV and dK
// in registers, and writes its dS^T to shared memory; then each warp forms 16
// rows x d/2 columns of dQ = dS K and adds them (scaled) into the fp32 dQ
// accumulator with atomics.
// Query/dO tiles are double-buffered with cp.async.
#include <math.h>

#include "device.cuh"
#include "kernels.h"

namespace {

constexpr int QB = 64;   // queries per tile (BA_BWD_BM)
constexpr int KB = 128;  // keys per tile (BA_BWD_BN)
constexpr int NT = 256;  // 8 warps, 16 keys each

template <int D>
struct BwdSmem {
  static constexpr int LD = D + 8;
  static constexpr int LDS = QB + 8;
  static constexpr size_t k = 0;
  static constexpr size_t v = k + size_t(KB) * LD * 2;
  static constexpr size_t q = v + size_t(KB) * LD * 2;
  static constexpr size_t go = q + size_t(2) * QB * LD * 2;
  static constexpr size_t ds = go + size_t(2) * QB * LD * 2;
  static constexpr size_t l2 = ds + size_t(KB) * LDS * 2;
  static constexpr size_t dl = l2 + size_t(2) * QB * 4;
  static constexpr size_t lim = dl + size_t(2) * QB * 4;
  static constexpr size_t bytes = lim + size_t(2) * QB * 4;
};

template <int D>
__global__ void __launch_bounds__(NT, 1) main_bwd_mma_kernel(BaBwdArgs a) {
  using L = BwdSmem<D>;
  constexpr int LD = L::LD, LDS = L::LDS, CH = D / 8;
  extern __shared__ __align__(16) unsigned char smem_raw[];
  auto* Ks = reinterpret_cast<__nv_bfloat16*>(smem_raw + L::k);
  auto* Vs = reinterpret_cast<__nv_bfloat16*>(smem_raw + L::v);
  auto* Qs = reinterpret_cast<__nv_bfloat16*>(smem_raw + L::q);
  auto* Gs = reinterpret_cast<__nv_bfloat16*>(smem_raw + L::go);
  auto* Ss = reinterpret_cast<__nv_bfloat16*>(smem_raw + L::ds);
  auto* L2s = reinterpret_cast<float*>(smem_raw + L::l2);
  auto* Dls = reinterpret_cast<float*>(smem_raw + L::dl);
  auto* Lims = reinterpret_cast<int*>(smem_raw + L::lim);

  const BaShape& sh = a.sh;
  const BaTables& tb = a.tb;
  const int kvh = int(blockIdx.x % sh.Hkv);
  const int oi = int(blockIdx.x / sh.Hkv);
  if (oi >= tb.n_bkv) { ba_set_status(tb.status, BA_DEV_BOUNDS); return; }
  const BaKvTile kt = tb.bkv[tb.border[oi]];
  const int nstream = sh.steps * sh.G;

  const auto* qg = static_cast<const __nv_bfloat16*>(a.q);
  const auto* dog = static_cast<const __nv_bfloat16*>(a.d_o);
  const auto* kmg = static_cast<const __nv_bfloat16*>(a.km);
  const auto* vmg = static_cast<const __nv_bfloat16*>(a.vm);
  const int64_t kstride = int64_t(sh.Hkv) * D;
  const int64_t qstride = int64_t(sh.Hq) * D;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, t4 = lane & 3;

  for (int c = tid; c < KB * CH; c += NT) {
    const int r = c / CH, col = (c % CH) * 8;
    const bool ok = r < kt.nkeys;
    const int64_t key = int64_t(kt.pos0) + (ok ? r : 0);
    cp_async16(smem_u32(Ks + r * LD + col), kmg + key * kstride + int64_t(kvh) * D + col, ok ? 16 : 0);
    cp_async16(smem_u32(Vs + r * LD + col), vmg + key * kstride + int64_t(kvh) * D + col, ok ? 16 : 0);
  }
  cp_async_commit();

  // iteration state: (query range, query tile, stream)
  int rr = kt.qr0, ti = 0, sidx = 0;
  const int rrend = kt.qr0 + kt.nqr;
  BaQRange range{0, 0, 0, 0};
  if (rr < rrend) {
    range = tb.bqr[rr];
    ti = range.t0;
  }

  auto load_q = [&](int tix, int sx, int buf) {
    const BaQTile qt = tb.bq[tix];
    const int j = sx / sh.G, h = kvh * sh.G + sx % sh.G;
    const int64_t base = (int64_t(j) * sh.rows * sh.Hq + h) * D;
    __nv_bfloat16* qd = Qs + buf * QB * LD;
    __nv_bfloat16* gd = Gs + buf * QB * LD;
    for (int c = tid; c < QB * CH; c += NT) {
      const int r = c / CH, col = (c % CH) * 8;
      const bool ok = r < qt.nrows;
      const int64_t off = base + int64_t(qt.nrow0 + (ok ? r : 0)) * qstride + col;
      cp_async16(smem_u32(qd + r * LD + col), qg + off, ok ? 16 : 0);
      cp_async16(smem_u32(gd + r * LD + col), dog + off, ok ? 16 : 0);
    }
    for (int r = tid; r < QB; r += NT) {
      const bool ok = r < qt.nrows;
      const int64_t srow = (int64_t(j) * sh.Hq + h) * sh.rows + qt.nrow0 + (ok ? r : 0);
      const float4 rec = a.rowrec[srow];
      L2s[buf * QB + r] = ok ? rec.x : INFINITY;
      Dls[buf * QB + r] = ok ? rec.y : 0.f;
      Lims[buf * QB + r] = ok ? tb.row_lim[qt.row0 + r] : -1;
    }
  };

  float dk[D / 8][4], dv[D / 8][4];
#pragma unroll
  for (int i = 0; i < D / 8; ++i) {
    dk[i][0] = dk[i][1] = dk[i][2] = dk[i][3] = 0.f;
    dv[i][0] = dv[i][1] = dv[i][2] = dv[i][3] = 0.f;
  }
  const int kA = warp * 16 + g, kB = kA + 8;
  const bool kokA = kA < kt.nkeys, kokB = kB < kt.nkeys;
  const int posA = kt.pos0 + kA, posB = kt.pos0 + kB;

  int buf = 0;
  if (rr < rrend) load_q(ti, sidx, buf);
  cp_async_commit();
  // a key tile that no query sees keeps zero gradients
  for (; rr < rrend;) {
    // next iteration
    int nrr = rr, nti = ti, nsx = sidx + 1;
    BaQRange nrange = range;
    if (nsx == nstream) {
      nsx = 0;
      ++nti;
      if (nti >= range.t1) {
        ++nrr;
        if (nrr < rrend) {
          nrange = tb.bqr[nrr];
          nti = nrange.t0;
        }
      }
    }
    const bool has_next = nrr < rrend;
    if (has_next) load_q(nti, nsx, buf ^ 1);
    cp_async_commit();
    cp_async_wait<1>();
    __syncthreads();

    const BaQTile qt = tb.bq[ti];
    const int j = sidx / sh.G, h = kvh * sh.G + sidx % sh.G;
    const __nv_bfloat16* qs = Qs + buf * QB * LD;
    const __nv_bfloat16* gs = Gs + buf * QB * LD;
    const float* l2 = L2s + buf * QB;
    const float* dl = Dls + buf * QB;
    const int* lim = Lims + buf * QB;

    // S^T = K_w Q^T and dP^T = V_w dO^T  (16 keys x 64 queries per warp)
    float st[8][4], dpt[8][4];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      st[i][0] = st[i][1] = st[i][2] = st[i][3] = 0.f;
      dpt[i][0] = dpt[i][1] = dpt[i][2] = dpt[i][3] = 0.f;
    }
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      uint32_t ka[4], va[4];
      ldsm_x4(smem_u32(Ks + (warp * 16 + (lane & 15)) * LD + kk * 16 + (lane >> 4) * 8), ka[0], ka[1], ka[2], ka[3]);
      ldsm_x4(smem_u32(Vs + (warp * 16 + (lane & 15)) * LD + kk * 16 + (lane >> 4) * 8), va[0], va[1], va[2], va[3]);
#pragma unroll
      for (int np = 0; np < 4; ++np) {
        const int off = (np * 16 + (lane & 7) + (lane >> 4) * 8) * LD + kk * 16 + ((lane >> 3) & 1) * 8;
        uint32_t b0, b1, b2, b3;
        ldsm_x4(smem_u32(qs + off), b0, b1, b2, b3);
        mma_bf16(st[2 * np], ka, b0, b1);
        mma_bf16(st[2 * np + 1], ka, b2, b3);
        ldsm_x4(smem_u32(gs + off), b0, b1, b2, b3);
        mma_bf16(dpt[2 * np], va, b0, b1);
        mma_bf16(dpt[2 * np + 1], va, b2, b3);
      }
    }
    // P^T and dS^T
    const bool diag = tb.bqr[rr].diag != 0;
#pragma unroll
    for (int nt = 0; nt < 8; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int q = nt * 8 + 2 * t4 + (e & 1);
        const bool kok = (e >> 1) ? kokB : kokA;
        const int pos = (e >> 1) ? posB : posA;
        const bool ok = kok && q < qt.nrows && (!diag || pos <= lim[q]);
        const float p = ok ? exp2f(st[nt][e] * sh.scale_log2 - l2[q]) : 0.f;
        st[nt][e] = p;
        dpt[nt][e] = p * (dpt[nt][e] - dl[q]);
      }
    // dV += P^T dO ; dK += dS^T Q
#pragma unroll
    for (int kq = 0; kq < 4; ++kq) {
      uint32_t pa[4], sa[4];
      pa[0] = pack_bf16(st[2 * kq][0], st[2 * kq][1]);
      pa[1] = pack_bf16(st[2 * kq][2], st[2 * kq][3]);
      pa[2] = pack_bf16(st[2 * kq + 1][0], st[2 * kq + 1][1]);
      pa[3] = pack_bf16(st[2 * kq + 1][2], st[2 * kq + 1][3]);
      sa[0] = pack_bf16(dpt[2 * kq][0], dpt[2 * kq][1]);
      sa[1] = pack_bf16(dpt[2 * kq][2], dpt[2 * kq][3]);
      sa[2] = pack_bf16(dpt[2 * kq + 1][0], dpt[2 * kq + 1][1]);
      sa[3] = pack_bf16(dpt[2 * kq + 1][2], dpt[2 * kq + 1][3]);
#pragma unroll
      for (int dp = 0; dp < D / 16; ++dp) {
        const int off = (kq * 16 + (lane & 7) + ((lane >> 3) & 1) * 8) * LD + dp * 16 + (lane >> 4) * 8;
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(smem_u32(gs + off), b0, b1, b2, b3);
        mma_bf16(dv[2 * dp], pa, b0, b1);
        mma_bf16(dv[2 * dp + 1], pa, b2, b3);
        ldsm_x4_t(smem_u32(qs + off), b0, b1, b2, b3);
        mma_bf16(dk[2 * dp], sa, b0, b1);
        mma_bf16(dk[2 * dp + 1], sa, b2, b3);
      }
    }
    // dS^T -> shared (bf16), keys x queries
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
      const int q = nt * 8 + 2 * t4;
      *reinterpret_cast<uint32_t*>(Ss + kA * LDS + q) = pack_bf16(dpt[nt][0], dpt[nt][1]);
      *reinterpret_cast<uint32_t*>(Ss + kB * LDS + q) = pack_bf16(dpt[nt][2], dpt[nt][3]);
    }
    __syncthreads();
    // dQ = dS K: warp w takes query rows 16(w % 4).. and d-half w / 4
    const int qw = warp & 3, half = warp >> 2;
    const int qA = qw * 16 + g, qB = qA + 8;
    const int64_t rowA = (int64_t(j) * sh.rows + qt.nrow0 + qA) * sh.Hq + h;
    const int64_t rowB = (int64_t(j) * sh.rows + qt.nrow0 + qB) * sh.Hq + h;
    {
      float dq[D / 16][4];
#pragma unroll
      for (int i = 0; i < D / 16; ++i) dq[i][0] = dq[i][1] = dq[i][2] = dq[i][3] = 0.f;
#pragma unroll
      for (int kq = 0; kq < KB / 16; ++kq) {
        uint32_t aa[4];
        ldsm_x4_t(smem_u32(Ss + (kq * 16 + (lane & 7) + (lane >> 4) * 8) * LDS + qw * 16 + ((lane >> 3) & 1) * 8),
                  aa[0], aa[1], aa[2], aa[3]);
#pragma unroll
        for (int dp = 0; dp < D / 32; ++dp) {
          uint32_t b0, b1, b2, b3;
          ldsm_x4_t(smem_u32(Ks + (kq * 16 + (lane & 7) + ((lane >> 3) & 1) * 8) * LD + half * (D / 2) + dp * 16 +
                             (lane >> 4) * 8),
                    b0, b1, b2, b3);
          mma_bf16(dq[2 * dp], aa, b0, b1);
          mma_bf16(dq[2 * dp + 1], aa, b2, b3);
        }
      }
#pragma unroll
      for (int dt = 0; dt < D / 16; ++dt) {
        const int col = half * (D / 2) + dt * 8 + 2 * t4;
        if (qA < qt.nrows) {
          atomicAdd(a.dqacc + rowA * D + col, sh.scale * dq[dt][0]);
          atomicAdd(a.dqacc + rowA * D + col + 1, sh.scale * dq[dt][1]);
        }
        if (qB < qt.nrows) {
          atomicAdd(a.dqacc + rowB * D + col, sh.scale * dq[dt][2]);
          atomicAdd(a.dqacc + rowB * D + col + 1, sh.scale * dq[dt][3]);
        }
      }
    }
    __syncthreads();
    if (!has_next) break;
    rr = nrr;
    ti = nti;
    sidx = nsx;
    range = nrange;
    buf ^= 1;
  }

  cp_async_wait<0>();
  // epilogue: natural-order dK_m (scaled) and dV_m
  auto* dkm = static_cast<__nv_bfloat16*>(a.dkm);
  auto* dvm = static_cast<__nv_bfloat16*>(a.dvm);
  if (kokA) {
    const int64_t base = (int64_t(kt.pos0 + kA) * sh.Hkv + kvh) * D;
#pragma unroll
    for (int dt = 0; dt < D / 8; ++dt) {
      const int col = dt * 8 + 2 * t4;
      *reinterpret_cast<uint32_t*>(dkm + base + col) = pack_bf16(sh.scale * dk[dt][0], sh.scale * dk[dt][1]);
      *reinterpret_cast<uint32_t*>(dvm + base + col) = pack_bf16(dv[dt][0], dv[dt][1]);
    }
  }
  if (kokB) {
    const int64_t base = (int64_t(kt.pos0 + kB) * sh.Hkv + kvh) * D;
#pragma unroll
    for (int dt = 0; dt < D / 8; ++dt) {
      const int col = dt * 8 + 2 * t4;
      *reinterpret_cast<uint32_t*>(dkm + base + col) = pack_bf16(sh.scale * dk[dt][2], sh.scale * dk[dt][3]);
      *reinterpret_cast<uint32_t*>(dvm + base + col) = pack_bf16(dv[dt][2], dv[dt][3]);
    }
  }
}

}  // namespace

cudaError_t ba_launch_main_bwd(const BaBwdArgs& a, cudaStream_t st) {
  const int64_t grid = int64_t(a.tb.n_bkv) * a.sh.Hkv;
  if (grid == 0) return cudaSuccess;
  if (a.sh.d == 128) {
    const int smem = int(BwdSmem<128>::bytes);
    if (cudaError_t e = set_dynamic_smem(main_bwd_mma_kernel<128>, size_t(smem)); e != cudaSuccess) return e;
    main_bwd_mma_kernel<128><<<unsigned(grid), NT, smem, st>>>(a);
  } else {
    const int smem = int(BwdSmem<64>::bytes);
    if (cudaError_t e = set_dynamic_smem(main_bwd_mma_kernel<64>, size_t(smem)); e != cudaSuccess) return e;
    main_bwd_mma_kernel<64><<<unsigned(grid), NT, smem, st>>>(a);
  }
  return cudaGetLastError();
}
