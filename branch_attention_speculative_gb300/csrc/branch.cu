// K7 — rank-local branch attention, backward: the branch keys' gradients.
//
// "Online Draft Co-Training ...", ai.info summary, Key Contributions 1 and
// "Methodology in Plain English": the branch part is small and lives on the
// rank that owns the anchor, so it needs no communication; rainbus page, core
// method: the backward accumulates gradients locally with no
// branch-dependent traffic.  Key sets (paperlens walkthrough, Wall 1):
//   TTT   — step-j query at anchor p sees branch keys (p, i), i <= j;
//   BLOCK — each of the B queries of an anchor sees all B keys of the block.
//
// One CTA handles one anchor unit (a token position for TTT, an anchor for
// BLOCK; natural order, since the branch part needs no zigzag) and one kv
// head: the unit's few branch keys are staged in shared memory as fp32, each
// warp takes query rows, a lane owns d/32 columns, dot products are
// warp-shuffle reductions, and dK_b / dV_b of the unit are summed over all of
// its rows (every step and q head of the group) before one store.  The work is
// tiny next to the main part and bound by HBM traffic of q and dO.
//
// It also finishes dQ: the main part arrives as bf16 in dq_b (written by the
// dQ kernel), the branch part is added in fp32 and the row is written back.
// The forward's branch part and Eq. 2 merge run in the main forward's
// epilogue instead, where each row's thread already holds its main part.
#include <math.h>

#include "device.cuh"
#include "kernels.h"

namespace {

__device__ __forceinline__ int rows_per_unit(const BaShape& sh) {
  return sh.family == BA_FAMILY_TTT ? sh.steps : (sh.family == BA_FAMILY_BLOCK ? sh.B : 1);
}

// branch-key slot of key i of unit u: TTT keys are [step, position],
// BLOCK keys are [anchor, offset]
__device__ __forceinline__ int64_t branch_slot(const BaShape& sh, int64_t u, int i) {
  return sh.family == BA_FAMILY_TTT ? int64_t(i) * sh.T + u : u * sh.B + i;
}

// (step j, row r) of query qi of unit u
__device__ __forceinline__ void unit_query(const BaShape& sh, int64_t u, int qi, int64_t& j, int64_t& r) {
  if (sh.family == BA_FAMILY_TTT) { j = qi; r = u; }
  else if (sh.family == BA_FAMILY_BLOCK) { j = 0; r = u * sh.B + qi; }
  else { j = 0; r = u; }
}

// branch keys of query qi of a unit: the step-j TTT query sees slots 0..j
// (j = step0 + qi, its global step), a block query all B keys of its block
__device__ __forceinline__ int keys_of_query(const BaShape& sh, int qi) {
  return sh.family == BA_FAMILY_TTT ? sh.step0 + qi + 1 : (sh.family == BA_FAMILY_BLOCK ? sh.B : 0);
}

template <int D>
__device__ __forceinline__ void load_row(const __nv_bfloat16* p, int lane, float* x) {
  constexpr int E = D / 32;
  if constexpr (E == 4) {
    const uint2 v = reinterpret_cast<const uint2*>(p)[lane];
    const float2 a = unpack_bf16(v.x), b = unpack_bf16(v.y);
    x[0] = a.x; x[1] = a.y; x[2] = b.x; x[3] = b.y;
  } else {
    const float2 a = unpack_bf16(reinterpret_cast<const uint32_t*>(p)[lane]);
    x[0] = a.x; x[1] = a.y;
  }
}

template <int D>
__device__ __forceinline__ void store_row_bf16(__nv_bfloat16* p, int lane, const float* x) {
  constexpr int E = D / 32;
  if constexpr (E == 4) {
    uint2 v;
    v.x = pack_bf16(x[0], x[1]);
    v.y = pack_bf16(x[2], x[3]);
    reinterpret_cast<uint2*>(p)[lane] = v;
  } else {
    reinterpret_cast<uint32_t*>(p)[lane] = pack_bf16(x[0], x[1]);
  }
}

constexpr int NKR = 8;  // branch keys per unit whose gradients a warp keeps in registers

// One unit's branch keys of one kv head into shared memory as fp32: row i of
// ks / vs is key slot branch_slot(u, i).  16-byte loads of 8 values.
template <int D>
__device__ void stage_keys(const BaShape& sh, const __nv_bfloat16* kb, const __nv_bfloat16* vb, int64_t u, int kvh,
                           float* ks, float* vs) {
  constexpr int CH = D / 8;  // 16-byte chunks per key row
  const int n = sh.nbk * CH;
  for (int e = threadIdx.x; e < 2 * n; e += blockDim.x) {
    const int m = e >= n ? 1 : 0;  // 0: K, 1: V
    const int ee = e - m * n;
    const int i = ee / CH, c = ee % CH;
    const int64_t off = (branch_slot(sh, u, i) * sh.Hkv + kvh) * D + c * 8;
    const uint4 v = *reinterpret_cast<const uint4*>((m ? vb : kb) + off);
    const float2 a = unpack_bf16(v.x), b = unpack_bf16(v.y), c2 = unpack_bf16(v.z), d2 = unpack_bf16(v.w);
    float4* dst = reinterpret_cast<float4*>((m ? vs : ks) + i * D + c * 8);
    dst[0] = make_float4(a.x, a.y, b.x, b.y);
    dst[1] = make_float4(c2.x, c2.y, d2.x, d2.y);
  }
}

// dK_b / dV_b of one unit and kv head from shared memory (fp32) to their bf16
// key slots (16-byte stores of 8 values), or added into the fp32 accumulators
// of a single-step call (each slot of a unit and kv head belongs to one CTA,
// so the read-add-write needs no atomics).
template <int D>
__device__ void store_key_grads(const BaShape& sh, const BaBwdArgs& a, int64_t u, int kvh, const float* dks,
                                const float* dvs) {
  constexpr int CH = D / 8;
  const int n = sh.nbk * CH;
  auto* dkb = static_cast<__nv_bfloat16*>(a.dkb);
  auto* dvb = static_cast<__nv_bfloat16*>(a.dvb);
  for (int e = threadIdx.x; e < 2 * n; e += blockDim.x) {
    const int m = e >= n ? 1 : 0;
    const int ee = e - m * n;
    const int i = ee / CH, c = ee % CH;
    const int64_t off = (branch_slot(sh, u, i) * sh.Hkv + kvh) * D + c * 8;
    const float4* src = reinterpret_cast<const float4*>((m ? dvs : dks) + i * D + c * 8);
    const float4 x = src[0], y = src[1];
    if (a.dkb_acc) {
      float4* acc = reinterpret_cast<float4*>((m ? a.dvb_acc : a.dkb_acc) + off);
      const float4 p = acc[0], q = acc[1];
      acc[0] = make_float4(p.x + x.x, p.y + x.y, p.z + x.z, p.w + x.w);
      acc[1] = make_float4(q.x + y.x, q.y + y.y, q.z + y.z, q.w + y.w);
    } else {
      *reinterpret_cast<uint4*>((m ? dvb : dkb) + off) =
          make_uint4(pack_bf16(x.x, x.y), pack_bf16(x.z, x.w), pack_bf16(y.x, y.y), pack_bf16(y.z, y.w));
    }
  }
}

template <int D>
__global__ void __launch_bounds__(128) branch_bwd_kernel(BaBwdArgs a) {
  extern __shared__ float smem[];
  constexpr int E = D / 32;
  const BaShape& sh = a.sh;
  float* ks = smem;
  float* vs = ks + sh.nbk * D;
  float* dks = vs + sh.nbk * D;
  float* dvs = dks + sh.nbk * D;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  const auto* qg = static_cast<const __nv_bfloat16*>(a.q);
  const auto* dog = static_cast<const __nv_bfloat16*>(a.d_o);
  const auto* kb = static_cast<const __nv_bfloat16*>(a.kb);
  const auto* vb = static_cast<const __nv_bfloat16*>(a.vb);
  auto* dq = static_cast<__nv_bfloat16*>(a.dq);
  const int64_t total = sh.units * sh.Hkv;
  const int nq = rows_per_unit(sh) * sh.G;
  for (int64_t w = blockIdx.x; w < total; w += gridDim.x) {
    const int64_t u = w / sh.Hkv;
    const int kvh = int(w % sh.Hkv);
    __syncthreads();
    if (sh.nbk > 0) {
      stage_keys<D>(sh, kb, vb, u, kvh, ks, vs);
      for (int e = threadIdx.x; e < sh.nbk * D; e += blockDim.x) { dks[e] = 0.f; dvs[e] = 0.f; }
    }
    __syncthreads();
    // Up to NKR keys (TTT up to depth 8): each warp keeps its rows' dK_b /
    // dV_b contributions in registers and adds them to shared memory once per
    // unit.  More keys (block branches): per-row shared-memory atomics.
    const bool in_regs = sh.nbk <= NKR;
    float dka[NKR][E], dva[NKR][E];
#pragma unroll
    for (int i = 0; i < NKR; ++i)
#pragma unroll
      for (int e = 0; e < E; ++e) dka[i][e] = dva[i][e] = 0.f;
    for (int idx = warp; idx < nq; idx += nwarps) {
      const int qi = idx / sh.G, g = idx % sh.G;
      int64_t j, r;
      unit_query(sh, u, qi, j, r);
      const int64_t qrow = (j * sh.rows + r) * sh.Hq + kvh * sh.G + g;
      float q[E], go[E], gq[E];
      load_row<D>(qg + qrow * D, lane, q);
      load_row<D>(dog + qrow * D, lane, go);
      load_row<D>(dq + qrow * D, lane, gq);
      const int64_t srow = (j * sh.Hq + kvh * sh.G + g) * sh.rows + r;  // stream-major
      const float4 rec = a.rowrec[srow];
      const float l2 = -rec.x;  // lse * log2e
      const float delta = rec.y;
      const int nk = keys_of_query(sh, qi);
      if (in_regs) {
#pragma unroll
        for (int i = 0; i < NKR; ++i) {
          if (i < nk) {
            float dot = 0.f, dpv = 0.f;
#pragma unroll
            for (int e = 0; e < E; ++e) {
              dot += q[e] * ks[i * D + lane * E + e];
              dpv += go[e] * vs[i * D + lane * E + e];
            }
            const float s2 = warp_sum(dot) * sh.scale_log2;
            const float dp = warp_sum(dpv);
            const float p = exp2f(s2 - l2);
            const float ds = p * (dp - delta);
#pragma unroll
            for (int e = 0; e < E; ++e) {
              gq[e] += sh.scale * ds * ks[i * D + lane * E + e];
              dka[i][e] += sh.scale * ds * q[e];
              dva[i][e] += p * go[e];
            }
          }
        }
      } else {
        for (int i = 0; i < nk; ++i) {
          float dot = 0.f, dpv = 0.f;
#pragma unroll
          for (int e = 0; e < E; ++e) {
            dot += q[e] * ks[i * D + lane * E + e];
            dpv += go[e] * vs[i * D + lane * E + e];
          }
          const float s2 = warp_sum(dot) * sh.scale_log2;
          const float dp = warp_sum(dpv);
          const float p = exp2f(s2 - l2);
          const float ds = p * (dp - delta);
#pragma unroll
          for (int e = 0; e < E; ++e) {
            gq[e] += sh.scale * ds * ks[i * D + lane * E + e];
            atomicAdd(&dks[i * D + lane * E + e], sh.scale * ds * q[e]);
            atomicAdd(&dvs[i * D + lane * E + e], p * go[e]);
          }
        }
      }
      store_row_bf16<D>(dq + qrow * D, lane, gq);
    }
    if (in_regs) {
#pragma unroll
      for (int i = 0; i < NKR; ++i) {
        if (i < sh.nbk) {
#pragma unroll
          for (int e = 0; e < E; ++e) {
            atomicAdd(&dks[i * D + lane * E + e], dka[i][e]);
            atomicAdd(&dvs[i * D + lane * E + e], dva[i][e]);
          }
        }
      }
    }
    __syncthreads();
    store_key_grads<D>(sh, a, u, kvh, dks, dvs);
  }
}

int64_t grid_for(int64_t total) {
  const int64_t cap = 152 * 16;
  return total < cap ? total : cap;
}

}  // namespace

cudaError_t ba_launch_branch_bwd(const BaBwdArgs& a, cudaStream_t st) {
  const int64_t total = a.sh.units * a.sh.Hkv;
  if (total == 0 || a.sh.nbk == 0) return cudaSuccess;
  const size_t smem = size_t(4) * a.sh.nbk * a.sh.d * sizeof(float);
  if (a.sh.d == 128) {
    if (cudaError_t e = set_dynamic_smem(branch_bwd_kernel<128>, smem); e != cudaSuccess) return e;
    branch_bwd_kernel<128><<<unsigned(grid_for(total)), 128, smem, st>>>(a);
  } else {
    if (cudaError_t e = set_dynamic_smem(branch_bwd_kernel<64>, smem); e != cudaSuccess) return e;
    branch_bwd_kernel<64><<<unsigned(grid_for(total)), 128, smem, st>>>(a);
  }
  return cudaGetLastError();
}
