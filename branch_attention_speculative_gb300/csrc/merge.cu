// K4 — the online-softmax log-sum-exp merge (Eq. 2).
//
// "Online Draft Co-Training ...", rainbus page, core method, Eq. 2:
//   l = log(e^l_m + e^l_b),
//   O = (e^(l_m - l) O_m + e^(l_b - l) O_b) / (e^(l_m - l) + e^(l_b - l)).
// An empty part (l = -inf) merges as the identity; two empty parts give
// O = 0 and l = -inf.  The log of the sum is taken shifted by the larger of
// the two.  In the forward path the merge also unpacks: it reads the packed
// partials and writes o and lse in natural order.  HBM-bound: one group of
// d/4 threads per row, float4 loads of the fp32 partials, bf16x4 stores.
#include <math.h>

#include "device.cuh"
#include "kernels.h"

namespace {

struct MergeIdentity {
  __device__ __forceinline__ int64_t operator()(int64_t row) const { return row; }
};


template <int D, class Map>
__global__ void __launch_bounds__(256) lse_merge_kernel(int64_t rows, const float* __restrict__ om,
                                                        const float* __restrict__ lm, const float* __restrict__ ob,
                                                        const float* __restrict__ lb, __nv_bfloat16* __restrict__ o,
                                                        float* __restrict__ l, Map map) {
  constexpr int TPR = D / 4;  // threads per row
  constexpr int RPB = 256 / TPR;
  const int sub = threadIdx.x % TPR;
  for (int64_t row = int64_t(blockIdx.x) * RPB + threadIdx.x / TPR; row < rows; row += int64_t(gridDim.x) * RPB) {
    const float a = lm[row];
    const float b = ob ? lb[row] : -INFINITY;
    const float top = fmaxf(a, b);
    const int64_t out = map(row);
    float4 res = make_float4(0.f, 0.f, 0.f, 0.f);
    float lout = -INFINITY;
    if (top != -INFINITY) {
      lout = top + logf(expf(a - top) + expf(b - top));
      const float wa = expf(a - lout);
      const float wb = expf(b - lout);
      const float inv = 1.0f / (wa + wb);
      // an empty part contributes nothing, whatever its O holds
      if (wa > 0.f) {
        const float4 x = reinterpret_cast<const float4*>(om + row * D)[sub];
        res.x = wa * x.x; res.y = wa * x.y; res.z = wa * x.z; res.w = wa * x.w;
      }
      if (wb > 0.f) {
        const float4 y = reinterpret_cast<const float4*>(ob + row * D)[sub];
        res.x += wb * y.x; res.y += wb * y.y; res.z += wb * y.z; res.w += wb * y.w;
      }
      res.x *= inv; res.y *= inv; res.z *= inv; res.w *= inv;
    }
    uint2 pk;
    pk.x = pack_bf16(res.x, res.y);
    pk.y = pack_bf16(res.z, res.w);
    reinterpret_cast<uint2*>(o + out * D)[sub] = pk;
    if (sub == 0) l[out] = lout;
  }
}

template <class Map>
cudaError_t launch(int64_t rows, int d, const float* om, const float* lm, const float* ob, const float* lb, void* o,
                   float* l, Map map, cudaStream_t st) {
  if (rows == 0) return cudaSuccess;
  const int rpb = 256 / (d / 4);
  int64_t blocks = (rows + rpb - 1) / rpb;
  if (blocks > 152 * 32) blocks = 152 * 32;
  auto* ob16 = static_cast<__nv_bfloat16*>(o);
  if (d == 128)
    lse_merge_kernel<128, Map><<<unsigned(blocks), 256, 0, st>>>(rows, om, lm, ob, lb, ob16, l, map);
  else
    lse_merge_kernel<64, Map><<<unsigned(blocks), 256, 0, st>>>(rows, om, lm, ob, lb, ob16, l, map);
  return cudaGetLastError();
}

// Eq. 2 for one query-head row held by `n` lanes (n * 4 = D); w* are the
// Eq. 2 weights e^(l_* - l) / (e^(l_m - l) + e^(l_b - l)).
template <int D>
__device__ __forceinline__ void merge_row(const float* om, const float* ob, float a, float b, int sub,
                                          __nv_bfloat16* o, float* l, bool write_l) {
  const float top = fmaxf(a, b);
  float4 res = make_float4(0.f, 0.f, 0.f, 0.f);
  float lout = -INFINITY;
  if (top != -INFINITY) {
    lout = top + logf(expf(a - top) + expf(b - top));
    const float wa = expf(a - lout), wb = expf(b - lout);
    const float inv = 1.0f / (wa + wb);
    if (wa > 0.f) {
      const float4 x = reinterpret_cast<const float4*>(om)[sub];
      res.x = wa * x.x; res.y = wa * x.y; res.z = wa * x.z; res.w = wa * x.w;
    }
    if (wb > 0.f) {
      const float4 y = reinterpret_cast<const float4*>(ob)[sub];
      res.x += wb * y.x; res.y += wb * y.y; res.z += wb * y.z; res.w += wb * y.w;
    }
    res.x *= inv; res.y *= inv; res.z *= inv; res.w *= inv;
  }
  uint2 pk;
  pk.x = pack_bf16(res.x, res.y);
  pk.y = pack_bf16(res.z, res.w);
  reinterpret_cast<uint2*>(o)[sub] = pk;
  if (write_l) *l = lout;
}

// Plan path: one warp per (step j, packed row r) unit and all of its heads, so
// the packed -> natural mapping (a few integer divisions) is paid once per
// unit, not per head; reads stay contiguous (heads are innermost in both
// layouts) and every lane moves 16-byte vectors.
template <int D>
__global__ void __launch_bounds__(256) lse_merge_plan_kernel(BaFwdArgs a) {
  constexpr int LPR = D / 4;            // lanes per head row
  constexpr int HPW = 32 / LPR;         // head rows per warp pass
  const BaShape& sh = a.sh;
  const int lane = threadIdx.x & 31;
  const int sub = lane % LPR, hoff = lane / LPR;
  const int64_t units = int64_t(sh.steps) * sh.rows;
  const int64_t warp0 = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = (int64_t(gridDim.x) * blockDim.x) >> 5;
  const bool has_b = sh.family != BA_FAMILY_CAUSAL;
  auto* o = static_cast<__nv_bfloat16*>(a.o);
  for (int64_t u = warp0; u < units; u += nwarps) {
    const int64_t j = u / sh.rows;
    const int64_t r = u - j * sh.rows;
    const int64_t nu = j * sh.rows + natural_row(sh, a.tb, r);
    const int64_t prow0 = u * sh.Hq, nrow0 = nu * sh.Hq;
    for (int h = hoff; h < sh.Hq; h += HPW) {
      const int64_t pr = prow0 + h, nr = nrow0 + h;
      merge_row<D>(a.om + pr * D, has_b ? a.ob + pr * D : nullptr, a.lm[pr], has_b ? a.lb[pr] : -INFINITY, sub,
                   o + nr * D, a.lse + nr, sub == 0);
    }
  }
}

}  // namespace

cudaError_t ba_launch_merge_plan(const BaFwdArgs& a, cudaStream_t st) {
  const int64_t units = int64_t(a.sh.steps) * a.sh.rows;
  if (units == 0) return cudaSuccess;
  int64_t blocks = (units + 7) / 8;
  if (blocks > 152 * 16) blocks = 152 * 16;
  if (a.sh.d == 128)
    lse_merge_plan_kernel<128><<<unsigned(blocks), 256, 0, st>>>(a);
  else
    lse_merge_plan_kernel<64><<<unsigned(blocks), 256, 0, st>>>(a);
  return cudaGetLastError();
}

cudaError_t ba_launch_merge_rows(int64_t rows, int d, const float* om, const float* lm, const float* ob,
                                 const float* lb, void* o, float* l, cudaStream_t st) {
  return launch(rows, d, om, lm, ob, lb, o, l, MergeIdentity{}, st);
}
