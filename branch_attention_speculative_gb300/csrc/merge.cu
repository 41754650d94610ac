// K4 — the online-softmax log-sum-exp merge (Eq. 2).
//
// "Online Draft Co-Training ...", rainbus page, core method, Eq. 2:
//   l = log(e^l_m + e^l_b),
//   O = (e^(l_m - l) O_m + e^(l_b - l) O_b) / (e^(l_m - l) + e^(l_b - l)).
// An empty part (l = -inf) merges as the identity; two empty parts give
// O = 0 and l = -inf.  The log of the sum is taken shifted by the larger of
// the two.  Both partials and the outputs are in natural row order, so the
// merge is a straight row-for-row pass.  HBM-bound: one group of d/4 threads
// per row, float4 loads of the fp32 partials, bf16x4 stores.
#include <math.h>

#include "device.cuh"
#include "kernels.h"

namespace {

template <int D>
__global__ void __launch_bounds__(256) lse_merge_kernel(int64_t rows, const float* __restrict__ om,
                                                        const float* __restrict__ lm, const float* __restrict__ ob,
                                                        const float* __restrict__ lb, __nv_bfloat16* __restrict__ o,
                                                        float* __restrict__ l) {
  constexpr int TPR = D / 4;  // threads per row
  constexpr int RPB = 256 / TPR;
  const int sub = threadIdx.x % TPR;
  for (int64_t row = int64_t(blockIdx.x) * RPB + threadIdx.x / TPR; row < rows; row += int64_t(gridDim.x) * RPB) {
    const float a = lm[row];
    const float b = ob ? lb[row] : -INFINITY;
    const float top = fmaxf(a, b);
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
    reinterpret_cast<uint2*>(o + row * D)[sub] = pk;
    if (sub == 0) l[row] = lout;
  }
}

}  // namespace

cudaError_t ba_launch_merge_rows(int64_t rows, int d, const float* om, const float* lm, const float* ob,
                                 const float* lb, void* o, float* l, cudaStream_t st) {
  if (rows == 0) return cudaSuccess;
  const int rpb = 256 / (d / 4);
  int64_t blocks = (rows + rpb - 1) / rpb;
  if (blocks > 152 * 32) blocks = 152 * 32;
  auto* o16 = static_cast<__nv_bfloat16*>(o);
  if (d == 128)
    lse_merge_kernel<128><<<unsigned(blocks), 256, 0, st>>>(rows, om, lm, ob, lb, o16, l);
  else
    lse_merge_kernel<64><<<unsigned(blocks), 256, 0, st>>>(rows, om, lm, ob, lb, o16, l);
  return cudaGetLastError();
}
