// K5 — backward preprocessing.
//
// For every query-head row: Delta = <dO, O> in fp32 (the row term of the
// softmax backward, dS = P * (dP - Delta)).  -lse (in base 2), Delta and the
// row's main-key limit go into one 16-byte record per (step, head, row), in
// natural row order and stream-major, so that the records of a query tile (a
// run of consecutive natural rows) are one contiguous TMA box.  The pages only
// say that the backward replays the ring ("Online Draft Co-Training ...",
// rainbus page, method step 5); Delta is what that replay needs per row when P
// is recomputed from the merged lse.
// HBM-bound: d/8 threads per row, 16-byte loads.
#include "device.cuh"
#include "kernels.h"

namespace {

template <int D>
__global__ void __launch_bounds__(256) bwd_prep_kernel(BaBwdArgs a) {
  constexpr int TPR = D / 8;  // threads per row, 8 bf16 each
  constexpr int RPB = 256 / TPR;
  const BaShape& sh = a.sh;
  const int sub = threadIdx.x % TPR;
  const int64_t rows = int64_t(sh.steps) * sh.rows * sh.Hq;
  const auto* o = static_cast<const uint4*>(a.o);
  const auto* go = static_cast<const uint4*>(a.d_o);
  // block-uniform trip count: the shuffles below need every lane of the warp
  for (int64_t base = int64_t(blockIdx.x) * RPB; base < rows; base += int64_t(gridDim.x) * RPB) {
    const int64_t row = base + threadIdx.x / TPR;
    const bool valid = row < rows;
    const int64_t h = row % sh.Hq;
    const int64_t jr = row / sh.Hq;
    const int64_t j = jr / sh.rows;
    const int64_t r = jr - j * sh.rows;
    uint4 ov = make_uint4(0, 0, 0, 0), gv = make_uint4(0, 0, 0, 0);
    if (valid) {
      ov = o[row * TPR + sub];
      gv = go[row * TPR + sub];
    }
    float acc = 0.f;
    const uint32_t* ow = reinterpret_cast<const uint32_t*>(&ov);
    const uint32_t* gw = reinterpret_cast<const uint32_t*>(&gv);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float2 x = unpack_bf16(ow[k]), y = unpack_bf16(gw[k]);
      acc += x.x * y.x + x.y * y.y;
    }
#pragma unroll
    for (int m = TPR / 2; m > 0; m >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, m);
    if (!valid) continue;
    if (sub == 0) {  // one 16-byte record per (step, head, row), stream-major
      const int64_t srow = (j * sh.Hq + h) * sh.rows + r;
      a.rowrec[srow] = make_float4(-a.lse[row] * BA_LOG2E, acc, __int_as_float(a.tb.nat_lim[r]), 0.f);
    }
  }
}

}  // namespace

cudaError_t ba_launch_bwd_prep(const BaBwdArgs& a, cudaStream_t st) {
  const int64_t rows = int64_t(a.sh.steps) * a.sh.rows * a.sh.Hq;
  if (rows == 0) return cudaSuccess;
  const int rpb = 256 / (a.sh.d / 8);
  int64_t blocks = (rows + rpb - 1) / rpb;
  if (blocks > 152 * 32) blocks = 152 * 32;
  if (a.sh.d == 128)
    bwd_prep_kernel<128><<<unsigned(blocks), 256, 0, st>>>(a);
  else
    bwd_prep_kernel<64><<<unsigned(blocks), 256, 0, st>>>(a);
  return cudaGetLastError();
}
