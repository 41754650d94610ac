// K1 — zigzag pack / unpack.
//
// Moves whole token (or anchor) rows between the natural order and the packed
// zigzag order ("Online Draft Co-Training ...", rainbus page, CP
// prerequisites and method step 2: rank r's shard holds chunks r and 2C-1-r
// of every sequence; branch rows follow their anchor's rank).  Pure data
// movement, bound by HBM bandwidth: one warp copies one row with 16-byte
// vector loads and stores, warps stride over the rows.
#include "device.cuh"
#include "kernels.h"

namespace {

__global__ void __launch_bounds__(256) zigzag_gather_kernel(const uint4* __restrict__ src, uint4* __restrict__ dst,
                                                            const int32_t* __restrict__ perm, int64_t outer,
                                                            int64_t units, int64_t unit_vecs, int inverse) {
  const int lane = threadIdx.x & 31;
  const int64_t warp = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = (int64_t(gridDim.x) * blockDim.x) >> 5;
  const int64_t total = outer * units;
  for (int64_t w = warp; w < total; w += nwarps) {
    const int64_t o = w / units;
    const int64_t i = w - o * units;
    const int64_t p = perm[i];
    const int64_t si = inverse ? i : p;
    const int64_t di = inverse ? p : i;
    const uint4* s = src + (o * units + si) * unit_vecs;
    uint4* d = dst + (o * units + di) * unit_vecs;
    for (int64_t v = lane; v < unit_vecs; v += 32) d[v] = __ldg(s + v);
  }
}

}  // namespace

cudaError_t ba_launch_zigzag_gather(const void* src, void* dst, const int32_t* perm, int64_t outer, int64_t units,
                                    int64_t unit_bytes, int inverse, cudaStream_t st) {
  if (outer * units == 0) return cudaSuccess;
  const int64_t warps = outer * units;
  int64_t blocks = (warps + 7) / 8;
  const int64_t cap = 152 * 16;
  if (blocks > cap) blocks = cap;
  zigzag_gather_kernel<<<dim3(unsigned(blocks)), dim3(256), 0, st>>>(
      static_cast<const uint4*>(src), static_cast<uint4*>(dst), perm, outer, units, unit_bytes / 16, inverse);
  return cudaGetLastError();
}
