// Quantisation for the 8-bit main forward: per-tensor amax of q, k_m and v_m,
// then e4m3 copies with scale amax / 448 (the largest finite e4m3 value), so
// each tensor's largest element maps to the top of the e4m3 range.  V is also
// transposed to [Hkv][d][T], which makes it a K-major operand of the PV GEMM.
// "Online Draft Co-Training ...", rainbus page, limitations and future work,
// item (4): carrying the decomposition to fp8 training; the page names no
// scaling scheme, and per-tensor amax scaling is the plainest one.
// HBM-bound: 16-byte loads of 8 bf16, 8- and 16-byte stores of e4m3.
#include <cuda_fp8.h>

#include "device.cuh"
#include "kernels.h"

namespace {

__device__ __forceinline__ float inv_scale(float amax) { return amax > 0.f ? 448.0f / amax : 1.0f; }

__device__ __forceinline__ uint32_t e4m3x4(float a, float b, float c, float d) {
  const uint32_t lo = __nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
  const uint32_t hi = __nv_cvt_float2_to_fp8x2(make_float2(c, d), __NV_SATFINITE, __NV_E4M3);
  return lo | (hi << 16);
}

// blockIdx.y picks the tensor: 0 q, 1 k_m, 2 v_m; n8[y] = elements / 8.
__global__ void __launch_bounds__(256) fp8_amax_kernel(const uint4* q, const uint4* k, const uint4* v, int64_t nq8,
                                                       int64_t nk8, float* amax) {
  const uint4* src = blockIdx.y == 0 ? q : (blockIdx.y == 1 ? k : v);
  const int64_t n = blockIdx.y == 0 ? nq8 : nk8;
  float m = 0.f;
  for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += int64_t(gridDim.x) * blockDim.x) {
    const uint4 x = src[i];
    const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 f = unpack_bf16(w[e]);
      m = fmaxf(m, fmaxf(fabsf(f.x), fabsf(f.y)));
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  __shared__ float part[8];
  if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int w = 1; w < 8; ++w) m = fmaxf(m, part[w]);
    // non-negative floats order like their bit patterns
    atomicMax(reinterpret_cast<unsigned int*>(amax + blockIdx.y), __float_as_uint(m));
  }
}

// blockIdx.y: 0 q -> q8, 1 k_m -> k8 (same layouts, 8 values per thread step).
__global__ void __launch_bounds__(256) fp8_quant_kernel(const uint4* q, const uint4* k, int64_t nq8, int64_t nk8,
                                                        const float* amax, uint2* q8, uint2* k8) {
  const uint4* src = blockIdx.y == 0 ? q : k;
  uint2* dst = blockIdx.y == 0 ? q8 : k8;
  const int64_t n = blockIdx.y == 0 ? nq8 : nk8;
  const float inv = inv_scale(amax[blockIdx.y]);
  for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += int64_t(gridDim.x) * blockDim.x) {
    const uint4 x = src[i];
    const float2 a = unpack_bf16(x.x), b = unpack_bf16(x.y), c = unpack_bf16(x.z), d = unpack_bf16(x.w);
    dst[i] = make_uint2(e4m3x4(a.x * inv, a.y * inv, b.x * inv, b.y * inv),
                        e4m3x4(c.x * inv, c.y * inv, d.x * inv, d.y * inv));
  }
}

// V [T][Hkv][D] bf16 -> vt8 [Hkv][D][T] e4m3.  One block: 128 keys of one kv
// head through shared memory (row pitch D + 2 elements, so a column read is
// free of bank conflicts); each thread then writes 16 keys of one d row.
template <int D>
__global__ void __launch_bounds__(256) fp8_vt_kernel(const __nv_bfloat16* v, int64_t T, int Hkv, const float* amax,
                                                     unsigned char* vt8) {
  constexpr int KB = 128, PITCH = D + 2;
  __shared__ __nv_bfloat16 tile[KB * PITCH];
  const int64_t key0 = int64_t(blockIdx.x) * KB;
  const int kvh = blockIdx.y;
  const float inv = inv_scale(amax[2]);
  // load: 128 rows of D values, 8 per 16-byte load
  for (int e = threadIdx.x; e < KB * (D / 8); e += blockDim.x) {
    const int r = e / (D / 8), c = (e % (D / 8)) * 8;
    uint4 x = make_uint4(0, 0, 0, 0);
    if (key0 + r < T) x = *reinterpret_cast<const uint4*>(v + ((key0 + r) * Hkv + kvh) * D + c);
    uint32_t* dst = reinterpret_cast<uint32_t*>(tile + r * PITCH + c);
    dst[0] = x.x;
    dst[1] = x.y;
    dst[2] = x.z;
    dst[3] = x.w;
  }
  __syncthreads();
  // store: D rows x 8 chunks of 16 keys
  for (int e = threadIdx.x; e < D * (KB / 16); e += blockDim.x) {
    const int dr = e % D, kc = e / D;
    if (key0 + kc * 16 >= T) continue;
    float f[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) f[i] = __bfloat162float(tile[(kc * 16 + i) * PITCH + dr]) * inv;
    const uint4 out = make_uint4(e4m3x4(f[0], f[1], f[2], f[3]), e4m3x4(f[4], f[5], f[6], f[7]),
                                 e4m3x4(f[8], f[9], f[10], f[11]), e4m3x4(f[12], f[13], f[14], f[15]));
    *reinterpret_cast<uint4*>(vt8 + (int64_t(kvh) * D + dr) * T + key0 + kc * 16) = out;
  }
}

}  // namespace

cudaError_t ba_launch_fp8_quantize(const BaFwdArgs& a, float* amax, void* q8, void* k8, void* vt8, cudaStream_t st) {
  const BaShape& sh = a.sh;
  if (sh.d != 128 || sh.T % 16 != 0) return cudaErrorInvalidConfiguration;
  const int64_t nq8 = int64_t(sh.steps) * sh.rows * sh.Hq * sh.d / 8;
  const int64_t nk8 = sh.T * sh.Hkv * sh.d / 8;
  cudaError_t e = cudaMemsetAsync(amax, 0, 3 * sizeof(float), st);
  if (e != cudaSuccess) return e;
  const int64_t most = nq8 > nk8 ? nq8 : nk8;
  int64_t blocks = (most + 255) / 256;
  if (blocks > 152 * 8) blocks = 152 * 8;
  if (blocks < 1) blocks = 1;
  fp8_amax_kernel<<<dim3(unsigned(blocks), 3), 256, 0, st>>>(static_cast<const uint4*>(a.q),
                                                             static_cast<const uint4*>(a.km),
                                                             static_cast<const uint4*>(a.vm), nq8, nk8, amax);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  fp8_quant_kernel<<<dim3(unsigned(blocks), 2), 256, 0, st>>>(static_cast<const uint4*>(a.q),
                                                              static_cast<const uint4*>(a.km), nq8, nk8, amax,
                                                              static_cast<uint2*>(q8), static_cast<uint2*>(k8));
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  const int64_t kb = (sh.T + 127) / 128;
  fp8_vt_kernel<128><<<dim3(unsigned(kb), unsigned(sh.Hkv)), 256, 0, st>>>(
      static_cast<const __nv_bfloat16*>(a.vm), sh.T, sh.Hkv, amax, static_cast<unsigned char*>(vt8));
  return cudaGetLastError();
}
