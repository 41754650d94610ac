// Kernel launchers (host side).  Each returns the launch's cudaError_t.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "ba_internal.h"

// All tensors are in the caller's natural layout: the kernels reach the zigzag
// chunks through the plan's tile coordinates instead of packed copies.
struct BaFwdArgs {
  BaShape sh;
  BaTables tb;
  const void *q, *km, *vm, *kb, *vb;  // inputs (bf16)
  void* o;                            // output (bf16)
  float* lse;                         // lse (fp32)
  // 8-bit forward: e4m3 copies of q, k_m and V^T ([Hkv][d][T]) in the
  // workspace and the amax of q, k_m, v_m (each scale = amax / 448)
  const void *q8, *k8, *vt8;
  const float* f8amax;
};

struct BaBwdArgs {
  BaShape sh;
  BaTables tb;
  const void *q, *km, *vm, *kb, *vb;  // inputs (bf16)
  const void *o, *d_o;                // forward output and its gradient (bf16)
  const float* lse;                   // forward lse (fp32)
  float4* rowrec;                     // per (step, head, row), stream-major: {-lse*log2e, Delta, limit, 0}
  void *dq, *dkm, *dvm, *dkb, *dvb;   // gradients (bf16)
  // single-step TTT calls: the key gradients are added into these fp32
  // accumulators (natural layouts) instead of being written to dkm .. dvb
  float *dkm_acc, *dvm_acc, *dkb_acc, *dvb_acc;
};

// K1: dst[o][i] = src[o][perm[i]] (inverse = 0) or dst[o][perm[i]] = src[o][i].
cudaError_t ba_launch_zigzag_gather(const void* src, void* dst, const int32_t* perm, int64_t outer,
                                    int64_t units, int64_t unit_bytes, int inverse, cudaStream_t st);
// Allows a kernel `bytes` of dynamic shared memory (host side, before a launch).
template <class Kernel>
inline cudaError_t set_dynamic_smem(Kernel* kernel, size_t bytes) {
  return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(bytes));
}

// K2 (+K3, K4 in its epilogue): causal main attention over each query tile's
// key segments, then per row the rank-local branch part and the Eq. 2 merge
// -> o, lse (tcgen05 / TMEM / TMA; head_dim 64 and 128).
cudaError_t ba_launch_main_fwd_tc(const BaFwdArgs& a, cudaStream_t st);
// K2 with 8-bit operands (head_dim 128): QK^T and PV on e4m3 copies.
cudaError_t ba_launch_main_fwd_fp8(const BaFwdArgs& a, cudaStream_t st);
// Quantisation for it: amax of q, k_m, v_m (into amax[3], zeroed first), then
// the e4m3 copies q8, k8 and the transposed vt8 [Hkv][d][T].
cudaError_t ba_launch_fp8_quantize(const BaFwdArgs& a, float* amax, void* q8, void* k8, void* vt8,
                                   cudaStream_t st);
// K4 alone on caller buffers (ba_lse_merge).
cudaError_t ba_launch_merge_rows(int64_t rows, int d, const float* om, const float* lm, const float* ob,
                                 const float* lb, void* o, float* l, cudaStream_t st);
// K5: Delta = rowsum(dO * O) and the row records.
cudaError_t ba_launch_bwd_prep(const BaBwdArgs& a, cudaStream_t st);
// K6: main-attention backward on tcgen05 (head_dim 64 and 128): the
// key-stationary kernel writes dK_m, dV_m (natural order); the
// query-stationary kernel writes the main part of dq_b (bf16).
cudaError_t ba_launch_main_bwd_kv_tc(const BaBwdArgs& a, cudaStream_t st);
cudaError_t ba_launch_main_bwd_q_tc(const BaBwdArgs& a, cudaStream_t st);
// K7 (+K8): branch backward: dK_b, dV_b (natural); adds each row's branch
// part to dq_b.
cudaError_t ba_launch_branch_bwd(const BaBwdArgs& a, cudaStream_t st);

// Self-test: a bounded wait on a barrier nothing completes (records BA_DEV_TIMEOUT).
cudaError_t ba_launch_selftest_wait_timeout(unsigned int* status, long long cycles, cudaStream_t st);
