// C ABI of libba.so: argument checks, workspace carving, table upload and the
// launch sequence of the forward and backward passes.  See include/ba.h.
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>
#include <new>
#include <type_traits>

#include "kernels.h"
#include "plan.h"

namespace {

thread_local char g_last_cuda_error[256] = "";

int cuda_fail(cudaError_t e) {
  std::strncpy(g_last_cuda_error, cudaGetErrorString(e), sizeof(g_last_cuda_error) - 1);
  return BA_ERR_CUDA;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

bool ok_tensor(const void* p) { return p != nullptr && aligned(p, 16); }

unsigned char* ws_at(void* ws, size_t off) { return static_cast<unsigned char*>(ws) + off; }

int check_ws(const ba_plan* p, void* ws, size_t bytes) {
  if (!ws || !aligned(ws, 256) || bytes < p->ws.total) return BA_ERR_WORKSPACE;
  return BA_OK;
}

BaTables device_tables(const ba_plan* p, void* ws) {
  const BaWorkspaceLayout& w = p->ws;
  unsigned char* t = ws_at(ws, w.tables);
  BaTables tb{};
  tb.row_lim = reinterpret_cast<const int32_t*>(t + w.t_row_lim);
  tb.nat_lim = reinterpret_cast<const int32_t*>(t + w.t_nat_lim);
  tb.tok_perm = reinterpret_cast<const int32_t*>(t + w.t_tok_perm);
  tb.anc_perm = reinterpret_cast<const int32_t*>(t + w.t_anc_perm);
  tb.fq = reinterpret_cast<const BaQTile*>(t + w.t_fq);
  tb.fseg = reinterpret_cast<const BaKvSeg*>(t + w.t_fseg);
  tb.forder = reinterpret_cast<const int32_t*>(t + w.t_forder);
  tb.bq = reinterpret_cast<const BaQTile*>(t + w.t_bq);
  tb.bkv = reinterpret_cast<const BaKvTile*>(t + w.t_bkv);
  tb.bqr = reinterpret_cast<const BaQRange*>(t + w.t_bqr);
  tb.border = reinterpret_cast<const int32_t*>(t + w.t_border);
  tb.n_fq = int32_t(p->fq.size());
  tb.n_fseg = int32_t(p->fseg.size());
  tb.n_bq = int32_t(p->bq.size());
  tb.n_bkv = int32_t(p->bkv.size());
  tb.n_bqr = int32_t(p->bqr.size());
  tb.status = reinterpret_cast<unsigned int*>(ws_at(ws, w.status));
  return tb;
}

// Resets the status word and uploads the plan's tables into the workspace.
cudaError_t prepare(const ba_plan* p, void* ws, cudaStream_t st) {
  cudaError_t e = cudaMemsetAsync(ws_at(ws, p->ws.status), 0, 256, st);
  if (e != cudaSuccess) return e;
  return cudaMemcpyAsync(ws_at(ws, p->ws.tables), p->image.data(), p->ws.table_bytes, cudaMemcpyHostToDevice, st);
}

// Role geometry for the zigzag gather: outer count, units, unit bytes, permutation.
struct Role {
  int64_t outer, units, unit_bytes;
  const int32_t* perm;
};

Role role_of(const ba_plan* p, const BaTables& tb, int role) {
  const BaShape& sh = p->shape;
  const bool block = sh.family == BA_FAMILY_BLOCK;
  const int64_t d2 = int64_t(sh.d) * 2;
  switch (role) {
    case 0:
      return block ? Role{1, p->NA, int64_t(sh.B) * sh.Hq * d2, tb.anc_perm}
                   : Role{sh.steps, sh.T, int64_t(sh.Hq) * d2, tb.tok_perm};
    case 1:
      return Role{1, sh.T, int64_t(sh.Hkv) * d2, tb.tok_perm};
    default:
      if (sh.family == BA_FAMILY_CAUSAL) return Role{0, 0, 0, tb.tok_perm};
      return block ? Role{1, p->NA, int64_t(sh.B) * sh.Hkv * d2, tb.anc_perm}
                   : Role{sh.steps, sh.T, int64_t(sh.Hkv) * d2, tb.tok_perm};
  }
}

cudaError_t pack(const ba_plan* p, const BaTables& tb, int role, const void* src, void* dst, int inverse,
                 cudaStream_t st) {
  const Role r = role_of(p, tb, role);
  return ba_launch_zigzag_gather(src, dst, r.perm, r.outer, r.units, r.unit_bytes, inverse, st);
}

#define BA_TRY(x)                              \
  do {                                         \
    cudaError_t e_ = (x);                      \
    if (e_ != cudaSuccess) return cuda_fail(e_); \
  } while (0)

enum KernelId {
  K_PACK = 0, K_MAIN_FWD, K_BWD_PREP, K_MAIN_BWD, K_MAIN_BWD_DQ, K_BRANCH_BWD, K_FP8_QUANT, K_MAIN_FWD_FP8, K_COUNT
};
const char* const kKernelNames[K_COUNT] = {"zigzag_pack", "main_fwd",   "bwd_prep",     "main_bwd_kv",
                                           "main_bwd_dq", "branch_bwd", "fp8_quantize", "main_fwd_fp8"};

// Records an event pair around one launch when profiling is on.
template <class F>
cudaError_t timed(ba_plan* p, int kid, cudaStream_t st, F&& launch) {
  if (!p->prof_on) return launch();
  const size_t i = p->prof_used;
  while (p->prof_events.size() < 2 * (i + 1)) {
    cudaEvent_t e;
    cudaError_t err = cudaEventCreate(&e);
    if (err != cudaSuccess) return err;
    p->prof_events.push_back(e);
  }
  auto* a = static_cast<cudaEvent_t>(p->prof_events[2 * i]);
  auto* b = static_cast<cudaEvent_t>(p->prof_events[2 * i + 1]);
  cudaError_t err = cudaEventRecord(a, st);
  if (err != cudaSuccess) return err;
  err = launch();
  if (err != cudaSuccess) return err;
  err = cudaEventRecord(b, st);
  if (err != cudaSuccess) return err;
  p->prof_kernel.push_back(kid);
  p->prof_used = i + 1;
  return cudaSuccess;
}

// Output pointers of a backward call: bf16 gradients, or (single-step calls)
// fp32 accumulators for the key gradients.
struct BwdOut {
  void *dq, *dkm, *dvm, *dkb, *dvb;
  float *dkm_acc, *dvm_acc, *dkb_acc, *dvb_acc;
};

// The shape one TTT step runs with: one query step, global slot `step`, whose
// queries read branch key slots 0..step.
int step_shape(const ba_plan* p, int32_t step, BaShape* sh) {
  if (!p || p->shape.family != BA_FAMILY_TTT || step < 0 || step >= p->shape.steps) return BA_ERR_INVALID_ARG;
  *sh = p->shape;
  sh->steps = 1;
  sh->step0 = step;
  sh->nbk = step + 1;
  return BA_OK;
}

int run_forward(ba_plan* p, const BaShape& sh, const void* q_b, const void* k_m, const void* v_m, const void* k_b,
                const void* v_b, void* o, float* lse, void* workspace, size_t workspace_bytes, void* stream,
                bool fp8 = false) {
  const bool has_b = sh.family != BA_FAMILY_CAUSAL;
  if (!ok_tensor(q_b) || !ok_tensor(k_m) || !ok_tensor(v_m) || !ok_tensor(o) || !ok_tensor(lse))
    return BA_ERR_INVALID_ARG;
  if (has_b && (!ok_tensor(k_b) || !ok_tensor(v_b))) return BA_ERR_INVALID_ARG;
  if (fp8 && !p->fp8_ok) return BA_ERR_UNSUPPORTED;
  if (int rc = check_ws(p, workspace, workspace_bytes)) return rc;
  if (fp8 && workspace_bytes < p->ws.total_fp8) return BA_ERR_WORKSPACE;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const BaWorkspaceLayout& w = p->ws;
  BA_TRY(prepare(p, workspace, st));
  BaFwdArgs a{};
  a.sh = sh;
  a.tb = device_tables(p, workspace);
  a.q = q_b;
  a.km = k_m;
  a.vm = v_m;
  a.kb = k_b;
  a.vb = v_b;
  a.o = o;
  a.lse = lse;
  if (fp8) {
    float* amax = reinterpret_cast<float*>(ws_at(workspace, w.f8_amax));
    a.q8 = ws_at(workspace, w.f8_q);
    a.k8 = ws_at(workspace, w.f8_k);
    a.vt8 = ws_at(workspace, w.f8_vt);
    a.f8amax = amax;
    BA_TRY(timed(p, K_FP8_QUANT, st, [&] {
      return ba_launch_fp8_quantize(a, amax, const_cast<void*>(a.q8), const_cast<void*>(a.k8),
                                    const_cast<void*>(a.vt8), st);
    }));
    BA_TRY(timed(p, K_MAIN_FWD_FP8, st, [&] { return ba_launch_main_fwd_fp8(a, st); }));
  } else {
    BA_TRY(timed(p, K_MAIN_FWD, st, [&] { return ba_launch_main_fwd_tc(a, st); }));
  }
  // the main kernel's epilogue adds each row's branch part by Eq. 2 and
  // writes o and lse: nothing else runs
  return BA_OK;
}

int run_backward(ba_plan* p, const BaShape& sh, const void* q_b, const void* k_m, const void* v_m, const void* k_b,
                 const void* v_b, const void* o, const float* lse, const void* d_o, const BwdOut& out,
                 void* workspace, size_t workspace_bytes, void* stream) {
  const bool has_b = sh.family != BA_FAMILY_CAUSAL;
  if (!ok_tensor(q_b) || !ok_tensor(k_m) || !ok_tensor(v_m) || !ok_tensor(o) || !ok_tensor(lse) ||
      !ok_tensor(d_o) || !ok_tensor(out.dq) || !ok_tensor(out.dkm) || !ok_tensor(out.dvm))
    return BA_ERR_INVALID_ARG;
  if (has_b && (!ok_tensor(k_b) || !ok_tensor(v_b) || !ok_tensor(out.dkb) || !ok_tensor(out.dvb)))
    return BA_ERR_INVALID_ARG;
  if (int rc = check_ws(p, workspace, workspace_bytes)) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const BaWorkspaceLayout& w = p->ws;
  BA_TRY(prepare(p, workspace, st));
  BaBwdArgs a{};
  a.sh = sh;
  a.tb = device_tables(p, workspace);
  a.q = q_b;
  a.km = k_m;
  a.vm = v_m;
  a.kb = k_b;
  a.vb = v_b;
  a.o = o;
  a.d_o = d_o;
  a.lse = lse;
  a.rowrec = reinterpret_cast<float4*>(ws_at(workspace, w.rowrec));
  a.dq = out.dq;
  a.dkm = out.dkm;
  a.dvm = out.dvm;
  a.dkb = out.dkb;
  a.dvb = out.dvb;
  a.dkm_acc = out.dkm_acc;
  a.dvm_acc = out.dvm_acc;
  a.dkb_acc = out.dkb_acc;
  a.dvb_acc = out.dvb_acc;
  BA_TRY(timed(p, K_BWD_PREP, st, [&] { return ba_launch_bwd_prep(a, st); }));
  BA_TRY(timed(p, K_MAIN_BWD, st, [&] { return ba_launch_main_bwd_kv_tc(a, st); }));
  BA_TRY(timed(p, K_MAIN_BWD_DQ, st, [&] { return ba_launch_main_bwd_q_tc(a, st); }));
  BA_TRY(timed(p, K_BRANCH_BWD, st, [&] { return ba_launch_branch_bwd(a, st); }));
  return BA_OK;
}

}  // namespace

ba_plan::~ba_plan() {
  for (void* e : prof_events) cudaEventDestroy(static_cast<cudaEvent_t>(e));
}

extern "C" {

int ba_plan_create(const ba_plan_desc* desc, ba_plan_t* out) {
  if (!out) return BA_ERR_INVALID_ARG;
  *out = nullptr;
  ba_plan* p = new (std::nothrow) ba_plan();
  if (!p) return BA_ERR_HOST_ALLOC;
  int rc;
  try {
    rc = ba_build_plan(desc, p);
  } catch (const std::bad_alloc&) {
    rc = BA_ERR_HOST_ALLOC;
  } catch (...) {
    rc = BA_ERR_INVALID_ARG;
  }
  if (rc != BA_OK) {
    delete p;
    return rc;
  }
  *out = p;
  return BA_OK;
}

void ba_plan_destroy(ba_plan_t plan) { delete plan; }

int ba_plan_validate(ba_plan_t p) {
  if (!p) return BA_ERR_INVALID_ARG;
  try {
    return ba_validate_plan(p);
  } catch (...) {
    return BA_ERR_HOST_ALLOC;
  }
}

int ba_plan_get_info(ba_plan_t p, ba_plan_info* info) {
  if (!p || !info) return BA_ERR_INVALID_ARG;
  const BaShape& sh = p->shape;
  info->main_tokens = sh.T;
  info->branch_queries = int64_t(sh.steps) * sh.rows;
  info->query_rows = info->branch_queries * sh.Hq;
  info->main_pairs = p->main_pairs;
  info->branch_pairs = p->branch_pairs;
  info->fwd_flops = 4.0 * sh.d * double(p->main_pairs + p->branch_pairs);
  info->bwd_flops = 2.5 * info->fwd_flops;
  info->fwd_tiles = int64_t(p->fq.size());
  info->fwd_tile_blocks = p->fwd_blocks;
  info->bwd_kv_tiles = int64_t(p->bkv.size());
  int64_t mx = 0;
  for (int64_t v : p->comm) mx = v > mx ? v : mx;
  info->comm_bytes_fwd_per_rank = mx;
  info->workspace_bytes = int64_t(p->ws.total);
  return BA_OK;
}

// record widths promised by ba.h for the schedule tables
static_assert(sizeof(BaQTile) == 10 * sizeof(int32_t), "BA_TABLE_*_QTILES record");
static_assert(sizeof(BaKvSeg) == 4 * sizeof(int32_t), "BA_TABLE_FWD_SEGS record");
static_assert(sizeof(BaKvTile) == 8 * sizeof(int32_t), "BA_TABLE_BWD_KVTILES record");
static_assert(sizeof(BaQRange) == 4 * sizeof(int32_t), "BA_TABLE_BWD_QRANGES record");

int ba_plan_get_table(ba_plan_t p, int32_t which, int32_t* out, int64_t capacity, int64_t* count) {
  if (!p) return BA_ERR_INVALID_ARG;
  // every schedule record is a run of int32 fields, copied out as they are
  const void* src = nullptr;
  int64_t n = 0;
  auto pick = [&](const auto& v) {
    using T = typename std::decay_t<decltype(v)>::value_type;
    static_assert(sizeof(T) % sizeof(int32_t) == 0, "int32 records");
    src = v.data();
    n = int64_t(v.size()) * int64_t(sizeof(T) / sizeof(int32_t));
  };
  switch (which) {
    case BA_TABLE_TOKEN_PERM: pick(p->tok_perm); break;
    case BA_TABLE_ANCHOR_PERM: pick(p->anc_perm); break;
    case BA_TABLE_ROW_LIMIT: pick(p->row_lim); break;
    case BA_TABLE_TOKEN_RANK: pick(p->tok_rank); break;
    case BA_TABLE_FWD_QTILES: pick(p->fq); break;
    case BA_TABLE_FWD_SEGS: pick(p->fseg); break;
    case BA_TABLE_BWD_QTILES: pick(p->bq); break;
    case BA_TABLE_BWD_KVTILES: pick(p->bkv); break;
    case BA_TABLE_BWD_QRANGES: pick(p->bqr); break;
    default: return BA_ERR_INVALID_ARG;
  }
  if (count) *count = n;
  if (!out) return BA_OK;
  if (capacity < n) return BA_ERR_INVALID_ARG;
  if (n > 0) std::memcpy(out, src, size_t(n) * sizeof(int32_t));
  return BA_OK;
}

int ba_plan_get_comm_volume(ba_plan_t p, int64_t* out, int32_t capacity) {
  if (!p || !out || capacity < p->C) return BA_ERR_INVALID_ARG;
  for (int r = 0; r < p->C; ++r) out[r] = p->comm[r];
  return BA_OK;
}

size_t ba_workspace_bytes(ba_plan_t p) { return p ? p->ws.total : 0; }

int ba_forward(ba_plan_t p, const void* q_b, const void* k_m, const void* v_m, const void* k_b, const void* v_b,
               void* o, float* lse, void* workspace, size_t workspace_bytes, void* stream) {
  if (!p) return BA_ERR_INVALID_ARG;
  return run_forward(p, p->shape, q_b, k_m, v_m, k_b, v_b, o, lse, workspace, workspace_bytes, stream);
}

int ba_backward(ba_plan_t p, const void* q_b, const void* k_m, const void* v_m, const void* k_b, const void* v_b,
                const void* o, const float* lse, const void* d_o, void* dq_b, void* dk_m, void* dv_m, void* dk_b,
                void* dv_b, void* workspace, size_t workspace_bytes, void* stream) {
  if (!p) return BA_ERR_INVALID_ARG;
  const BwdOut out{dq_b, dk_m, dv_m, dk_b, dv_b, nullptr, nullptr, nullptr, nullptr};
  return run_backward(p, p->shape, q_b, k_m, v_m, k_b, v_b, o, lse, d_o, out, workspace, workspace_bytes, stream);
}

size_t ba_workspace_bytes_fp8(ba_plan_t p) { return p ? p->ws.total_fp8 : 0; }

int ba_forward_fp8(ba_plan_t p, const void* q_b, const void* k_m, const void* v_m, const void* k_b, const void* v_b,
                   void* o, float* lse, void* workspace, size_t workspace_bytes, void* stream) {
  if (!p) return BA_ERR_INVALID_ARG;
  return run_forward(p, p->shape, q_b, k_m, v_m, k_b, v_b, o, lse, workspace, workspace_bytes, stream, true);
}

int ba_forward_step(ba_plan_t p, int32_t step, const void* q_s, const void* k_m, const void* v_m, const void* k_b,
                    const void* v_b, void* o_s, float* lse_s, void* workspace, size_t workspace_bytes, void* stream) {
  BaShape sh;
  if (int rc = step_shape(p, step, &sh)) return rc;
  return run_forward(p, sh, q_s, k_m, v_m, k_b, v_b, o_s, lse_s, workspace, workspace_bytes, stream);
}

int ba_backward_step(ba_plan_t p, int32_t step, const void* q_s, const void* k_m, const void* v_m, const void* k_b,
                     const void* v_b, const void* o_s, const float* lse_s, const void* d_o_s, void* dq_s,
                     float* dk_m_acc, float* dv_m_acc, float* dk_b_acc, float* dv_b_acc, void* workspace,
                     size_t workspace_bytes, void* stream) {
  BaShape sh;
  if (int rc = step_shape(p, step, &sh)) return rc;
  if (!ok_tensor(dk_m_acc) || !ok_tensor(dv_m_acc) || !ok_tensor(dk_b_acc) || !ok_tensor(dv_b_acc))
    return BA_ERR_INVALID_ARG;
  const BwdOut out{dq_s, dk_m_acc, dv_m_acc, dk_b_acc, dv_b_acc, dk_m_acc, dv_m_acc, dk_b_acc, dv_b_acc};
  return run_backward(p, sh, q_s, k_m, v_m, k_b, v_b, o_s, lse_s, d_o_s, out, workspace, workspace_bytes, stream);
}

int ba_check_device_status(ba_plan_t p, void* workspace, void* stream) {
  if (!p || !workspace) return BA_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  BA_TRY(cudaStreamSynchronize(st));
  unsigned int word = 0;
  BA_TRY(cudaMemcpy(&word, ws_at(workspace, p->ws.status), sizeof(word), cudaMemcpyDeviceToHost));
  if (word != 0) BA_TRY(cudaMemset(ws_at(workspace, p->ws.status), 0, sizeof(word)));
  switch (word) {
    case BA_DEV_OK: return BA_OK;
    case BA_DEV_TIMEOUT: return BA_ERR_DEVICE_TIMEOUT;
    default: return BA_ERR_DEVICE_BOUNDS;
  }
}

int ba_zigzag_pack(ba_plan_t p, int32_t role, const void* src, void* dst, int32_t inverse, void* workspace,
                   size_t workspace_bytes, void* stream) {
  if (!p || role < 0 || role > 2 || !ok_tensor(src) || !ok_tensor(dst) || src == dst) return BA_ERR_INVALID_ARG;
  if (role == 2 && p->shape.family == BA_FAMILY_CAUSAL) return BA_ERR_INVALID_ARG;
  if (int rc = check_ws(p, workspace, workspace_bytes)) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  BA_TRY(prepare(p, workspace, st));
  BA_TRY(pack(p, device_tables(p, workspace), role, src, dst, inverse ? 1 : 0, st));
  return BA_OK;
}

int ba_selftest_wait_timeout(ba_plan_t p, void* workspace, size_t workspace_bytes, int64_t cycles, void* stream) {
  if (!p || cycles < 0 || cycles > (int64_t(1) << 32)) return BA_ERR_INVALID_ARG;
  if (int rc = check_ws(p, workspace, workspace_bytes)) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  BA_TRY(cudaMemsetAsync(ws_at(workspace, p->ws.status), 0, 256, st));
  BA_TRY(ba_launch_selftest_wait_timeout(reinterpret_cast<unsigned int*>(ws_at(workspace, p->ws.status)),
                                         static_cast<long long>(cycles), st));
  return BA_OK;
}

int ba_lse_merge(int64_t rows, int32_t head_dim, const float* o_m, const float* l_m, const float* o_b,
                 const float* l_b, void* o, float* l, void* stream) {
  if (rows < 0 || (head_dim != 64 && head_dim != 128)) return BA_ERR_INVALID_ARG;
  if (rows == 0) return BA_OK;
  if (!ok_tensor(o_m) || !ok_tensor(o_b) || !ok_tensor(o) || !l_m || !l_b || !l) return BA_ERR_INVALID_ARG;
  BA_TRY(ba_launch_merge_rows(rows, head_dim, o_m, l_m, o_b, l_b, o, l, static_cast<cudaStream_t>(stream)));
  return BA_OK;
}

const char* ba_status_string(int s) {
  switch (s) {
    case BA_OK: return "ok";
    case BA_ERR_INVALID_ARG: return "invalid argument";
    case BA_ERR_UNSUPPORTED: return "unsupported configuration";
    case BA_ERR_CUDA: return "CUDA error";
    case BA_ERR_DEVICE_TIMEOUT: return "device wait timed out";
    case BA_ERR_DEVICE_BOUNDS: return "device table index out of range";
    case BA_ERR_WORKSPACE: return "workspace missing, too small or misaligned";
    case BA_ERR_HOST_ALLOC: return "host allocation failed";
    default: return "unknown status";
  }
}

int ba_profile_enable(ba_plan_t p, int32_t enable) {
  if (!p) return BA_ERR_INVALID_ARG;
  p->prof_on = enable != 0;
  return BA_OK;
}

int ba_profile_read(ba_plan_t p, ba_kernel_time* out, int32_t capacity, int32_t* count) {
  if (!p) return BA_ERR_INVALID_ARG;
  for (size_t i = 0; i < p->prof_used; ++i) {
    auto* a = static_cast<cudaEvent_t>(p->prof_events[2 * i]);
    auto* b = static_cast<cudaEvent_t>(p->prof_events[2 * i + 1]);
    BA_TRY(cudaEventSynchronize(b));
    float ms = 0.f;
    BA_TRY(cudaEventElapsedTime(&ms, a, b));
    p->prof_ms[p->prof_kernel[i]] += ms;
    p->prof_launches[p->prof_kernel[i]] += 1;
  }
  p->prof_used = 0;
  p->prof_kernel.clear();
  int n = 0;
  for (int k = 0; k < K_COUNT; ++k) {
    if (p->prof_launches[k] == 0) continue;
    if (out && n < capacity) {
      std::memset(out[n].name, 0, sizeof(out[n].name));
      std::strncpy(out[n].name, kKernelNames[k], sizeof(out[n].name) - 1);
      out[n].launches = p->prof_launches[k];
      out[n].total_ms = p->prof_ms[k];
    }
    ++n;
    p->prof_ms[k] = 0;
    p->prof_launches[k] = 0;
  }
  if (count) *count = n;
  return BA_OK;
}

const char* ba_last_cuda_error(void) { return g_last_cuda_error; }

const char* ba_version(void) { return "0.1 sm_103a"; }

}  // extern "C"
