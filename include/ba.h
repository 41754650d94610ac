/*
 * ba.h — C ABI of the branch-attention library (libba.so), GB300 / sm_103a.
 *
 * Draft branch attention as decomposed in "Online Draft Co-Training for
 * Speculative Decoding in Large-Scale, Long-Context RL Post-Training"
 * (arXiv 2609.07108): every branch query attends (a) the causal prefix of its
 * main sequence and (b) the keys of its own branch.  Part (a) is computed as
 * causal attention over packed, load-balanced zigzag chunks (virtual
 * context-parallel ranks visited in ring order), part (b) as rank-local
 * attention over the branch keys, and the two are merged exactly by the
 * online-softmax log-sum-exp reduction (Eq. 2).  Sources: ai.info summary,
 * Key Contributions 1 and "Methodology in Plain English"; rainbus page, core
 * method (Eq. 2, Eq. 3), method step 2 and step 5, Figure 1.
 *
 * Conventions for every entry point
 * ---------------------------------
 * - Plain C types only.  `stream` is a cudaStream_t passed as void* (NULL is
 *   the legacy default stream).  Device pointers point into memory of the
 *   current CUDA device; the library allocates no device memory and no
 *   pinned memory on the compute calls: the caller owns every device buffer,
 *   including the workspace.
 * - Tensors are dense, contiguous, row-major, bf16 (2 bytes per element)
 *   unless stated otherwise, 16-byte aligned.  "Natural" layouts:
 *     TTT (EAGLE-3 Training-Time Test, depth D):
 *         q_b, o, d_o, dq_b  [D][T][Hq][d]       lse  [D][T][Hq] fp32
 *         k_b, v_b, dk_b, dv_b [D][T][Hkv][d]
 *     BLOCK (DFlash / DSpark, block size B, NA = num_seqs * A anchors, in the
 *            order of the `anchors` array):
 *         q_b, o, d_o, dq_b  [NA][B][Hq][d]      lse  [NA][B][Hq] fp32
 *         k_b, v_b, dk_b, dv_b [NA][B][Hkv][d]
 *     CAUSAL (main queries, no branch keys):
 *         q_b, o, d_o, dq_b  [1][T][Hq][d]       lse  [1][T][Hq] fp32
 *         k_b, v_b, dk_b, dv_b unused (may be NULL)
 *     main keys/values and their gradients k_m, v_m, dk_m, dv_m [T][Hkv][d].
 *   lse is the natural-log log-sum-exp of scale * <q, k> over the query's
 *   whole key set (main prefix and branch keys).
 * - Query head h reads kv head h / (Hq / Hkv).
 * - Calls are asynchronous on `stream`.  Argument errors are returned before
 *   anything is enqueued.  Launch failures return BA_ERR_CUDA.  Device-side
 *   faults that the kernels detect themselves (bounded waits that expire,
 *   table indexes out of range) are recorded in a status word inside the
 *   workspace and reported by ba_check_device_status.
 * - No C++ exception crosses this boundary.
 */
#ifndef BA_H_
#define BA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct ba_plan* ba_plan_t;

typedef enum {
  BA_OK = 0,
  BA_ERR_INVALID_ARG = -1,    /* bad descriptor, pointer, size or alignment  */
  BA_ERR_UNSUPPORTED = -2,    /* valid but not built (e.g. head_dim 96)      */
  BA_ERR_CUDA = -3,           /* a CUDA runtime call or launch failed         */
  BA_ERR_DEVICE_TIMEOUT = -4, /* a bounded device wait expired                */
  BA_ERR_DEVICE_BOUNDS = -5,  /* a kernel found a table index out of range    */
  BA_ERR_WORKSPACE = -6,      /* workspace missing, too small or misaligned   */
  BA_ERR_HOST_ALLOC = -7      /* host memory for the plan could not be had    */
} ba_status;

typedef enum {
  BA_FAMILY_TTT = 0,    /* EAGLE-3 TTT: depth-D branch at every position       */
  BA_FAMILY_BLOCK = 1,  /* DFlash / DSpark: B-token bidirectional block/anchor */
  BA_FAMILY_CAUSAL = 2  /* main queries only: plain causal varlen attention    */
} ba_family;

/* Plan descriptor.  Host memory; copied by ba_plan_create. */
typedef struct {
  int32_t family;              /* ba_family                                      */
  int32_t num_seqs;            /* S >= 1                                         */
  const int32_t* cu_seqlens;   /* host [S+1]: 0 = cu[0] < cu[1] < ... = T        */
  int32_t heads_q, heads_kv;   /* heads_q % heads_kv == 0                        */
  int32_t head_dim;            /* 64 or 128                                      */
  float softmax_scale;         /* usually 1/sqrt(head_dim)                       */
  int32_t cp_degree;           /* virtual C >= 1; every length % (2C) == 0       */
  int32_t ttt_depth;           /* TTT: D in [1, 16]                              */
  int32_t block_size;          /* BLOCK: B in [1, 64]                            */
  int32_t anchors_per_seq;     /* BLOCK: A >= 1                                  */
  const int32_t* anchors;      /* BLOCK: host [S*A] absolute packed positions,
                                  strictly ascending within each sequence and
                                  inside it                                     */
} ba_plan_desc;

/* Figures a plan knows without running anything. */
typedef struct {
  int64_t main_tokens;          /* T                                            */
  int64_t branch_queries;       /* D*T (TTT), NA*B (BLOCK), T (CAUSAL)           */
  int64_t query_rows;           /* branch_queries * Hq                          */
  int64_t main_pairs;           /* unmasked (query-head row, main key) pairs     */
  int64_t branch_pairs;         /* unmasked (query-head row, branch key) pairs   */
  double fwd_flops;             /* 4 * d * (main_pairs + branch_pairs)           */
  double bwd_flops;             /* 2.5 * fwd_flops (recompute of S included)     */
  int64_t fwd_tiles;            /* main-attention query tiles (per stream)       */
  int64_t fwd_tile_blocks;      /* key blocks those tiles visit (per stream)     */
  int64_t bwd_kv_tiles;         /* main-attention key tiles (per kv head)        */
  int64_t comm_bytes_fwd_per_rank; /* Eq. 3 volume the ring would move (max rank) */
  int64_t workspace_bytes;      /* = ba_workspace_bytes(plan)                    */
} ba_plan_info;

/* Tables a plan can copy out (host) for inspection and tests. */
typedef enum {
  BA_TABLE_TOKEN_PERM = 0,   /* int32 [T]: packed token -> natural token         */
  BA_TABLE_ANCHOR_PERM = 1,  /* int32 [NA]: packed anchor -> natural anchor index */
  BA_TABLE_ROW_LIMIT = 2,    /* int32 [rows]: packed row -> last visible main pos */
  BA_TABLE_TOKEN_RANK = 3,   /* int32 [T]: natural token -> owning virtual rank   */
  /* The main-attention schedule, as the kernels read it (int32 records):     */
  BA_TABLE_FWD_QTILES = 4,   /* [n][10] forward query tiles: {row0, nrows, seg0,
                                nseg, lim_min, lim_max, work, chunk, nrow0, 0};
                                rows row0.. are packed rows (ROW_LIMIT index),
                                nrow0.. the same rows in natural order          */
  BA_TABLE_FWD_SEGS = 5,     /* [n][4] key segments of the forward tiles, ring
                                order: {k0, nkeys, pos0, diag}; keys pos0 ..
                                pos0 + nkeys - 1 (natural), cut by each row's
                                limit when diag = 1                             */
  BA_TABLE_BWD_QTILES = 6,   /* [n][10] backward query tiles, fields as FWD_QTILES */
  BA_TABLE_BWD_KVTILES = 7,  /* [n][8] backward key tiles: {k0, nkeys, pos0, qr0,
                                nqr, work, chunk, 0}, in groups of two tiles of
                                one chunk that share their query ranges (one
                                thread-block cluster); nkeys = 0 for the fillers
                                that complete a group                           */
  BA_TABLE_BWD_QRANGES = 8   /* [n][4] query-tile ranges of the key tiles, ring-
                                replay order: {t0, t1, diag, 0} (BWD_QTILES
                                indices t0 .. t1 - 1)                           */
} ba_table;

/* Build a plan: zigzag chunk map (2C chunks per sequence, rank r holding
 * chunks r and 2C-1-r; rainbus page, CP prerequisites, Figure 1(a)), anchor
 * ownership (a branch lives on its anchor's rank), per-row key limits, the
 * main-attention tile lists in ring order with fully masked tiles dropped,
 * longest-first, and the Eq. 3 volume.  Host only: launches nothing and needs
 * no GPU.  On success *out owns host memory freed by ba_plan_destroy.
 * Errors: BA_ERR_INVALID_ARG (descriptor), BA_ERR_UNSUPPORTED (head_dim),
 * BA_ERR_HOST_ALLOC. */
int ba_plan_create(const ba_plan_desc* desc, ba_plan_t* out);
void ba_plan_destroy(ba_plan_t plan);
/* Host self-check of a plan: every table index the kernels follow lies
 * inside the buffer it addresses, permutations are permutations, unmasked
 * key segments really are below every row limit of their tile.  BA_OK or
 * BA_ERR_INVALID_ARG. */
int ba_plan_validate(ba_plan_t plan);
int ba_plan_get_info(ba_plan_t plan, ba_plan_info* info);
/* Copies table `which` into host `out` (capacity in elements); *count gets the
 * table length.  BA_ERR_INVALID_ARG if out is too small. */
int ba_plan_get_table(ba_plan_t plan, int32_t which, int32_t* out, int64_t capacity,
                      int64_t* count);

/* Eq. 3 forward volume per virtual rank (rainbus page, core method):
 * the bytes of main K and V that rank r would receive over the C-1 ring steps,
 * counted from the plan's schedule; branch keys never move.  out: host
 * int64 [capacity >= C]. */
int ba_plan_get_comm_volume(ba_plan_t plan, int64_t* out, int32_t capacity);

/* Bytes of device workspace that ba_forward / ba_backward need (one size
 * serves both).  The workspace must be 256-byte aligned and must not be used
 * by two calls at once; consecutive calls may share it. */
size_t ba_workspace_bytes(ba_plan_t plan);

/* Forward (rainbus page, method step 2; Figure 1(b)).  Runs causal main
 * attention for each query tile over its key chunks in ring order, with the
 * online-softmax merge between ring steps; the zigzag layout lives only in the
 * plan's tile tables, so q_b, k_m and v_m are read in place (no packed
 * copies).  Each row then gets its rank-local branch part and the Eq. 2 merge
 * of the two parts in the same kernel, which writes o and lse in natural
 * order.
 * Inputs q_b, k_m, v_m, k_b, v_b; outputs o (bf16) and lse (fp32). */
int ba_forward(ba_plan_t plan, const void* q_b, const void* k_m, const void* v_m,
               const void* k_b, const void* v_b, void* o, float* lse,
               void* workspace, size_t workspace_bytes, void* stream);

/* Backward (rainbus page, method step 5: the ring is replayed and gradients
 * accumulate locally; core method: no branch-dependent traffic).  Given the
 * forward's o and lse and the output gradient d_o, writes dq_b, dk_m, dv_m,
 * dk_b, dv_b (bf16, natural layouts).  P is recomputed from the merged lse,
 * which is exact for both key sets because Eq. 2's merged result is the
 * single softmax over their union. */
int ba_backward(ba_plan_t plan, const void* q_b, const void* k_m, const void* v_m,
                const void* k_b, const void* v_b, const void* o, const float* lse,
                const void* d_o, void* dq_b, void* dk_m, void* dv_m, void* dk_b, void* dv_b,
                void* workspace, size_t workspace_bytes, void* stream);

/* Forward with 8-bit main attention (rainbus page, limitations and future
 * work, item (4): extending the decomposition to fp8 training; the same page
 * warns about precision at bf16 / fp8 beyond 256K).  Same inputs, outputs and
 * key sets as ba_forward; the main part's QK^T and PV run on e4m3 copies of
 * q_b, k_m and v_m with per-tensor scales (amax / 448, found on the device at
 * every call), while the scores, the softmax, the row sums and the lse stay
 * fp32 and the branch part and the Eq. 2 merge are computed as in ba_forward.
 * Accuracy is that of e4m3 (3 mantissa bits): o agrees with the exact result
 * to about 5-6% relative RMS on normally distributed inputs, and lse to a few
 * hundredths.  Needs head_dim 128 and every zigzag chunk starting on a
 * multiple of 16 tokens (BA_ERR_UNSUPPORTED otherwise), and a workspace of
 * ba_workspace_bytes_fp8(plan) bytes, which holds the e4m3 copies. */
size_t ba_workspace_bytes_fp8(ba_plan_t plan);
int ba_forward_fp8(ba_plan_t plan, const void* q_b, const void* k_m, const void* v_m,
                   const void* k_b, const void* v_b, void* o, float* lse,
                   void* workspace, size_t workspace_bytes, void* stream);

/* EAGLE-3 TTT one step at a time (ai.info summary, Main Findings: the
 * EAGLE-3 draft's training-time test runs its steps as separate passes, the
 * queries, keys and values of a step being produced from the draft's output of
 * the step before; rainbus page, core method: the branch keys of a step stay
 * local to the anchor's rank).  For a TTT plan of depth D, `step` s in
 * [0, D) is the step whose queries attend the causal main prefix [seq_start, p]
 * and the branch keys (p, 0..s) of their position p.  Running steps 0..D-1
 * through ba_forward_step gives the same o and lse, bit for bit, as one
 * ba_forward over all D steps.
 *   q_s, o_s        [T][Hq][d] bf16: step s's slice of q_b / o (any address,
 *                   e.g. q_b + s*T*Hq*d)
 *   lse_s           [T][Hq] fp32
 *   k_b, v_b        the whole [D][T][Hkv][d] branch buffers: slots 0..s must
 *                   hold their keys / values; slots above s are never read, so
 *                   they may still be unwritten
 *   k_m, v_m, workspace as for ba_forward (the plan's workspace size serves).
 * Errors as ba_forward, and BA_ERR_INVALID_ARG for a plan that is not TTT or
 * a step outside [0, D). */
int ba_forward_step(ba_plan_t plan, int32_t step, const void* q_s, const void* k_m, const void* v_m,
                    const void* k_b, const void* v_b, void* o_s, float* lse_s,
                    void* workspace, size_t workspace_bytes, void* stream);

/* Backward of one TTT step (rainbus page, method step 5: the ring is replayed
 * and gradients accumulate locally).  Given step s's q_s, o_s, lse_s and output
 * gradient d_o_s (slices as in ba_forward_step), writes dq_s ([T][Hq][d] bf16)
 * and ADDS step s's contributions into fp32 accumulators the caller owns:
 *   dk_m_acc, dv_m_acc  [T][Hkv][d] fp32  (main keys: every step adds)
 *   dk_b_acc, dv_b_acc  [D][T][Hkv][d] fp32  (slots 0..s receive this step's
 *                       share; slots above s are not touched)
 * Zero the accumulators before the first step of a backward pass; after all D
 * steps (in any order) they hold the gradients ba_backward returns in bf16, up
 * to rounding.  Steps that share accumulators must not overlap on the GPU.
 * Errors as ba_backward, and BA_ERR_INVALID_ARG for a plan that is not TTT, a
 * step outside [0, D) or a missing / misaligned accumulator. */
int ba_backward_step(ba_plan_t plan, int32_t step, const void* q_s, const void* k_m, const void* v_m,
                     const void* k_b, const void* v_b, const void* o_s, const float* lse_s,
                     const void* d_o_s, void* dq_s, float* dk_m_acc, float* dv_m_acc,
                     float* dk_b_acc, float* dv_b_acc, void* workspace, size_t workspace_bytes,
                     void* stream);

/* Synchronises `stream`, reads and clears the status word in `workspace`,
 * and returns the first device-side error recorded since the word was last
 * reset (BA_OK if none).  ba_forward, ba_backward and ba_zigzag_pack reset the
 * word when they start, so check after the call whose faults you want. */
int ba_check_device_status(ba_plan_t plan, void* workspace, void* stream);

/* Zigzag pack (inverse = 0) or unpack (inverse = 1) of one tensor through the
 * plan's permutation (rainbus page, CP prerequisites and method step 2: each
 * rank's shard holds, sequence by sequence, chunk r then chunk 2C-1-r; the
 * shards of ranks 0..C-1 are concatenated).  role 0: query-shaped (q_b, o,
 * d_o); role 1: main K/V shaped; role 2: branch K/V shaped.  src and dst are
 * distinct device buffers of that role's natural size.  The permutation is
 * uploaded into `workspace` (ba_workspace_bytes bytes). */
int ba_zigzag_pack(ba_plan_t plan, int32_t role, const void* src, void* dst, int32_t inverse,
                   void* workspace, size_t workspace_bytes, void* stream);

/* Forward pass that allocates nothing (no counterpart on the pages).
 * For callers that cannot allocate device memory where they run attention,
 * e.g. a plugin called from another framework's execution loop, where a
 * cudaMalloc would break that framework's memory plan or stall its stream.
 * Same inputs, outputs and results as ba_forward, but the workspace is one
 * file-scope device array of BA_NOALLOC_SCRATCH_BYTES (64 MiB) that every GPU
 * loading this library holds until the process exits.  Plans whose
 * ba_workspace_bytes exceeds that limit are rejected with BA_ERR_WORKSPACE
 * before anything runs.  The first call on a device looks the array's device
 * address up (cudaGetSymbolAddress) with that device current; make that first
 * call before any stream capture.  The address is kept per device for the
 * life of the process: after cudaDeviceReset (or anything else that tears the
 * device's context down) this entry point must not be called again in that
 * process.  All calls share the array and it keeps the last call's contents
 * (what must start at zero is cleared by each call); calls that overlap on the
 * GPU race on it, so order them.  The kernels' own fault reports (a bounded
 * wait that ran out, a table index out of range) land in the status word of
 * that hidden array, which no entry point reads back: on this path only launch
 * errors are returned, and a caller that needs the device-side checks uses
 * ba_forward with a workspace and ba_check_device_status.  No cudaMalloc,
 * cudaFree or other allocating routine is called. */
#define BA_NOALLOC_SCRATCH_BYTES (64ull << 20)
int ba_forward_noalloc(ba_plan_t plan, const void* q_b, const void* k_m, const void* v_m, const void* k_b,
                       const void* v_b, void* o, float* lse, void* stream);

/* Failure-path self-test (no counterpart on the pages): launches one CTA
 * that waits, with the library's bounded mbarrier wait, on a barrier that
 * nothing completes.  After `cycles` SM clocks (at most 2^32) the wait gives
 * up, records a timeout in the workspace status word and the kernel returns;
 * ba_check_device_status then reports BA_ERR_DEVICE_TIMEOUT.  Nothing traps,
 * faults or spins without bound. */
int ba_selftest_wait_timeout(ba_plan_t plan, void* workspace, size_t workspace_bytes, int64_t cycles,
                             void* stream);

/* Eq. 2 on caller buffers, row by row, no permutation (rainbus page, core
 * method, Eq. 2):  l = log(e^l_m + e^l_b),
 *   o = (e^(l_m-l) o_m + e^(l_b-l) o_b) / (e^(l_m-l) + e^(l_b-l)).
 * o_m, o_b fp32 [rows][head_dim]; l_m, l_b fp32 [rows] (natural log; -inf
 * marks an empty part, which merges as the identity; two empty parts give
 * o = 0, l = -inf).  Outputs o bf16 [rows][head_dim], l fp32 [rows].
 * head_dim in {64, 128}. */
int ba_lse_merge(int64_t rows, int32_t head_dim, const float* o_m, const float* l_m,
                 const float* o_b, const float* l_b, void* o, float* l, void* stream);

/* Optional per-kernel timing.  While enabled, the library brackets each of
 * its kernel launches inside ba_forward / ba_backward with a pair of CUDA
 * events recorded on the launching stream (events are created by the library
 * and reused; no device memory is allocated).  ba_profile_read waits for the
 * recorded events, adds their elapsed times per kernel name since the last
 * read, writes up to `capacity` entries and returns the entry count in
 * *count.  Names: zigzag_pack, main_fwd, bwd_prep, main_bwd_kv, main_bwd_dq,
 * branch_bwd, fp8_quantize, main_fwd_fp8. */
typedef struct {
  char name[24];
  int64_t launches;
  double total_ms;
} ba_kernel_time;
int ba_profile_enable(ba_plan_t plan, int32_t enable);
int ba_profile_read(ba_plan_t plan, ba_kernel_time* out, int32_t capacity, int32_t* count);

/* Text of the last CUDA error this thread saw inside the library ("" if
 * none); valid until the thread's next failing call. */
const char* ba_last_cuda_error(void);

/* Human-readable name of a status code (static storage). */
const char* ba_status_string(int status);

/* Library version and the architecture it was built for, e.g. "0.1 sm_103a". */
const char* ba_version(void);

#ifdef __cplusplus
}
#endif

#endif /* BA_H_ */
