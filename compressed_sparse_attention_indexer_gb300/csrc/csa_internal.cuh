// Internal definitions shared by the kernels of libcsa (not part of the ABI).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <mutex>

#include "csa.h"

namespace csa {

// Flagship tensor-core shape: H=64 heads, 576-wide rows (512 V + 64 rope),
// indexer 64 heads x 128.
constexpr int kTcH = 64, kTcD = 576, kTcV = 512, kTcHi = 64, kTcDi = 128;

// Status word bits (device side, OR-ed; integer atomics only).
constexpr int kStatusBadIndex = 1;
constexpr int kStatusTimeout = 2;

// Per-query plan flags.
constexpr int kPlanScore = 1;  // the indexer scores this query (vis > K, or forced)
constexpr int kPlanBad = 2;    // invalid length: output zeros, nothing read

constexpr int kRopeTable = 32;  // rotary frequencies kept in the config (R <= 64)

struct DevCfg {
  int H, D, V, R, Hi, Di, ratio, K, win, hca_ratio, dtype;
  int idx_fp8;  // indexer keys are FP8 E4M3 rows with a per-row fp32 scale
  float scale, rope_base;
  int max_context, max_vis;
  // polls after which the attention tile kernel's consumer waits give up
  // (negative: the default, about a second); set through the test hook
  // csa_debug_set_wait_polls
  int wait_polls;
  double rope_theta[kRopeTable];  // base^(-2i/R), i < min(R/2, kRopeTable), set on the host
};

// cos and sin of pos * theta for inverse RoPE.  The angle (up to ~6.6e4 rad)
// is formed in fp64 and reduced to [-pi, pi] by Cody-Waite reduction with
// 2*pi split into two fp64 parts (each step one fused multiply-add, so the
// reduction is exact to fp64 rounding), then sincosf of the reduced fp32
// argument.
__device__ __forceinline__ float2 rope_cos_sin(double pos, double theta) {
  const double a = pos * theta;
  const double k = rint(a * 0.15915494309189535);   // a / (2 pi)
  double r = fma(-k, 6.283185307179586, a);          // 2 pi, leading part
  r = fma(-k, 2.4492935982947064e-16, r);            // 2 pi, trailing part
  float sn, cs;
  sincosf((float)r, &sn, &cs);
  return make_float2(cs, sn);
}

struct DevBatch {
  int B, S;
  const int* ctx_len;
  const void* q;
  const void* q_idx;
  const float* w;
  const void* raw; const int64_t* raw_off; int64_t raw_stride, raw_rows;
  const void* cmp; const int64_t* cmp_off; int64_t cmp_stride, cmp_rows;
  const void* idx; const int64_t* idx_off; int64_t idx_stride, idx_rows;
  const float* idx_scale;  // [idx_rows] when the keys are FP8
  const void* hca; const int64_t* hca_off; int64_t hca_stride, hca_rows;
  // paged pools: a non-null table maps request bi's logical block k to pool
  // block table[bi * table_stride + k] of `block` rows (negative: unmapped)
  const int* raw_table; const int* cmp_table; const int* idx_table; const int* hca_table;
  int raw_block, cmp_block, idx_block, hca_block, table_stride;
};

// Pool row of logical row r of request bi: through the pool's block table when
// it is paged, else the request's first row plus r.  -1 for a row in an
// unmapped block or past the table (the callers' range checks then report it).
// (The paged lookup is a call, so that the contiguous path inlined into the
// hot loops stays small; logical rows are below 2^31.)
static __device__ __noinline__ int64_t paged_row(const int* table, int block, int tstride, int bi, int64_t r) {
  if (r < 0 || r > 0x7fffffffLL) return -1;
  const int k = (int)r / block;
  if (k >= tstride) return -1;
  const int pb = table[(int64_t)bi * tstride + k];
  return pb < 0 ? -1 : (int64_t)pb * block + ((int)r - k * block);
}
__device__ __forceinline__ int64_t pool_row(const int* table, int block, int tstride,
                                            const int64_t* off, int bi, int64_t r) {
  if (!table) return off[bi] + r;
  return paged_row(table, block, tstride, bi, r);
}
__device__ __forceinline__ int64_t raw_row(const DevBatch& b, int bi, int64_t r) {
  return pool_row(b.raw_table, b.raw_block, b.table_stride, b.raw_off, bi, r);
}
__device__ __forceinline__ int64_t cmp_row(const DevBatch& b, int bi, int64_t r) {
  return pool_row(b.cmp_table, b.cmp_block, b.table_stride, b.cmp_off, bi, r);
}
__device__ __forceinline__ int64_t idx_row(const DevBatch& b, int bi, int64_t r) {
  return pool_row(b.idx_table, b.idx_block, b.table_stride, b.idx_off, bi, r);
}
__device__ __forceinline__ int64_t hca_row(const DevBatch& b, int bi, int64_t r) {
  return pool_row(b.hca_table, b.hca_block, b.table_stride, b.hca_off, bi, r);
}

// Per-query quantities of the step (visibility, window, bypass).
struct QueryPlan {
  int pos, vis, nwin, cnt, vis2, flags;
};

// Rows of one indexer work item (tensor-core and SIMT paths).
constexpr int kIdxChunk = 128;

// Query q = b*S + s of the batch: pos = L_b - S + s, vis = floor((pos+1)/ratio),
// nwin = min(WIN, pos+1), cnt = min(vis, K), vis2 = floor((pos+1)/hca_ratio).
// The indexer scores the query when vis > K (or every query with score_all).
// A length outside [S, max_context] marks the query bad: nothing is read.
// ("Perf: skip redundant CSA scoring and fuse gather unpack": bypass when the
// visible rows fit Top-K; "Fix: port the DeepSeek-V4 MoE, hc_pre and prefill
// fixes to DSpark": at most WIN + min(vis, K) sparse rows per query.)
__device__ __forceinline__ QueryPlan query_plan(const DevCfg& c, int S, int L, int s,
                                                int score_all) {
  QueryPlan p;
  p.pos = p.vis = p.nwin = p.cnt = p.vis2 = 0;
  p.flags = 0;
  if (L < S || L > c.max_context) {
    p.flags = kPlanBad;
    return p;
  }
  p.pos = L - S + s;
  p.vis = (p.pos + 1) / c.ratio;
  p.nwin = min(c.win, p.pos + 1);
  p.vis2 = c.hca_ratio > 0 ? (p.pos + 1) / c.hca_ratio : 0;
  p.cnt = min(p.vis, c.K);
  p.flags = (p.vis > c.K || (score_all && p.vis > 0)) ? kPlanScore : 0;
  return p;
}

// Rows the indexer scores for a request: the largest vis among its scored
// queries (vis grows with s, so the last scored query decides).
__device__ __forceinline__ int request_rows(const DevCfg& c, int S, int L, int score_all) {
  if (L < S || L > c.max_context) return 0;
  int rows = 0;
  for (int s = 0; s < S; ++s) {
    const int vis = (L - S + s + 1) / c.ratio;
    if (vis > c.K || (score_all && vis > 0)) rows = max(rows, vis);
  }
  return rows;
}

// A score as an order-preserving 32-bit key (a larger score, a larger key):
// adding +0.0 turns -0.0 into +0.0 (IEEE round to nearest), then negative
// values have every bit flipped and the others only the sign bit; NaN is 0,
// below every number.  The indexer can store its scores in this form for the
// Top-K kernel of the same call.
__device__ __forceinline__ uint32_t score_order_key(float f) {
  const float g = f + 0.f;
  uint32_t u = __float_as_uint(g);
  u ^= (uint32_t)((int32_t)u >> 31) | 0x80000000u;
  return g != g ? 0u : u;
}

// Indexer items of a request (the work list's prefix[b + 1] - prefix[b]):
// its 128-row key chunks, times its query groups when split by qsplit.
__device__ __forceinline__ int request_items(const DevCfg& c, int S, int L, int score_all, int qsplit) {
  int n = (request_rows(c, S, L, score_all) + kIdxChunk - 1) / kIdxChunk;
  if (qsplit) n *= (S + qsplit - 1) / qsplit;
  return n;
}

// Indexer work list: prefix[b] = first item (128-row chunk) of request b,
// prefix[B] = number of items.  Passed by value when the host knows the
// lengths and B <= kMaxHostReq, else computed on the device by the prep
// kernel into the workspace (host_B = -1 then).
constexpr int kMaxHostReq = 1024;
struct ItemList {
  int host_B;
  int prefix[kMaxHostReq + 1];
};

// The attention job lists of a call, as prefixes over the queries.  With
// `split`, per query its W jobs (64-row tiles of the window stream, then of
// the heavy stream: nothing of the Top-K) and its C jobs (tiles of the
// compressed stream); without, no W jobs and every tile of the query (window,
// compressed, heavy) in the C list.  Built on the host when it knows the
// lengths (host_T = number of queries), else by the job-list kernel into the
// workspace (host_T = -1, no split: W prefix at ws.job_prefix[0 .. T], C
// prefix at ws.job_prefix[T + 1 .. 2T + 1]).  `early`: tile CTAs that share
// the W jobs (0: all of them); the others start when the Top-K kernel's
// blocks leave their SMs.
// With host-built lists the launcher also fills each tile CTA's first
// queries (cta_q[0][i]: the query of CTA i's first W job, cta_q[1][i]: of its
// first C job) and the list totals, so that a CTA finds its jobs without
// searching the prefixes (cta_first = 0: no per-CTA entries, search).
//
// The C list is split over the tile CTAs unevenly when the first cw_early
// CTAs (the ones that find a free SM when the grid starts) start well before
// the others (which start when the Top-K blocks leave their SMs): with
// cw_a = 0 the jobs an even split leaves over go to the early CTAs first;
// with cw_a > 0 the split is in proportion to weights, cw_a for each early
// and cw_b for each late CTA; see c_list_start.
constexpr int kMaxTileCtas = 256;
struct JobLists {
  int host_T;
  int split;
  int early;
  int cw_early, cw_a, cw_b;
  int NW, NC;  // list totals (host-built lists)
  int cta_first;
  uint16_t cta_q[2][kMaxTileCtas];
  int cta_span[2][kMaxTileCtas][2];  // the job range [first, end) of query cta_q[list][i]
  int wprefix[kMaxHostReq + 1];
  int cprefix[kMaxHostReq + 1];
};

// First C job of tile CTA i of G.  wa > 0: the C list's NC jobs split in
// proportion to the CTAs' weights (the first E weigh wa each, the rest wb);
// with equal weights this is i * NC / G.  wa == 0: every CTA takes NC / G
// jobs, and the NC % G left over go one each to the first E CTAs, then to
// the CTAs after them.
__host__ __device__ __forceinline__ int c_list_start(int i, int NC, int G, int E, int wa, int wb) {
  if (E > G) E = G;
  if (wa == 0) {
    const int per = NC / G, r = NC - per * G;
    const int r1 = r < E ? r : E;  // the early CTAs' extra jobs
    if (i <= E) return i * per + (i < r1 ? i : r1);
    const int r2 = r - r1, j = i - E;
    return i * per + r1 + (j < r2 ? j : r2);
  }
  const int64_t ci = i <= E ? (int64_t)i * wa : (int64_t)E * wa + (int64_t)(i - E) * wb;
  const int64_t cg = (int64_t)E * wa + (int64_t)(G - E) * wb;
  return (int)((int64_t)NC * ci / cg);
}

// Device workspace owned by a handle.
struct Workspace {
  int* status;        // [1]
  int* item_prefix;   // [max_batch + 1] device-computed work list (see ItemList)
  float* scores;      // [max_T, max_vis]
  int* topk_idx;      // [max_T, K]
  int* topk_cnt;      // [max_T]
  int* job_prefix;    // [2 (max_T + 1)] attention job lists (device-built, see JobLists)
  int* topk_ready;    // [max_T] per query: the step epoch whose Top-K output is complete
  int* seg_ready;     // [max_T * max_jobs] per segment slot: the launch epoch whose partial is complete
  int* idx_done;      // [2, max_batch] per request: indexer items scored (two sets, see launch_indexer)
  __nv_bfloat16* part_o;  // [max_T * max_jobs, H, V] per-segment normalised attention output
                          // (bf16: the range of fp32, so any row magnitude survives)
  float* part_lse;    // [max_T * max_jobs, H] per-segment log-sum-exp (log2 units)
  int max_T, max_batch;
  int64_t scores_ld;
};

__device__ __forceinline__ void set_status(int* status, int bit) { atomicOr(status, bit); }

// Programmatic dependent launch: wait for the grid this one depends on to
// complete (a no-op when launched without the attribute), and let the next
// grid in the stream start launching.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;\n" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
}

// Records why a launch helper gives up (the entry point's error message then
// names the failing call and its CUDA error); returns -1.  The record is per
// host thread and is consumed by the entry point that made the call.
int launch_fail(const char* what, cudaError_t e);

// Launch with or without the programmatic-stream-serialisation attribute.
// Returns 1 on a successful launch, -1 otherwise.
template <typename... KArgs, typename... Args>
int launch_kernel(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                  bool pdl, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = pdl ? at : nullptr;
  cfg.numAttrs = pdl ? 1 : 0;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, static_cast<Args&&>(args)...);
  return e == cudaSuccess ? 1 : launch_fail("cudaLaunchKernelEx", e);
}

// Host-side set-up that belongs to one device, done once per device and
// process, safely from several host threads: a kernel's shared-memory opt-in
// (cudaFuncSetAttribute) is a property of the function on the device that is
// current when it is set, so a process that drives several GPUs needs it on
// each of them.  run(set) calls set() the first time the current device
// comes through and returns true once set() has succeeded there; false if
// set() failed (it is retried by the next call) or the current device cannot
// be determined or has an ordinal of kMaxDevices or more (as a CUDA error
// code, see run()).
constexpr int kMaxDevices = 64;
class PerDeviceOnce {
 public:
  // set() returns cudaSuccess or the error of the call that failed; run()
  // returns it (cudaErrorInvalidDevice for an ordinal >= kMaxDevices)
  template <typename F>
  cudaError_t run(F&& set) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    if (done_[dev].load(std::memory_order_acquire)) return cudaSuccess;
    std::lock_guard<std::mutex> lock(mu_);
    if (done_[dev].load(std::memory_order_relaxed)) return cudaSuccess;
    e = set();
    if (e != cudaSuccess) return e;
    done_[dev].store(true, std::memory_order_release);
    return cudaSuccess;
  }

 private:
  std::mutex mu_;
  std::atomic<bool> done_[kMaxDevices]{};
};

// Raises kern's dynamic shared-memory limit on the current device to the most
// the device allows it: the per-block opt-in maximum minus the kernel's own
// static shared memory (queried, not assumed, so that it holds whatever the
// compiler adds).  A launch then fails only if it asks for more than that.
template <typename Kern>
cudaError_t allow_max_dynamic_smem(Kern* kern) {
  cudaFuncAttributes fa;
  cudaError_t e = cudaFuncGetAttributes(&fa, kern);
  if (e != cudaSuccess) return e;
  int dev = 0, optin = 0;
  e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              optin - (int)fa.sharedSizeBytes);
}

// The driver's cuTensorMapEncodeTiled, looked up once per process (a
// function-local static: its initialisation is thread-safe); NULL if the
// driver does not provide it.
void* tensor_map_encoder();

// ---- launch wrappers (defined in the kernel files) -------------------------
// Each returns the number of kernels launched (>= 0) or -1 on a launch error.
// `pdl`: launch as a programmatic dependent of the previous kernel.
int launch_prep(const DevCfg& c, const DevBatch& b, const Workspace& ws, int score_all, int qsplit,
                cudaStream_t st, bool pdl);
// done / done_clear (may be NULL): with the tcgen05 kernel, each CTA adds
// (release) to done[b] the number of request b's items it has scored once
// their scores are stored, and the kernel's CTA 0 zeroes the whole set
// done_clear[0, ws.max_batch) (the set the next such launch uses, whatever
// its batch size); *published says whether it did.
// keys (tcgen05 kernel only): the scores are stored as score_order_key bits;
// *keyed says whether they were.
int launch_indexer(const DevCfg& c, const DevBatch& b, const Workspace& ws, const ItemList& items,
                   int score_all, float* scores, int64_t ld, int num_sms, cudaStream_t st,
                   bool pdl, int* done = nullptr, int* done_clear = nullptr,
                   bool* published = nullptr, bool keys = false, bool* keyed = nullptr);
bool indexer_tc5_fits(const DevCfg& c, int S);
// queries per group when a request's work is split by query group (see
// indexer_qsplit): the warp-MMA indexer's q_idx group, and the tcgen05
// indexer's unit (one MMA of N = 4 x 64 over a key chunk)
constexpr int kMmaGroup = 8;
constexpr int kT5Group = 4;
int indexer_qsplit(const DevCfg& c, int S);
int launch_indexer_tc5(const DevCfg& c, const DevBatch& b, const Workspace& ws,
                       const ItemList& items, int score_all, float* scores, int64_t ld,
                       int num_sms, int qsplit, cudaStream_t st, bool pdl, int* done = nullptr,
                       int* done_clear = nullptr, bool keys = false);
// The cache update before a step: pool[slot[t]] = src[t] (row_bytes each) for
// t < n; strides in bytes; status may be NULL.
int launch_writeback(const void* src, int64_t src_stride, const int64_t* slot, int n, void* pool,
                     int64_t pool_stride, int64_t pool_rows, int64_t row_bytes, int* status,
                     cudaStream_t st, bool pdl);
// early: this library's own kernel of the same call runs right before (the
// lengths are then read before the grid dependency wait)
// ready / epoch: when ready is not NULL, each query's block stores `epoch`
// into ready[q] once its outputs are complete (the attention kernel of the
// same step starts that query's compressed tiles on it)
// done (with early and b): the indexer of the same call publishes each
// request's scored items there (see launch_indexer); a block then waits for
// its request's items instead of the indexer grid, and for the grid only at
// its end.  qsplit: the indexer's queries per item group (indexer_qsplit).
// keys: the scores are score_order_key bits (only with the register kernel,
// topk_use_reg).
int launch_topk(const DevCfg& c, const DevBatch* b, int nq, const float* scores, int64_t ld,
                const int* n_override, int* idx_out, int* cnt_out, int* status, int max_vis,
                cudaStream_t st, bool pdl, bool early, int* ready = nullptr, int epoch = 0,
                const int* done = nullptr, int qsplit = 0, bool keys = false);
bool topk_use_reg(int max_vis);
int launch_attention(const DevCfg& c, const DevBatch& b, const Workspace& ws, const int* topk_idx,
                     const int* topk_cnt, void* out, float* lse_out, int num_sms,
                     cudaStream_t st, bool pdl);
// early: launched right after this library's Top-K kernel of the same step,
// which signals each query through ws.topk_ready with `epoch`: the tile
// kernel reads the caller's inputs before its grid wait and starts a query's
// compressed tiles once that query's Top-K output is complete.
// seg_epoch: this launch's value of the per-segment ready flags (never 0 and
// never the previous launch's), through which the merge kernel starts a
// query once every partial of it is written.
int launch_attention_tc5(const DevCfg& c, const DevBatch& b, const Workspace& ws,
                         JobLists& jobs, const int* topk_idx, const int* topk_cnt, void* out,
                         float* lse_out, int num_sms, cudaStream_t st, bool pdl, bool early,
                         int epoch, int seg_epoch);
// Builds the job lists on the host when the lengths are known; `topk_blocks`:
// Top-K blocks of the step that select (their SMs are busy when the tile
// kernel starts), 0 when no Top-K kernel runs right before.
void host_jobs(const DevCfg& c, int B, int S, const int32_t* lens_host, int num_sms, int topk_blocks,
               JobLists* jobs);
int max_jobs_per_query(const DevCfg& c);
constexpr int kAttnMma = 0, kAttnTc5 = 1;
int attention_impl();

bool tensor_core_shape(const DevCfg& c);
constexpr int kIndexerMma = 0, kIndexerTc5 = 1;
int indexer_impl();

}  // namespace csa
