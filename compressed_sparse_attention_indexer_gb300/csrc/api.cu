// The C ABI (include/csa.h): argument validation, workspace ownership and the
// launch sequence of each entry point.  No computation happens on the host.
#include <math.h>
#include <stdarg.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <mutex>
#include <string>
#include <vector>

#include <cuda.h>

#include "csa_internal.cuh"

struct csa_handle {
  csa_config cfg;
  csa::DevCfg dc;
  csa::Workspace ws;
  void* ws_base;
  size_t ws_bytes;
  int device;
  int num_sms;
  int last_launches;
  // per-stage timing (csa_profile_enable): event pairs recorded around each
  // launch on its stream, resolved by csa_profile_read
  bool prof = false;
  struct Mark { int stage; cudaEvent_t a, b; };
  std::vector<Mark> marks;
  std::vector<cudaEvent_t> spare;
  csa::ItemList items;  // host-built indexer work list of the current call
  csa::JobLists jobs;   // host-built attention job lists of the current call
  int max_jobs = 0;     // attention tiles per query, at most
  int epoch = 0;        // decode steps launched (the Top-K ready flags' value)
  int seg_epoch = 0;    // tile-kernel launches (the segment ready flags' value)
  int done_set = 0;     // the indexer completion-counter set (ws.idx_done) the next publishing launch uses
};

namespace {
// queries per request up to which a decode step's Top-K blocks wait on the
// indexer's per-request counters (see csa_decode_step)
constexpr int kCounterMaxS = 1;
enum Stage { kStagePlan = 0, kStageIndexer = 1, kStageTopk = 2, kStageAttention = 3, kStages = 4 };

cudaEvent_t take_event(csa_handle* h) {
  if (!h->spare.empty()) {
    cudaEvent_t e = h->spare.back();
    h->spare.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  cudaEventCreate(&e);
  return e;
}

// Runs one launch helper, bracketed by events when profiling is on.
template <typename F>
int staged(csa_handle* h, int stage, cudaStream_t st, F&& launch) {
  if (!h->prof) return launch();
  cudaEvent_t a = take_event(h), b = take_event(h);
  cudaEventRecord(a, st);
  const int r = launch();
  cudaEventRecord(b, st);
  if (r > 0) h->marks.push_back({stage, a, b});
  else { h->spare.push_back(a); h->spare.push_back(b); }
  return r;
}
}  // namespace

namespace {

thread_local std::string g_err;

int fail(int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_err = buf;
  return code;
}

int cuda_fail(cudaError_t e, const char* what) {
  return fail(CSA_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

constexpr int kMaxVisCap = 40960;  // keys of one query held in shared memory by the Top-K kernel

int validate_cfg(const csa_config* c) {
  if (!c) return fail(CSA_ERR_INVALID_ARG, "cfg is NULL");
  if (c->heads < 1 || c->row_dim < 1 || c->v_dim < 1 || c->v_dim > c->row_dim)
    return fail(CSA_ERR_INVALID_ARG, "need heads >= 1 and 1 <= v_dim <= row_dim");
  if ((c->row_dim - c->v_dim) % 2 != 0)
    return fail(CSA_ERR_INVALID_ARG, "rope dims row_dim - v_dim must be even");
  if (c->idx_heads < 1 || c->idx_dim < 1) return fail(CSA_ERR_INVALID_ARG, "bad indexer shape");
  if (c->ratio < 1 || c->topk < 1 || c->win < 1 || c->hca_ratio < 0)
    return fail(CSA_ERR_INVALID_ARG, "need ratio, topk, win >= 1 and hca_ratio >= 0");
  if (c->dtype != CSA_DTYPE_F32 && c->dtype != CSA_DTYPE_BF16)
    return fail(CSA_ERR_UNSUPPORTED, "dtype must be CSA_DTYPE_F32 or CSA_DTYPE_BF16");
  if (c->idx_dtype != 0 && c->idx_dtype != CSA_DTYPE_FP8_E4M3)
    return fail(CSA_ERR_UNSUPPORTED, "idx_dtype must be 0 (the layer dtype) or CSA_DTYPE_FP8_E4M3");
  if (c->idx_dtype == CSA_DTYPE_FP8_E4M3 &&
      (c->dtype != CSA_DTYPE_BF16 || c->idx_heads != csa::kTcHi || c->idx_dim != csa::kTcDi))
    return fail(CSA_ERR_UNSUPPORTED, "FP8 indexer keys need dtype bf16, idx_heads %d, idx_dim %d",
                csa::kTcHi, csa::kTcDi);
  if (c->max_batch < 1 || c->max_queries_per_req < 1 || c->max_context < 1)
    return fail(CSA_ERR_INVALID_ARG, "workspace maxima must be >= 1");
  if (c->max_context / c->ratio > kMaxVisCap)
    return fail(CSA_ERR_UNSUPPORTED, "max_context / ratio = %d exceeds %d",
                c->max_context / c->ratio, kMaxVisCap);
  if (c->topk > kMaxVisCap) return fail(CSA_ERR_UNSUPPORTED, "topk above %d", kMaxVisCap);
  if (!(c->rope_base > 0.f)) return fail(CSA_ERR_INVALID_ARG, "rope_base must be > 0");
  if ((int64_t)c->max_batch * c->max_queries_per_req > (1 << 24))
    return fail(CSA_ERR_UNSUPPORTED, "max_batch * max_queries_per_req too large");
  // shapes outside the tensor-core set run on the SIMT path, which holds V/32
  // accumulators per lane
  if (c->v_dim > 512) return fail(CSA_ERR_UNSUPPORTED, "v_dim above 512");
  return CSA_OK;
}

int validate_batch_cfg(const csa_config& c, const csa_batch* b) {
  if (!b) return fail(CSA_ERR_INVALID_ARG, "batch is NULL");
  if (b->B < 0 || b->S < 1) return fail(CSA_ERR_INVALID_ARG, "need B >= 0 and S >= 1");
  if (b->B > c.max_batch || b->S > c.max_queries_per_req)
    return fail(CSA_ERR_WORKSPACE, "B=%d S=%d above create-time maxima %d, %d", b->B, b->S,
                c.max_batch, c.max_queries_per_req);
  if (b->B == 0) return CSA_OK;
  const int es = c.dtype == CSA_DTYPE_BF16 ? 2 : 4;
  const bool fp8 = c.idx_dtype == CSA_DTYPE_FP8_E4M3;
  // a paged pool's offsets are not read
  const void* dummy = b->q;
  struct P { const void* p; const char* n; } ptrs[] = {
      {b->ctx_len, "ctx_len"}, {b->q, "q"}, {b->q_idx, "q_idx"}, {b->w, "w"},
      {b->raw_kv, "raw_kv"}, {b->raw_table ? dummy : b->raw_off, "raw_off"}, {b->cmp_kv, "cmp_kv"},
      {b->cmp_table ? dummy : b->cmp_off, "cmp_off"}, {b->idx_k, "idx_k"},
      {b->idx_table ? dummy : b->idx_off, "idx_off"}};
  for (const P& x : ptrs)
    if (!x.p) return fail(CSA_ERR_INVALID_ARG, "%s is NULL", x.n);
  for (const P& x : ptrs)
    if (!aligned16(x.p)) return fail(CSA_ERR_INVALID_ARG, "%s is not 16-byte aligned", x.n);
  struct Pool { int64_t stride, rows; int width; const char* n; } pools[] = {
      {b->raw_stride, b->raw_rows, c.row_dim, "raw"},
      {b->cmp_stride, b->cmp_rows, c.row_dim, "cmp"},
      {b->idx_stride, b->idx_rows, c.idx_dim, "idx"},
      {b->hca_stride, b->hca_rows, c.row_dim, "hca"}};
  for (int i = 0; i < 4; ++i) {
    const Pool& x = pools[i];
    if (i == 3 && c.hca_ratio == 0) continue;
    if (x.stride < x.width) return fail(CSA_ERR_INVALID_ARG, "%s_stride below the row width", x.n);
    if ((x.stride * (i == 2 && fp8 ? 1 : es)) % 16 != 0)
      return fail(CSA_ERR_INVALID_ARG, "%s_stride * element size is not a multiple of 16", x.n);
    if (x.rows < 0) return fail(CSA_ERR_INVALID_ARG, "%s_rows < 0", x.n);
  }
  if (fp8 && (!b->idx_scale || !aligned16(b->idx_scale)))
    return fail(CSA_ERR_INVALID_ARG, "idx_scale is NULL or not 16-byte aligned with FP8 keys");
  if (c.hca_ratio > 0) {
    const void* hoff = b->hca_table ? b->hca_kv : b->hca_off;
    if (!b->hca_kv || !hoff) return fail(CSA_ERR_INVALID_ARG, "hca_kv/hca_off NULL with hca_ratio > 0");
    if (!aligned16(b->hca_kv) || !aligned16(hoff))
      return fail(CSA_ERR_INVALID_ARG, "hca_kv/hca_off not 16-byte aligned");
  }
  struct T { const int32_t* t; int32_t blk; const char* n; } tabs[] = {
      {b->raw_table, b->raw_block, "raw"}, {b->cmp_table, b->cmp_block, "cmp"},
      {b->idx_table, b->idx_block, "idx"}, {b->hca_table, b->hca_block, "hca"}};
  bool paged = false;
  for (const T& x : tabs) {
    if (!x.t) continue;
    paged = true;
    if ((reinterpret_cast<uintptr_t>(x.t) & 3u) != 0)
      return fail(CSA_ERR_INVALID_ARG, "%s_table is not 4-byte aligned", x.n);
    if (x.blk < 1) return fail(CSA_ERR_INVALID_ARG, "%s_block < 1 with a %s_table", x.n, x.n);
  }
  if (paged && b->table_stride < 1) return fail(CSA_ERR_INVALID_ARG, "table_stride < 1 with a block table");
  if (b->idx_table && b->idx_block % 128 != 0)
    return fail(CSA_ERR_INVALID_ARG, "idx_block = %d is not a multiple of 128", b->idx_block);
  if (b->ctx_len_host) {
    for (int i = 0; i < b->B; ++i) {
      const int L = b->ctx_len_host[i];
      if (L < b->S || L > c.max_context)
        return fail(CSA_ERR_WORKSPACE, "ctx_len[%d] = %d outside [S, max_context] = [%d, %d]", i, L,
                    b->S, c.max_context);
    }
  }
  return CSA_OK;
}

int validate_batch(const csa_handle* h, const csa_batch* b) {
  if (!h) return fail(CSA_ERR_INVALID_ARG, "handle is NULL");
  return validate_batch_cfg(h->cfg, b);
}

csa::DevBatch dev_batch(const csa_batch* b) {
  csa::DevBatch d;
  d.B = b->B; d.S = b->S; d.ctx_len = b->ctx_len;
  d.q = b->q; d.q_idx = b->q_idx; d.w = b->w;
  d.raw = b->raw_kv; d.raw_off = b->raw_off; d.raw_stride = b->raw_stride; d.raw_rows = b->raw_rows;
  d.cmp = b->cmp_kv; d.cmp_off = b->cmp_off; d.cmp_stride = b->cmp_stride; d.cmp_rows = b->cmp_rows;
  d.idx = b->idx_k; d.idx_off = b->idx_off; d.idx_stride = b->idx_stride; d.idx_rows = b->idx_rows;
  d.idx_scale = b->idx_scale;
  d.raw_table = b->raw_table; d.cmp_table = b->cmp_table;
  d.idx_table = b->idx_table; d.hca_table = b->hca_table;
  d.raw_block = b->raw_block; d.cmp_block = b->cmp_block;
  d.idx_block = b->idx_block; d.hca_block = b->hca_block;
  d.table_stride = b->table_stride;
  d.hca = b->hca_kv; d.hca_off = b->hca_off; d.hca_stride = b->hca_stride; d.hca_rows = b->hca_rows;
  return d;
}

// The indexer's work list (see csa::ItemList): built here when the host knows
// the lengths and B is small enough to pass by value; otherwise host_B = -1
// and the prep kernel builds it on the device.
void host_items(const csa_handle* h, const csa_batch* b, int score_all, csa::ItemList* it) {
  it->host_B = -1;
  if (!b->ctx_len_host || b->B > csa::kMaxHostReq) return;
  const csa_config& c = h->cfg;
  int acc = 0;
  for (int i = 0; i < b->B; ++i) {
    it->prefix[i] = acc;
    const int L = b->ctx_len_host[i];
    int rows = 0;
    for (int s = 0; s < b->S; ++s) {
      const int vis = (L - b->S + s + 1) / c.ratio;
      if (vis > c.topk || (score_all && vis > 0)) rows = vis > rows ? vis : rows;
    }
    int n = (rows + csa::kIdxChunk - 1) / csa::kIdxChunk;
    const int qs = csa::indexer_qsplit(h->dc, b->S);
    if (qs) n *= (b->S + qs - 1) / qs;  // (query group, key chunk) items
    acc += n;
  }
  it->prefix[b->B] = acc;
  it->host_B = b->B;
}

// Programmatic dependent launch between the kernels of a call (and with the
// stream's previous kernel): on unless CSA_PDL=0.  Every kernel waits for its
// predecessor before touching global memory, so the overlap is only of launch
// latency and prologues.
bool use_pdl() {
  static int v = -1;
  if (v < 0) {
    const char* e = getenv("CSA_PDL");
    v = (e && strcmp(e, "0") == 0) ? 0 : 1;
  }
  return v == 1;
}

// attention: the tcgen05 tile kernel + merge for the tensor-core shape
// (unless CSA_ATTN=mma or the batch does not fit it), else the warp-MMA or
// SIMT kernel
// early: the Top-K kernel of the same call runs right before (see
// launch_attention_tc5)
// The tile CTAs' split of the job lists follows from the batch alone (the
// queries whose Top-K blocks select, vis > K, keep SMs busy when the tile
// kernel of a decode step starts), whichever entry point launches it, so the
// same batch and Top-K give the same output bits from csa_decode_step and
// csa_sparse_attn.
int run_attention(csa_handle* h, const csa_batch* b, const csa::DevBatch& db, const int* idx,
                  const int* cnt, void* out, float* lse, cudaStream_t st, bool pdl, bool early) {
  if (csa::tensor_core_shape(h->dc) && csa::attention_impl() == csa::kAttnTc5) {
    int selecting = 0;
    if (b->ctx_len_host)
      for (int i = 0; i < b->B; ++i)
        for (int s = 0; s < b->S; ++s)
          selecting += (b->ctx_len_host[i] - b->S + s + 1) / h->cfg.ratio > h->cfg.topk ? 1 : 0;
    csa::host_jobs(h->dc, b->B, b->S, b->ctx_len_host, h->num_sms, selecting, &h->jobs);
    h->seg_epoch = h->seg_epoch == 0x7fffffff ? 1 : h->seg_epoch + 1;
    const int r = csa::launch_attention_tc5(h->dc, db, h->ws, h->jobs, idx, cnt, out, lse,
                                            h->num_sms, st, pdl, early, h->epoch, h->seg_epoch);
    if (r != -2) return r;
  }
  return csa::launch_attention(h->dc, db, h->ws, idx, cnt, out, lse, h->num_sms, st, pdl);
}

struct Launches {
  int n = 0;
  bool ok = true;
  void add(int r) {
    if (r < 0) ok = false; else n += r;
  }
};

thread_local std::string g_launch_why;  // see csa::launch_fail

int finish(csa_handle* h, const Launches& L) {
  h->last_launches = L.n;
  std::string why;
  why.swap(g_launch_why);
  if (!L.ok) {
    if (!why.empty()) return fail(CSA_ERR_CUDA, "kernel launch: %s", why.c_str());
    cudaError_t e = cudaGetLastError();
    return cuda_fail(e, "kernel launch");
  }
  return CSA_OK;
}

// plan (if needed) + indexer into `scores`.  done (not NULL): the tcgen05
// indexer publishes each request's scored items to the handle's current
// counter set and zeroes the other one; *done then points at the set it used
// (NULL if no kernel published), and the next publishing launch uses the other.
void run_indexer(csa_handle* h, const csa_batch* b, const csa::DevBatch& db, int score_all,
                 float* scores, int64_t ld, cudaStream_t st, Launches& L, int** done = nullptr,
                 bool keys = false, bool* keyed = nullptr) {
  csa::ItemList& items = h->items;
  host_items(h, b, score_all, &items);
  const bool pdl = use_pdl();
  if (items.host_B < 0)
    L.add(staged(h, kStagePlan, st,
                 [&] {
                   return csa::launch_prep(h->dc, db, h->ws, score_all,
                                           csa::indexer_qsplit(h->dc, b->S), st, pdl);
                 }));
  int* cur = nullptr;
  int* other = nullptr;
  if (done && h->ws.idx_done) {
    cur = h->ws.idx_done + (size_t)h->done_set * h->ws.max_batch;
    other = h->ws.idx_done + (size_t)(h->done_set ^ 1) * h->ws.max_batch;
  }
  bool published = false, wrote_keys = false;
  L.add(staged(h, kStageIndexer, st, [&] {
    return csa::launch_indexer(h->dc, db, h->ws, items, score_all, scores, ld, h->num_sms, st, pdl,
                               cur, other, &published, keys, &wrote_keys);
  }));
  if (keyed) *keyed = wrote_keys;
  if (done) *done = published ? cur : nullptr;
  if (published) h->done_set ^= 1;
}

// ---- allocation-free variant of indexer + Top-K ----------------------------
// Its scratch (status word, indexer work list, score matrix) lives in this
// file-scope device array, loaded with the module; nothing is allocated per
// call.  One array per device and process, so calls that overlap in time
// (other streams or threads on the same device) share it and race.
constexpr size_t kStaticScratchBytes = size_t(8) << 20;  // 8 MiB
static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

// The array's device address is a property of the CUDA context the module is
// loaded in: normally one (the primary context) per device, but a device reset
// or a driver-API context made current loads the module again, possibly at
// another address.  The address is therefore kept per context, keyed by the
// context's unique id, and looked up the first time a context calls in.
struct StaticSlot {
  unsigned long long ctx_id;
  void* addr;
  int sms;
};
constexpr int kMaxStaticContexts = 64;
std::mutex g_static_mu;
StaticSlot g_static_slots[kMaxStaticContexts];
int g_static_nslots = 0;

// Unique id of the calling thread's current context (cuCtxGetCurrent and
// cuCtxGetId, through the runtime's driver entry points so that nothing links
// the driver library directly).  After a runtime call has run on the current
// device (cudaGetDevice does not create a context, the caller's cudaSetDevice
// or any earlier call does), its primary context is current.  False if the
// driver lacks the calls or no context is current.
bool current_context_id(unsigned long long* id) {
  typedef CUresult (*GetCurrent)(CUcontext*);
  typedef CUresult (*GetId)(CUcontext, unsigned long long*);
  static const GetCurrent get_current = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult r;
    return (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &r) ==
                cudaSuccess && r == cudaDriverEntryPointSuccess)
               ? reinterpret_cast<GetCurrent>(p) : nullptr;
  }();
  static const GetId get_id = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult r;
    return (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &r) ==
                cudaSuccess && r == cudaDriverEntryPointSuccess)
               ? reinterpret_cast<GetId>(p) : nullptr;
  }();
  if (!get_current || !get_id) return false;
  CUcontext ctx = nullptr;
  if (get_current(&ctx) != CUDA_SUCCESS || !ctx) return false;
  return get_id(ctx, id) == CUDA_SUCCESS;
}

// The config as the kernels read it (what csa_decode_create stores in a
// handle).
csa::DevCfg static_devcfg(const csa_config& c) {
  csa::DevCfg d;
  d.H = c.heads; d.D = c.row_dim; d.V = c.v_dim; d.R = c.row_dim - c.v_dim;
  d.Hi = c.idx_heads; d.Di = c.idx_dim; d.ratio = c.ratio; d.K = c.topk;
  d.win = c.win; d.hca_ratio = c.hca_ratio; d.dtype = c.dtype;
  d.idx_fp8 = c.idx_dtype == CSA_DTYPE_FP8_E4M3;
  d.scale = c.softmax_scale > 0.f ? c.softmax_scale : (float)(1.0 / sqrt((double)c.row_dim));
  d.rope_base = c.rope_base;
  d.max_context = c.max_context;
  d.max_vis = c.max_context / c.ratio;
  d.wait_polls = -1;
  for (int i = 0; i < csa::kRopeTable; ++i)
    d.rope_theta[i] = (d.R > 0 && i < d.R / 2)
                          ? pow((double)c.rope_base, -2.0 * (double)i / (double)d.R) : 0.0;
  return d;
}

// Bytes of scratch a batch needs: the status word, the work list, the
// [B*S, max_context/ratio] fp32 score matrix, each 256-byte aligned.
size_t static_scratch_need(const csa_config& c, const csa_batch* b, size_t* o_prefix,
                           size_t* o_scores) {
  auto al = [](size_t x) { return (x + 255) & ~size_t(255); };
  const size_t ld = (size_t)(c.max_context / c.ratio > 0 ? c.max_context / c.ratio : 1);
  *o_prefix = 256;
  *o_scores = *o_prefix + al(sizeof(int) * ((size_t)b->B + 1));
  return *o_scores + al(sizeof(float) * ld * (size_t)b->B * (size_t)b->S);
}

}  // namespace

namespace csa {
int launch_fail(const char* what, cudaError_t e) {
  if (g_launch_why.empty()) {  // the first failure of a call is the one to report
    g_launch_why = what;
    if (e != cudaSuccess) {
      g_launch_why += ": ";
      g_launch_why += cudaGetErrorString(e);
    }
  }
  return -1;
}
}  // namespace csa

extern "C" {

int32_t csa_abi_version(void) { return CSA_ABI_VERSION; }

const char* csa_last_error(void) { return g_err.c_str(); }

int32_t csa_last_launch_count(const csa_handle* h) { return h ? h->last_launches : -1; }

int csa_decode_create(const csa_config* cfg, csa_handle** out) {
  if (!out) return fail(CSA_ERR_INVALID_ARG, "out is NULL");
  int rc = validate_cfg(cfg);
  if (rc) return rc;
  csa_handle* h = new csa_handle();
  h->cfg = *cfg;
  csa::DevCfg& d = h->dc;
  d.H = cfg->heads; d.D = cfg->row_dim; d.V = cfg->v_dim; d.R = cfg->row_dim - cfg->v_dim;
  d.Hi = cfg->idx_heads; d.Di = cfg->idx_dim; d.ratio = cfg->ratio; d.K = cfg->topk;
  d.win = cfg->win; d.hca_ratio = cfg->hca_ratio; d.dtype = cfg->dtype;
  d.idx_fp8 = cfg->idx_dtype == CSA_DTYPE_FP8_E4M3;
  d.scale = cfg->softmax_scale > 0.f ? cfg->softmax_scale : (float)(1.0 / sqrt((double)cfg->row_dim));
  d.rope_base = cfg->rope_base;
  d.max_context = cfg->max_context;
  d.max_vis = cfg->max_context / cfg->ratio;
  d.wait_polls = -1;
  for (int i = 0; i < csa::kRopeTable; ++i)
    d.rope_theta[i] = (d.R > 0 && i < d.R / 2)
                          ? pow((double)cfg->rope_base, -2.0 * (double)i / (double)d.R) : 0.0;

  cudaError_t e = cudaGetDevice(&h->device);
  if (e != cudaSuccess) { delete h; return cuda_fail(e, "cudaGetDevice"); }
  e = cudaDeviceGetAttribute(&h->num_sms, cudaDevAttrMultiProcessorCount, h->device);
  if (e != cudaSuccess) { delete h; return cuda_fail(e, "cudaDeviceGetAttribute"); }

  const int maxT = cfg->max_batch * cfg->max_queries_per_req;
  const int64_t ld = d.max_vis > 0 ? d.max_vis : 1;
  auto al = [](size_t x) { return (x + 255) & ~size_t(255); };
  size_t off = 0;
  const size_t o_status = off; off += al(sizeof(int));
  const size_t o_prefix = off; off += al(sizeof(int) * (cfg->max_batch + 1));
  const size_t o_scores = off; off += al(sizeof(float) * ld * maxT);
  const size_t o_idx = off; off += al(sizeof(int) * (size_t)cfg->topk * maxT);
  const size_t o_cnt = off; off += al(sizeof(int) * maxT);
  const bool tc = csa::tensor_core_shape(d);
  h->max_jobs = tc ? csa::max_jobs_per_query(d) : 0;
  const size_t o_jobs = off; off += al(sizeof(int) * 2 * (maxT + 1));
  const size_t o_ready = off; off += al(sizeof(int) * maxT);
  const size_t o_part = off; off += tc ? al(sizeof(__nv_bfloat16) * (size_t)maxT * h->max_jobs * d.H * d.V) : 0;
  const size_t o_plse = off; off += tc ? al(sizeof(float) * (size_t)maxT * h->max_jobs * d.H) : 0;
  const size_t o_sready = off; off += tc ? al(sizeof(int) * (size_t)maxT * h->max_jobs) : 0;
  const size_t o_done = off; off += al(sizeof(int) * 2 * (size_t)cfg->max_batch);
  h->ws_bytes = off;
  e = cudaMalloc(&h->ws_base, off);
  if (e != cudaSuccess) { delete h; return cuda_fail(e, "cudaMalloc(workspace)"); }
  char* base = static_cast<char*>(h->ws_base);
  e = cudaMemset(base + o_status, 0, sizeof(int));
  if (e == cudaSuccess) e = cudaMemset(base + o_ready, 0, sizeof(int) * maxT);  // epoch 0: never a step's
  if (e == cudaSuccess && tc) e = cudaMemset(base + o_sready, 0, sizeof(int) * (size_t)maxT * h->max_jobs);
  if (e == cudaSuccess) e = cudaMemset(base + o_done, 0, sizeof(int) * 2 * (size_t)cfg->max_batch);
  if (e != cudaSuccess) { cudaFree(h->ws_base); delete h; return cuda_fail(e, "cudaMemset"); }
  csa::Workspace& w = h->ws;
  w.status = reinterpret_cast<int*>(base + o_status);
  w.item_prefix = reinterpret_cast<int*>(base + o_prefix);
  w.scores = reinterpret_cast<float*>(base + o_scores);
  w.topk_idx = reinterpret_cast<int*>(base + o_idx);
  w.topk_cnt = reinterpret_cast<int*>(base + o_cnt);
  w.job_prefix = reinterpret_cast<int*>(base + o_jobs);
  w.topk_ready = reinterpret_cast<int*>(base + o_ready);
  w.part_o = tc ? reinterpret_cast<__nv_bfloat16*>(base + o_part) : nullptr;
  w.part_lse = tc ? reinterpret_cast<float*>(base + o_plse) : nullptr;
  w.seg_ready = tc ? reinterpret_cast<int*>(base + o_sready) : nullptr;
  w.idx_done = reinterpret_cast<int*>(base + o_done);
  w.max_T = maxT;
  w.max_batch = cfg->max_batch;
  w.scores_ld = ld;
  *out = h;
  g_err.clear();
  return CSA_OK;
}

void csa_decode_destroy(csa_handle* h) {
  if (!h) return;
  cudaDeviceSynchronize();
  for (auto& m : h->marks) { cudaEventDestroy(m.a); cudaEventDestroy(m.b); }
  for (auto e : h->spare) cudaEventDestroy(e);
  cudaFree(h->ws_base);
  delete h;
}

int csa_indexer_topk(csa_handle* h, const csa_batch* b, int32_t* topk_idx, int32_t* topk_cnt,
                     void* stream) {
  int rc = validate_batch(h, b);
  if (rc) return rc;
  if (!topk_idx || !topk_cnt) return fail(CSA_ERR_INVALID_ARG, "topk_idx/topk_cnt NULL");
  if (b->B == 0) { h->last_launches = 0; return CSA_OK; }
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const csa::DevBatch db = dev_batch(b);
  const bool pdl = use_pdl();
  Launches L;
  // the internal scores go to Top-K as order-preserving keys when the
  // register kernel selects (it then skips the conversion)
  bool keyed = false;
  run_indexer(h, b, db, 0, h->ws.scores, h->ws.scores_ld, st, L, nullptr,
              csa::topk_use_reg(h->dc.max_vis), &keyed);
  const bool early = L.n > 0;  // the plan or indexer kernel runs right before
  L.add(staged(h, kStageTopk, st, [&] {
    return csa::launch_topk(h->dc, &db, b->B * b->S, h->ws.scores, h->ws.scores_ld, nullptr,
                            topk_idx, topk_cnt, h->ws.status, h->dc.max_vis, st, pdl, early,
                            nullptr, 0, nullptr, 0, keyed);
  }));
  return finish(h, L);
}

int csa_sparse_attn(csa_handle* h, const csa_batch* b, const int32_t* topk_idx,
                    const int32_t* topk_cnt, void* out, float* lse_out, void* stream) {
  int rc = validate_batch(h, b);
  if (rc) return rc;
  if (!topk_idx || !topk_cnt || !out) return fail(CSA_ERR_INVALID_ARG, "topk_idx/topk_cnt/out NULL");
  if (!aligned16(out)) return fail(CSA_ERR_INVALID_ARG, "out is not 16-byte aligned");
  if (b->B == 0) { h->last_launches = 0; return CSA_OK; }
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const csa::DevBatch db = dev_batch(b);
  const bool pdl = use_pdl();
  Launches L;
  L.add(staged(h, kStageAttention, st, [&] {
    return run_attention(h, b, db, topk_idx, topk_cnt, out, lse_out, st, pdl, false);
  }));
  return finish(h, L);
}

int csa_decode_step(csa_handle* h, const csa_batch* b, void* out, float* lse_out,
                    int32_t* topk_idx_out, int32_t* topk_cnt_out, void* stream) {
  int rc = validate_batch(h, b);
  if (rc) return rc;
  if (!out) return fail(CSA_ERR_INVALID_ARG, "out is NULL");
  if (!aligned16(out)) return fail(CSA_ERR_INVALID_ARG, "out is not 16-byte aligned");
  if (b->B == 0) { h->last_launches = 0; return CSA_OK; }
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const csa::DevBatch db = dev_batch(b);
  int* idx = topk_idx_out ? topk_idx_out : h->ws.topk_idx;
  int* cnt = topk_cnt_out ? topk_cnt_out : h->ws.topk_cnt;
  const bool pdl = use_pdl();
  // this step's value of the per-query Top-K ready flags (never 0, the value
  // the flags start with)
  h->epoch = h->epoch == 0x7fffffff ? 1 : h->epoch + 1;
  Launches L;
  // Top-K blocks start per request (indexer completion counters) in
  // single-token decode; with more queries per request it measured slower
  // than waiting for the indexer grid (S = 8: 105.2 against 102.4 us per
  // step; a 512-token prefill chunk, hundreds of blocks polling one
  // request's counter: 782 against 437 us)
  int* done = nullptr;
  // the internal scores go to Top-K as order-preserving keys when the
  // register kernel selects (it then skips the conversion)
  bool keyed = false;
  run_indexer(h, b, db, 0, h->ws.scores, h->ws.scores_ld, st, L, b->S <= kCounterMaxS ? &done : nullptr,
              csa::topk_use_reg(h->dc.max_vis), &keyed);
  const bool early = L.n > 0;  // the plan or indexer kernel runs right before
  L.add(staged(h, kStageTopk, st, [&] {
    return csa::launch_topk(h->dc, &db, b->B * b->S, h->ws.scores, h->ws.scores_ld, nullptr, idx,
                            cnt, h->ws.status, h->dc.max_vis, st, pdl, early, h->ws.topk_ready,
                            h->epoch, done, csa::indexer_qsplit(h->dc, b->S), keyed);
  }));
  L.add(staged(h, kStageAttention, st, [&] {
    return run_attention(h, b, db, idx, cnt, out, lse_out, st, pdl, true);
  }));
  return finish(h, L);
}

int csa_indexer_scores(csa_handle* h, const csa_batch* b, float* scores, int64_t ld,
                       int32_t score_all, void* stream) {
  int rc = validate_batch(h, b);
  if (rc) return rc;
  if (!scores) return fail(CSA_ERR_INVALID_ARG, "scores is NULL");
  if (ld < h->dc.max_vis) return fail(CSA_ERR_INVALID_ARG, "ld below max_context / ratio");
  if (b->B == 0) { h->last_launches = 0; return CSA_OK; }
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const csa::DevBatch db = dev_batch(b);
  Launches L;
  run_indexer(h, b, db, score_all ? 1 : 0, scores, ld, st, L);
  return finish(h, L);
}

int csa_topk_select(csa_handle* h, int32_t nq, const float* scores, int64_t ld, const int32_t* n,
                    int32_t* topk_idx, int32_t* topk_cnt, void* stream) {
  if (!h) return fail(CSA_ERR_INVALID_ARG, "handle is NULL");
  if (nq < 0) return fail(CSA_ERR_INVALID_ARG, "nq < 0");
  if (nq == 0) { h->last_launches = 0; return CSA_OK; }
  if (!scores || !n || !topk_idx || !topk_cnt) return fail(CSA_ERR_INVALID_ARG, "NULL pointer");
  if (ld < 1) return fail(CSA_ERR_INVALID_ARG, "ld < 1");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const bool pdl = use_pdl();
  Launches L;
  L.add(staged(h, kStageTopk, st, [&] {
    return csa::launch_topk(h->dc, nullptr, nq, scores, ld, n, topk_idx, topk_cnt, h->ws.status,
                            h->dc.max_vis, st, pdl, false);
  }));
  return finish(h, L);
}

int csa_indexer_topk_static(const csa_config* cfg, const csa_batch* b, int32_t* topk_idx,
                            int32_t* topk_cnt, int32_t* status_out, void* stream) {
  int rc = validate_cfg(cfg);
  if (rc) return rc;
  rc = validate_batch_cfg(*cfg, b);
  if (rc) return rc;
  if (!topk_idx || !topk_cnt) return fail(CSA_ERR_INVALID_ARG, "topk_idx/topk_cnt NULL");
  size_t o_prefix = 0, o_scores = 0;
  const size_t need = static_scratch_need(*cfg, b, &o_prefix, &o_scores);
  if (need > kStaticScratchBytes)
    return fail(CSA_ERR_WORKSPACE,
                "B*S = %d queries x max_context/ratio = %d scores need %zu bytes of scratch, above "
                "the %zu bytes of the allocation-free entry point (use csa_indexer_topk)",
                b->B * b->S, cfg->max_context / cfg->ratio, need, kStaticScratchBytes);
  // set-up, once per context (normally once per device), with the device
  // current: the scratch array's address and the SM count
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  unsigned long long ctx = 0;
  void* looked_up = nullptr;
  if (!current_context_id(&ctx)) {
    // no context is current on this thread yet: the lookup, a runtime call
    // that needs one, makes the device's primary context current
    e = cudaGetSymbolAddress(&looked_up, g_static_scratch);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(static scratch)");
    if (!current_context_id(&ctx))
      return fail(CSA_ERR_CUDA, "no current CUDA context (cuCtxGetCurrent / cuCtxGetId)");
  }
  void* base = nullptr;
  int sms = 0;
  {
    std::lock_guard<std::mutex> lock(g_static_mu);
    int k = 0;
    while (k < g_static_nslots && g_static_slots[k].ctx_id != ctx) ++k;
    if (k == g_static_nslots) {
      if (k == kMaxStaticContexts)
        return fail(CSA_ERR_UNSUPPORTED, "more than %d CUDA contexts used the allocation-free entry point",
                    kMaxStaticContexts);
      void* a = looked_up;
      if (!a) {
        e = cudaGetSymbolAddress(&a, g_static_scratch);
        if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(static scratch)");
      }
      int n = 0;
      e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
      if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute");
      g_static_slots[k] = StaticSlot{ctx, a, n};
      g_static_nslots = k + 1;
    }
    base = g_static_slots[k].addr;
    sms = g_static_slots[k].sms;
  }
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (b->B == 0) {  // nothing to select: the status reads clean
    if (status_out) {
      e = cudaMemsetAsync(status_out, 0, sizeof(int32_t), st);
      if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync(status_out)");
    }
    return CSA_OK;
  }
  char* sb = static_cast<char*>(base);
  // a handle on the stack that borrows the static scratch: the same launch
  // sequence as csa_indexer_topk, with no workspace of its own
  csa_handle h;
  h.cfg = *cfg;
  h.dc = static_devcfg(*cfg);
  h.ws_base = nullptr;
  h.ws_bytes = 0;
  h.device = dev;
  h.num_sms = sms;
  h.last_launches = 0;
  csa::Workspace& w = h.ws;
  w.status = reinterpret_cast<int*>(sb);
  w.item_prefix = reinterpret_cast<int*>(sb + o_prefix);
  w.scores = reinterpret_cast<float*>(sb + o_scores);
  w.topk_idx = nullptr;
  w.topk_cnt = nullptr;
  w.job_prefix = nullptr;
  w.topk_ready = nullptr;
  w.part_o = nullptr;
  w.part_lse = nullptr;
  w.seg_ready = nullptr;
  w.idx_done = nullptr;
  w.max_T = b->B * b->S;
  w.max_batch = b->B;
  w.scores_ld = h.dc.max_vis > 0 ? h.dc.max_vis : 1;
  // the status word must read zero when the kernels start; the work list and
  // the scores are fully written before they are read
  e = cudaMemsetAsync(w.status, 0, sizeof(int), st);
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync(status)");
  const csa::DevBatch db = dev_batch(b);
  const bool pdl = use_pdl();
  Launches L;
  run_indexer(&h, b, db, 0, w.scores, w.scores_ld, st, L);
  const bool early = L.n > 0;  // the plan or indexer kernel runs right before
  L.add(csa::launch_topk(h.dc, &db, b->B * b->S, w.scores, w.scores_ld, nullptr, topk_idx, topk_cnt,
                         w.status, h.dc.max_vis, st, pdl, early));
  rc = finish(&h, L);
  if (rc) return rc;
  if (status_out) {
    e = cudaMemcpyAsync(status_out, w.status, sizeof(int), cudaMemcpyDeviceToDevice, st);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpyAsync(status)");
  }
  return CSA_OK;
}

int csa_cache_writeback(const void* rows, int64_t rows_stride, const int64_t* slot, int32_t n,
                        void* pool, int64_t pool_stride, int64_t pool_rows, int64_t row_bytes,
                        int32_t* status, void* stream) {
  if (n < 0) return fail(CSA_ERR_INVALID_ARG, "n < 0");
  if (row_bytes < 0 || pool_rows < 0) return fail(CSA_ERR_INVALID_ARG, "negative row_bytes or pool_rows");
  if (n == 0 || row_bytes == 0) { g_err.clear(); return CSA_OK; }
  if (!rows || !slot || !pool) return fail(CSA_ERR_INVALID_ARG, "rows/slot/pool NULL");
  if (rows_stride < row_bytes || pool_stride < row_bytes)
    return fail(CSA_ERR_INVALID_ARG, "a stride below row_bytes");
  if (csa::launch_writeback(rows, rows_stride, slot, n, pool, pool_stride, pool_rows, row_bytes,
                            status, static_cast<cudaStream_t>(stream), false) < 0) {
    std::string why;
    why.swap(g_launch_why);
    return fail(CSA_ERR_CUDA, "kernel launch: %s", why.empty() ? "failed" : why.c_str());
  }
  g_err.clear();
  return CSA_OK;
}

int csa_debug_set_wait_polls(csa_handle* h, int32_t polls) {
  if (!h) return fail(CSA_ERR_INVALID_ARG, "handle is NULL");
  h->dc.wait_polls = polls < 0 ? -1 : polls;
  return CSA_OK;
}

int csa_profile_enable(csa_handle* h, int32_t enable) {
  if (!h) return fail(CSA_ERR_INVALID_ARG, "handle is NULL");
  h->prof = enable != 0;
  return CSA_OK;
}

int csa_profile_read(csa_handle* h, float* ms, int32_t* launches) {
  if (!h || !ms || !launches) return fail(CSA_ERR_INVALID_ARG, "NULL argument");
  for (int i = 0; i < kStages; ++i) { ms[i] = 0.f; launches[i] = 0; }
  for (auto& m : h->marks) {
    cudaError_t e = cudaEventSynchronize(m.b);
    if (e != cudaSuccess) return cuda_fail(e, "cudaEventSynchronize");
    float t = 0.f;
    e = cudaEventElapsedTime(&t, m.a, m.b);
    if (e != cudaSuccess) return cuda_fail(e, "cudaEventElapsedTime");
    ms[m.stage] += t;
    launches[m.stage] += 1;
    h->spare.push_back(m.a);
    h->spare.push_back(m.b);
  }
  h->marks.clear();
  return CSA_OK;
}

int csa_check_batch(const csa_config* cfg, const csa_batch* b) {
  int rc = validate_cfg(cfg);
  if (rc) return rc;
  return validate_batch_cfg(*cfg, b);
}

int csa_get_status(csa_handle* h, void* stream) {
  if (!h) return fail(CSA_ERR_INVALID_ARG, "handle is NULL");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  int v = 0;
  e = cudaMemcpy(&v, h->ws.status, sizeof(int), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpy(status)");
  e = cudaMemset(h->ws.status, 0, sizeof(int));
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemset(status)");
  if (v & csa::kStatusTimeout) return fail(CSA_ERR_TIMEOUT, "a device wait gave up");
  if (v & csa::kStatusBadIndex)
    return fail(CSA_ERR_BAD_INDEX, "a length or row index in device memory was out of range");
  return CSA_OK;
}

}  // extern "C"
