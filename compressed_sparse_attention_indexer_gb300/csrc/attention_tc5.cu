// Steps (c) + (d) on the fifth-generation tensor cores, in two kernels.
//
// hw-native-sys/pypto-lib:
//  - "Fix: port the DeepSeek-V4 MoE, hc_pre and prefill fixes to DSpark", PR
//    description: a query reads at most WIN + min(max_visible_cmp, IDX_TOPK)
//    sparse rows;
//  - "Perf: skip redundant CSA scoring and fuse gather unpack", PR
//    description: gathered rows go straight into their consumer;
//  - "Perf: fuse HCA merge, inverse RoPE, and packing", PR description: raw
//    and compressed softmax results are merged, then inverse RoPE is applied.
//
// attn_tile_kernel: persistent, one CTA per SM, warp-specialised.  A job is
// one 64-row tile of one stream (window, compressed, heavy) of one query; a
// CTA takes a contiguous range of the job list (the CTAs that start beside
// the Top-K blocks take more), and the jobs of one query inside that range
// form a segment whose output accumulates in TMEM.
//   warps 5-10, two groups of three: group g gathers every other job into
//            job buffer g with coalesced 16-byte cp.async, rows scattered
//            over the pools, into nine 128-byte-swizzled 64-dim sub-tiles
//            (72 KB); each thread fences its copies for the async proxy and
//            arrives on the buffer's barrier.  Two buffers: one job's rows
//            land while the previous job is computed, and the next job's
//            rows are asked of L2 while its buffer is still busy.  In a
//            decode step a query's compressed tiles start once its Top-K
//            block has published its output (a per-query flag);
//   warp 4   loads the query's 64 heads x 576 (72 KB, TMA) when the query
//            changes and issues the tcgen05 MMAs as their inputs become
//            ready: S[64 heads x 64 rows] = Q . R^T over 576 dims (M = 64,
//            N = 64) into one of two TMEM score buffers; after the softmax,
//            O^T[512 dims x 64 heads] += V^T . P^T (M = 128 per 128-dim
//            chunk, N = 64; V read in place as an MN-major operand, P^T
//            from the rope sub-tile that QK no longer needs) into TMEM;
//   warps 0-3 softmax, two threads per head (lanes i and i + 16 of warp w:
//            head 16w + i, which the M = 64 layout puts in TMEM lane
//            32w + i; rows 0-31 and 32-63): scale and mask the job's scores,
//            keep a per-head reference max that moves only when a tile max
//            exceeds it by 2^8 (then O^T is rescaled in TMEM by all 128
//            threads), write the head's row of P^T as bf16 and sum the
//            rounded weights.  At a segment's end all four warps read O^T
//            (thread = dim), write the normalised partial output (bf16,
//            heads x dims) and the heads' log-sum-exp to the workspace, and
//            publish the segment (a per-segment flag).
// attn_merge_kernel: per query and 64 output dims, the log-sum-exp merge of
// the query's segments in job order, inverse RoPE on the last R dims, the
// bf16 store; after a tile kernel launched just before it, a block starts as
// soon as its query's segments are published.  Because the merge is exact,
// segment softmax + merge equals one softmax over the union of the streams'
// rows.
#include <cudaTypedefs.h>
#include <stddef.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "csa_internal.cuh"
#include "tc5.cuh"

namespace csa {

namespace {

constexpr int kLoadWarps = 3;              // per row-loader group
constexpr int kA5Threads = 32 * (5 + 2 * kLoadWarps);  // warps 0-3 softmax, 4 MMA + Q, 5-10 row loaders
constexpr int kTile = 64;                  // rows per job
constexpr int kQuadsPerWarp = (kTile / 4 + kLoadWarps - 1) / kLoadWarps;
constexpr int kNSub = 9;                   // 64-dim sub-tiles of a 576-wide row
constexpr int kSub = kTile * 128;          // 64 rows x 64 dims bf16: 8 KB
constexpr int kBuf = kNSub * kSub;         // a job's rows: 72 KB (rope sub-tile -> P^T)
constexpr int kQSub = kTcH * 128;          // 64 heads x 64 dims: 8 KB
constexpr int kQBytes = 9 * kQSub;         // the query's heads, resident: 72 KB
constexpr int kA5Dyn = 1024 + kQBytes + 2 * kBuf;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRescale = 8.f;            // lazy rescale threshold (log2 units)
constexpr int kMergeDims = 64;             // output dims per merge block
constexpr int kMergeMaxJobs = 64;          // jobs per query the merge handles (else the warp-MMA path)
// TMEM columns: two score buffers (M = 64 layout: head h in lane
// 32(h / 16) + h % 16, row j in column j), four 128-dim chunks of O^T
constexpr uint32_t kTmemS = 0, kTmemO = 256;

struct __align__(16) A5Smem {
  // per job buffer: its rows have landed / the MMAs that read them are done
  uint64_t full[2], empty[2];
  uint64_t mfull[2], mempty[2], s_full[2], s_empty[2];
  // p_full per job buffer: with one barrier the softmax could complete two
  // jobs' phases before the MMA thread polls the first, and a parity wait
  // cannot tell phase n from phase n + 2; per buffer, job n + 2's phase needs
  // job n's PV first
  uint64_t p_full[2];
  uint64_t pv_done, o_full, o_empty, qfull, qdone, done;
  uint32_t tmem_base;
  int abort;
  // per job parity and softmax warp: bit 0 some head needs a rescale, bit 1
  // the warp saw a wait give up (every softmax thread then leaves together)
  int flag[2][4];
  uint64_t mask[2][kLoadWarps];    // per buffer and loader warp: bit i = row i of the job exists
  alignas(16) float alpha[2][kTcH];  // per job parity: per-head rescale factor
  alignas(16) float linv[2][kTcH];   // per segment parity: per-head 1 / (sum of the weights)
};
static_assert(offsetof(A5Smem, alpha) % 16 == 0 && offsetof(A5Smem, linv) % 16 == 0,
              "per-head statistics are read with 16-byte loads");

// descriptor of an MN-major operand in the 128-byte swizzle layout: 64
// contiguous MN elements per 128-byte row, 8-row K groups 1024 bytes apart
// (SBO), the next 64 MN elements `lbo` bytes further (LBO)
__device__ __forceinline__ uint64_t sdesc_mn_sw128(uint32_t saddr, uint32_t lbo) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)(1024u >> 4) << 32;
  d |= (uint64_t)1u << 46;
  d |= (uint64_t)2u << 61;
  return d;
}

// 2^x with the hardware approximation (relative error ~2^-22; -inf -> 0),
// ample for weights that are rounded to bf16 next.  The argument is never
// NaN here: a masked score is -inf and the reference is finite whenever a
// row exists.
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
}

// Coherent global loads of values another running kernel writes (never the
// read-only path), and the acquire load of a flag.
__device__ __forceinline__ int ld_cg(const int* p) {
  int v;
  asm volatile("ld.global.cg.b32 %0, [%1];\n" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ int ld_acquire(const int* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];\n" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// One job list (see JobLists): jobs of query q are [prefix[q], prefix[q+1]).
struct JobCursor {
  const int* prefix;
  int q, first, end;
  // q0 >= 0: the query holding `job`, known already (span: its job range
  // [p[q0], p[q0 + 1]), if known too); else found by search
  __device__ __forceinline__ void init(const int* p, int T, int job, int q0, const int* span) {
    prefix = p;
    int l = q0;
    if (l < 0) {
      l = 0;
      int r = T - 1;
      while (l < r) {
        const int m = (l + r + 1) >> 1;
        if (p[m] <= job) l = m; else r = m - 1;
      }
    }
    q = l;
    first = span ? span[0] : p[l];
    end = span ? span[1] : p[l + 1];
  }
  __device__ __forceinline__ void advance(int job) {
    while (job >= end) {
      ++q;
      first = end;
      end = prefix[q + 1];
    }
  }
};

// The split of the two job lists over the tile CTAs.  CTA i takes the W jobs
// [wstart(i), wstart(i+1)), spread over the first E CTAs (the ones that start
// while the Top-K kernel still runs), then the C jobs [cstart(i),
// cstart(i+1)), spread over all G (c_list_start: evenly with the left-over
// jobs on the first E CTAs, or by weights).  Job ids: W jobs
// 0 .. NW-1, C jobs NW .. NW+NC-1; a segment's partial output sits at the id
// of its first job.
struct Sched {
  const int* wp;
  const int* cp;
  const uint16_t* cq;  // per-CTA first queries (cta_q of the lists) or null
  const int* cspan;    // their job ranges (cta_span of the lists), with cq
  int T, NW, NC, G, E;
  int CE, wa, wb;      // C-list weights (see JobLists)
  __device__ __forceinline__ int wstart(int i) const {
    return i >= E ? NW : (int)((int64_t)i * NW / E);
  }
  __device__ __forceinline__ int cstart(int i) const { return c_list_start(i, NC, G, CE, wa, wb); }
  __device__ __forceinline__ void weights(const JobLists& jobs) {
    const bool w = jobs.host_T >= 0 && jobs.cw_early > 0 && (jobs.cw_a == 0 || (jobs.cw_a > 0 && jobs.cw_b > 0));
    CE = w ? jobs.cw_early : G;
    wa = w ? jobs.cw_a : 1;
    wb = w ? jobs.cw_b : 1;
  }
};

// A job of a CTA's sequence: its query, list (0 = W, 1 = C), index within
// the query's jobs of that list, id, and whether it opens / closes a segment
// (the CTA's consecutive jobs of one query in one list).
struct JobRef {
  int q, list, local, gid;
  bool first, last;
};

// Walks a CTA's jobs in order (n increasing; the same n may be asked again).
struct JobWalk {
  JobCursor wc, cc;
  int nw, nc, wlo, clo, NW;
  __device__ __forceinline__ void init(const Sched& s, int cta) {
    wlo = s.wstart(cta);
    nw = s.wstart(cta + 1) - wlo;
    clo = s.cstart(cta);
    nc = s.cstart(cta + 1) - clo;
    NW = s.NW;
    if (nw > 0)
      wc.init(s.wp, s.T, wlo, s.cq ? (int)s.cq[cta] : -1, s.cq ? s.cspan + 2 * cta : nullptr);
    if (nc > 0)
      cc.init(s.cp, s.T, clo, s.cq ? (int)s.cq[kMaxTileCtas + cta] : -1,
              s.cq ? s.cspan + 2 * (kMaxTileCtas + cta) : nullptr);
  }
  __device__ __forceinline__ JobRef get(int n) {
    JobRef r;
    if (n < nw) {
      const int idx = wlo + n;
      wc.advance(idx);
      r.q = wc.q;
      r.list = 0;
      r.local = idx - wc.first;
      r.gid = idx;
      r.first = n == 0 || idx == wc.first;
      r.last = n == nw - 1 || idx + 1 == wc.end;
    } else {
      const int m = n - nw, idx = clo + m;
      cc.advance(idx);
      r.q = cc.q;
      r.list = 1;
      r.local = idx - cc.first;
      r.gid = NW + idx;
      r.first = m == 0 || idx == cc.first;
      r.last = m == nc - 1 || idx + 1 == cc.end;
    }
    return r;
  }
};

// The job's query plan and its three stream lengths (bound on the compressed
// count from the Top-K count the attention kernel reads).
struct JobCtx {
  QueryPlan p;
  int bi;
  int n[3];
  int nt[3];
};

// The job's query plan and its stream lengths, from the caller's inputs
// only; the compressed count (a Top-K output) is filled in by job_topk_cnt.
__device__ __forceinline__ JobCtx job_ctx(const DevCfg& c, const DevBatch& b, int q, int len) {
  JobCtx x;
  x.bi = q / b.S;
  x.p = query_plan(c, b.S, len, q - x.bi * b.S, 0);
  x.n[0] = x.p.nwin;
  x.n[1] = 0;
  x.n[2] = x.p.vis2;
  // tiles per stream from the bound min(vis, K), as the job list counts them
  x.nt[0] = (x.p.nwin + kTile - 1) / kTile;
  x.nt[1] = (x.p.cnt + kTile - 1) / kTile;
  x.nt[2] = (x.p.vis2 + kTile - 1) / kTile;
  return x;
}

// The compressed stream's length: the Top-K count, bounded by min(vis, K).
__device__ __forceinline__ void job_topk_cnt(JobCtx& x, int q, const int* topk_cnt) {
  int cnt = 0;
  if (!(x.p.flags & kPlanBad)) {
    cnt = ld_cg(topk_cnt + q);
    cnt = cnt < 0 ? 0 : (cnt > x.p.cnt ? x.p.cnt : cnt);
  }
  x.n[1] = cnt;
}

// The stream and tile of a job (see JobLists): with the split, W jobs are
// the window tiles, then the heavy tiles, and C jobs the compressed tiles;
// without it a query's jobs are its window, compressed, then heavy tiles.
__device__ __forceinline__ void job_stream(const JobCtx& x, const JobRef& r, bool split, int& sid,
                                           int& t) {
  if (split && r.list == 1) { sid = 1; t = r.local; }
  else if (r.local < x.nt[0]) { sid = 0; t = r.local; }
  else if (!split && r.local < x.nt[0] + x.nt[1]) { sid = 1; t = r.local - x.nt[0]; }
  else { sid = 2; t = r.local - x.nt[0] - (split ? 0 : x.nt[1]); }
}


// Pool row of stream row i of the job, or -1 (read as zeros by the gather and
// masked by the softmax) when the row does not exist or is out of range.
// `j` is the row's Top-K index for the compressed stream (loaded by the
// caller ahead of the count it is checked against).  `off` is the request's
// first pool row of the stream, or -1 when that pool is paged (then the
// pool's block table gives the row).
template <bool kPaged>
__device__ __forceinline__ int job_row(const DevBatch& b, const JobCtx& x, int sid, int i, int j,
                                       int64_t off, int* status) {
  if (i >= x.n[sid]) return -1;
  int64_t gr;
  int64_t rows;
  if (sid == 0) {
    const int64_t r = x.p.pos - x.p.nwin + 1 + i;
    gr = (kPaged && b.raw_table) ? raw_row(b, x.bi, r) : off + r;
    rows = b.raw_rows;
  } else if (sid == 1) {
    if (j < 0 || j >= x.p.vis) {
      set_status(status, kStatusBadIndex);
      return -1;
    }
    gr = (kPaged && b.cmp_table) ? cmp_row(b, x.bi, j) : off + j;
    rows = b.cmp_rows;
  } else {
    gr = (kPaged && b.hca_table) ? hca_row(b, x.bi, i) : off + i;
    rows = b.hca_rows;
  }
  if (gr < 0 || gr >= rows) {
    set_status(status, kStatusBadIndex);
    return -1;
  }
  return (int)gr;
}

// kPaged: some pool has a block table (else every pool is contiguous and the
// row lookups are one add)
template <bool kPaged>
__global__ void __launch_bounds__(kA5Threads, 1)
    attn_tile_kernel(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ JobLists jobs,
                     DevCfg c, DevBatch b, Workspace ws, const int* topk_idx, const int* topk_cnt,
                     int early, int epoch, int seg_epoch) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  __shared__ A5Smem sm;
  const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
  const uint32_t qres = base;                 // 72 KB: the query's 64 heads
  const uint32_t bufs = qres + kQBytes;       // 2 x 72 KB: the jobs' rows
  uint8_t* gen = smem_raw + (bufs - smem_u32(smem_raw));

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int T = b.B * b.S;
  // Launched right after this library's Top-K kernel of the same step with
  // host-built job lists (flags = early != 0), every input but the Top-K
  // outputs was complete before the step's first kernel passed its own wait,
  // so nothing waits for the previous grid up front: setup, Q and the W jobs
  // overlap the Top-K kernel, and a query's C jobs start once that query's
  // Top-K block has published its output (ws.topk_ready[q] == epoch).
  // Otherwise (a caller's kernel before this one, or job lists built on the
  // device) every thread waits for the previous grid first.
  const bool flags = early && jobs.host_T >= 0;
  if (!flags) pdl_wait();
  Sched sc;
  sc.wp = jobs.host_T >= 0 ? jobs.wprefix : ws.job_prefix;
  sc.cp = jobs.host_T >= 0 ? jobs.cprefix : ws.job_prefix + (T + 1);
  sc.cq = jobs.host_T >= 0 && jobs.cta_first ? &jobs.cta_q[0][0] : nullptr;
  sc.cspan = &jobs.cta_span[0][0][0];
  sc.T = T;
  sc.NW = jobs.host_T >= 0 ? jobs.NW : sc.wp[T];
  sc.NC = jobs.host_T >= 0 ? jobs.NC : sc.cp[T];
  sc.G = gridDim.x;
  sc.E = (jobs.host_T >= 0 && jobs.early > 0 && jobs.early < (int)gridDim.x) ? jobs.early : (int)gridDim.x;
  sc.weights(jobs);
  const int J = (sc.wstart(blockIdx.x + 1) - sc.wstart(blockIdx.x)) +
                (sc.cstart(blockIdx.x + 1) - sc.cstart(blockIdx.x));
  pdl_trigger();
  if (J == 0) {
    if (flags) pdl_wait();  // this grid completes after its predecessor
    return;
  }
  volatile int* abort = &sm.abort;
  // polls before a consumer wait gives up (the default: about a second)
  const uint32_t wpolls = c.wait_polls < 0 ? tc5::kBackoffPolls : (uint32_t)c.wait_polls;

  // every role walks the CTA's jobs from the same start; its first query and
  // job range (host lists: kernel parameters of this CTA) load alongside the
  // set-up below
  JobWalk walk0;
  walk0.init(sc, blockIdx.x);

  if (warp == 4) {
    tc5::tmem_alloc(smem_u32(&sm.tmem_base), 512);
    tc5::tmem_relinquish();
  }
  if (tid == 0) {
    for (int g = 0; g < 2; ++g) {
      tc5::mbar_init(smem_u32(&sm.full[g]), kLoadWarps);  // one arrival per loader warp
      tc5::mbar_init(smem_u32(&sm.empty[g]), 1);          // an MMA commit
      tc5::mbar_init(smem_u32(&sm.mfull[g]), kLoadWarps);  // one arrival per loader warp
      tc5::mbar_init(smem_u32(&sm.mempty[g]), 128);  // the softmax threads
      tc5::mbar_init(smem_u32(&sm.s_full[g]), 1);
      tc5::mbar_init(smem_u32(&sm.s_empty[g]), 128);
      tc5::mbar_init(smem_u32(&sm.p_full[g]), 128);
    }
    tc5::mbar_init(smem_u32(&sm.pv_done), 1);
    tc5::mbar_init(smem_u32(&sm.o_full), 1);
    tc5::mbar_init(smem_u32(&sm.o_empty), 128);
    tc5::mbar_init(smem_u32(&sm.qfull), 1);
    tc5::mbar_init(smem_u32(&sm.qdone), 1);
    tc5::mbar_init(smem_u32(&sm.done), 1);
    sm.abort = 0;
    tc5::fence_mbar_init();
  }
  tc5::fence_before_sync();
  __syncthreads();
  tc5::fence_after_sync();
  const uint32_t tmem = sm.tmem_base;

  if (warp >= 5) {
    // ------------------------------------------------------------ row loaders
    // Group g (three warps) takes jobs lo+g, lo+g+2, ... into job buffer g.
    // Lane l of a warp moves 16-byte chunk l & 7 of row quads lw, lw+3, ...
    // (rows 4 quad + l / 8), with cp.async into the 128-byte swizzled
    // sub-tiles; a row that does not exist (or is out of range) reads zeros.
    // Once the buffer's previous job has released it, the whole job is in
    // flight at once; each thread then waits for its copies and fences them
    // for the async proxy, and one lane per warp arrives on the buffer's
    // barrier.
    const int g = (warp - 5) / kLoadWarps, lw = (warp - 5) % kLoadWarps;
    const uint32_t buf = bufs + g * kBuf;
    const __nv_bfloat16* null_src = static_cast<const __nv_bfloat16*>(b.q);
    const int ch = lane & 7;
    const uint64_t rpol = tc5::policy_evict_first();  // rows are read once per step
    JobWalk walk = walk0;
    int m = 0;
    bool waited = !flags;
    for (int n = g; n < J; n += 2, ++m) {
      if (__shfl_sync(0xffffffffu, *abort, 0)) break;
      const JobRef r = walk.get(n);
      const int q = r.q, bi = q / b.S;
      const bool split = jobs.host_T >= 0 && jobs.split;
      // the job's independent loads go out together: the request's length,
      // its pool offsets and (unless the job is a W job) the first poll of
      // the query's Top-K flag
      const int len = b.ctx_len[bi];
      const int64_t o_raw = (kPaged && b.raw_table) ? -1 : b.raw_off[bi];
      const int64_t o_cmp = (kPaged && b.cmp_table) ? -1 : b.cmp_off[bi];
      const int64_t o_hca = (!b.hca || (kPaged && b.hca_table)) ? -1 : b.hca_off[bi];
      int flag0 = epoch;
      if (flags && lane == 0 && !(split && r.list == 0)) flag0 = ld_acquire(ws.topk_ready + q);
      JobCtx x = job_ctx(c, b, q, len);
      int sid, t;
      job_stream(x, r, split, sid, t);
      const __nv_bfloat16* pool = static_cast<const __nv_bfloat16*>(
          sid == 0 ? b.raw : (sid == 1 ? b.cmp : b.hca));
      const int64_t stride = sid == 0 ? b.raw_stride : (sid == 1 ? b.cmp_stride : b.hca_stride);
      const int64_t off = sid == 0 ? o_raw : (sid == 1 ? o_cmp : o_hca);
      // this lane's rows: their Top-K indices are loaded together with the
      // count they are checked against
      int jr[kQuadsPerWarp];
#pragma unroll
      for (int i = 0; i < kQuadsPerWarp; ++i) jr[i] = -1;
      if (sid == 1) {
        if (flags) {
          // this query's Top-K output: lane 0 acquires its flag (the first
          // poll above, then bounded polls), and the warp barrier below
          // orders that before every lane's reads of the output
          bool ok = true;
          if (lane == 0 && flag0 != epoch) {
            uint32_t ns = 32;
            uint32_t i = 0;
            while (ld_acquire(ws.topk_ready + q) != epoch) {
              if (++i >= wpolls || (((i & 15u) == 15u) && *abort)) {
                *abort = 1;
                ok = false;
                break;
              }
              if (i >= 8) {
                __nanosleep(ns);
                ns = ns * 2 > 256 ? 256 : ns * 2;
              }
            }
          }
          if (!__shfl_sync(0xffffffffu, ok, 0)) break;
          __syncwarp();
        } else if (!waited) {
          pdl_wait();
          waited = true;
        }
#pragma unroll
        for (int i = 0; i < kQuadsPerWarp; ++i) {
          const int rq = lw + kLoadWarps * i;
          const int ri = t * kTile + 4 * rq + (lane >> 3);
          if (rq < kTile / 4 && ri < c.K) jr[i] = ld_cg(topk_idx + (int64_t)q * c.K + ri);
        }
        job_topk_cnt(x, q, topk_cnt);
      }
      const __nv_bfloat16* src[kQuadsPerWarp];
      uint64_t bits = 0;
#pragma unroll
      for (int i = 0; i < kQuadsPerWarp; ++i) {
        const int rq = lw + kLoadWarps * i;
        src[i] = nullptr;
        if (rq < kTile / 4) {
          const int gr = job_row<kPaged>(b, x, sid, t * kTile + 4 * rq + (lane >> 3), jr[i], off, ws.status);
          if (gr >= 0) src[i] = pool + (int64_t)gr * stride;
        }
        const uint32_t v = __ballot_sync(0xffffffffu, src[i] != nullptr);
#pragma unroll
        for (int k = 0; k < 4; ++k)
          if ((v >> (8 * k)) & 1u) bits |= 1ull << (4 * rq + k);
      }
      // while the buffer's previous job is still being consumed, ask L2 for
      // this job's rows (lane l of a row: its 128-byte line l, and line 8 by
      // lane 0), so the copies below hit L2
      if (m >= 1) {
#pragma unroll
        for (int i = 0; i < kQuadsPerWarp; ++i)
          if (src[i]) {
            const char* row = reinterpret_cast<const char*>(src[i]);
            prefetch_l2_line(row + ch * 128);
            if (ch == 0) prefetch_l2_line(row + 8 * 128);
          }
      }
      bool ok = true;
      if (lane == 0) {
        if (m >= 1 && !tc5::mbar_wait_backoff(smem_u32(&sm.mempty[g]), (m - 1) & 1, abort, 256, wpolls))
          ok = false;
        if (ok) {
          sm.mask[g][lw] = bits;
          tc5::mbar_arrive(smem_u32(&sm.mfull[g]));
        }
      }
      if (!__shfl_sync(0xffffffffu, ok, 0)) break;
      if (lane == 0 && m >= 1 &&
          !tc5::mbar_wait_backoff(smem_u32(&sm.empty[g]), (m - 1) & 1, abort, 256, wpolls))
        ok = false;
      if (!__shfl_sync(0xffffffffu, ok, 0)) break;
#pragma unroll 3
      for (int k = 0; k < kNSub; ++k) {
#pragma unroll
        for (int i = 0; i < kQuadsPerWarp; ++i) {
          const int rq = lw + kLoadWarps * i;
          if (rq < kTile / 4) {
            const int rt = 4 * rq + (lane >> 3);  // row within the job
            const uint32_t dst = buf + k * kSub + rt * 128 + ((ch ^ (rt & 7)) << 4);
            cp_async16_hint(dst, src[i] ? (const void*)(src[i] + k * 64 + ch * 8) : (const void*)null_src,
                            src[i] ? 16 : 0, rpol);
          }
        }
      }
      cp_async_commit();
      cp_async_wait<0>();
      fence_proxy_async();
      __syncwarp();
      if (lane == 0) tc5::mbar_arrive(smem_u32(&sm.full[g]));
    }
    cp_async_wait<0>();
  } else if (warp == 4) {
    // ------------------------------------------------------------ Q loads + MMA issue
    // Event driven: each poll issues whichever of QK(next) and PV(oldest
    // pending) is ready, so that a job's PV never waits behind the next
    // job's rows.  Descriptors advance by (byte offset >> 4) from bases.
    if (lane == 0) {
      tc5::prefetch_tmap(&qmap);
      const uint32_t idesc_s = tc5::idesc_bf16_f32(64, 64);                // QK: 64 heads x 64 rows
      const uint32_t idesc_o = tc5::idesc_bf16_f32(128, kTcH) | (1u << 15);  // PV: A MN-major
      const uint64_t dq = tc5::sdesc_k_sw128(qres);
      const uint64_t dbuf = tc5::sdesc_k_sw128(bufs);
      const uint64_t dv = sdesc_mn_sw128(bufs, kSub);
      JobWalk qw = walk0, pw = walk0;  // the next QK job and the next PV job
      int nk = 0, np = 0;  // CTA-local index of the next job to QK / to PV
      int nq = 0, nqd = 0, seg = 0;
      int qseg = -1;       // first job of the segment whose Q is resident (or loading)
      int kseg = 0;        // first job of nk's segment
      int qstate = 0;      // 0 Q of qseg resident, 1 waiting for qdone, 2 waiting for qfull
      uint32_t idle = 0;
      while (np < J) {
        bool progressed = false;
        if (np < nk) {
          const JobRef r = pw.get(np);
          const bool first = r.first, last = r.last;
          const int g = np & 1;
          if ((!first || seg == 0 || tc5::mbar_try_wait(smem_u32(&sm.o_empty), (seg - 1) & 1)) &&
              tc5::mbar_try_wait(smem_u32(&sm.p_full[g]), (np >> 1) & 1)) {
            // O^T += V^T . P^T (overwrite at a segment's first job)
            tc5::fence_after_sync();
            const uint32_t vo = (g * kBuf) >> 4;                  // buffer offset, 16-byte units
            const uint64_t dp = dbuf + vo + ((8 * kSub) >> 4);    // P^T in the rope sub-tile
#pragma unroll
            for (int cc = 0; cc < 4; ++cc)
#pragma unroll
              for (int i = 0; i < 4; ++i)
                tc5::mma_bf16(tmem + kTmemO + 64 * cc, dv + vo + ((2 * cc * kSub + i * 2048) >> 4),
                              dp + 2 * i, idesc_o, (!first || i > 0) ? 1u : 0u);
            tc5::mma_commit(smem_u32(&sm.empty[g]));
            tc5::mma_commit(smem_u32(&sm.pv_done));
            if (last) {
              tc5::mma_commit(smem_u32(&sm.o_full));
              ++seg;
            }
            ++np;
            progressed = true;
          }
        }
        if (nk < J) {
          const JobRef r = qw.get(nk);
          if (r.first) kseg = nk;
          if (kseg != qseg) {
            // a new segment: its query's heads replace Q once the QK MMAs of
            // the previous segment are done (qdone)
            if (qstate == 0) qstate = nk == 0 ? 3 : 1;
            if (qstate == 1 && tc5::mbar_try_wait(smem_u32(&sm.qdone), nqd & 1)) {
              ++nqd;
              qstate = 3;
            }
            if (qstate == 3) {
              tc5::mbar_expect_tx(smem_u32(&sm.qfull), kQBytes);
              for (int k = 0; k < 9; ++k)
                tc5::tma_load_2d(qres + k * kQSub, &qmap, k * 64, r.q * kTcH, smem_u32(&sm.qfull));
              qstate = 2;
            }
            if (qstate == 2 && tc5::mbar_try_wait(smem_u32(&sm.qfull), nq & 1)) {
              ++nq;
              qstate = 0;
              qseg = kseg;
            }
          }
          const int g = nk & 1, m = nk >> 1;
          if (kseg == qseg && (m == 0 || tc5::mbar_try_wait(smem_u32(&sm.s_empty[g]), (m - 1) & 1)) &&
              tc5::mbar_try_wait(smem_u32(&sm.full[g]), m & 1)) {
            // S = Q . R^T over 576 dims (M = 64 heads, N = 64 rows).  (Issued
            // whole: issuing it in pieces with a ready PV between them was
            // measured slower.)
            tc5::fence_after_sync();
            const uint64_t db = dbuf + ((g * kBuf) >> 4);
            const uint32_t ds = tmem + kTmemS + 64 * g;
#pragma unroll
            for (int k = 0; k < kNSub; ++k)
#pragma unroll
              for (int i = 0; i < 4; ++i)
                tc5::mma_bf16(ds, dq + ((k * kQSub + 32 * i) >> 4), db + ((k * kSub + 32 * i) >> 4),
                              idesc_s, (k | i) ? 1u : 0u);
            tc5::mma_commit(smem_u32(&sm.s_full[g]));
            // Q is reloaded at every segment start: its last QK frees it
            if (r.last && nk + 1 < J) tc5::mma_commit(smem_u32(&sm.qdone));
            ++nk;
            progressed = true;
          }
        }
        if (progressed) {
          idle = 0;
        } else {
          if (++idle > (1u << 25)) {
            *abort = 1;
            break;
          }
          if (idle > 8) __nanosleep(32);
          if ((idle & 63u) == 0 && *abort) break;
        }
      }
      if (qstate == 2) tc5::mbar_wait_drain(smem_u32(&sm.qfull), nq & 1);
      tc5::mma_commit(smem_u32(&sm.done));
      tc5::mbar_wait_drain(smem_u32(&sm.done), 0);
    }
  } else {
    // ------------------------------------------------------------ softmax + epilogue
    // Two threads per head: lanes i and i + 16 of warp w own head h = 16w + i
    // (its TMEM lane in the M = 64 score layout), rows 0-31 and 32-63 of the
    // job respectively; the reference max and the sum of the weights are
    // shared by the pair (one shuffle each) and kept identically in both.
    // The four warps meet once per job at a named barrier; a thread whose
    // wait gave up skips its work but still reaches the barrier, and the
    // flags read after it make every softmax thread leave at the same job.
    const int hf = lane >> 4;  // which half of the job's rows
    const int h = 16 * warp + (lane & 15);
    const uint32_t lanes = (uint32_t)(warp * 32) << 16;
    const float sc2 = c.scale * kLog2e;
    float mref = -INFINITY, lrun = 0.f;
    JobWalk walk = walk0;
    int seg = 0, slot = 0;
    bool bad = false;  // a wait of this thread gave up
    for (int n = 0; n < J; ++n) {
      const JobRef r = walk.get(n);
      const bool first = r.first, last = r.last;
      if (first) slot = r.gid;
      const int g = n & 1, m = n >> 1;
      uint64_t mk = 0;
      if (!bad && !tc5::mbar_wait_backoff(smem_u32(&sm.mfull[g]), m & 1, abort, 64, wpolls)) bad = true;
      if (!bad) {
#pragma unroll
        for (int w = 0; w < kLoadWarps; ++w) mk |= sm.mask[g][w];
      }
      tc5::mbar_arrive(smem_u32(&sm.mempty[g]));
      if (!bad && !tc5::mbar_wait_backoff(smem_u32(&sm.s_full[g]), m & 1, abort, 64, wpolls)) bad = true;
      float s[32];
      if (!bad) {
        tc5::fence_after_sync();
        tc5::tmem_ld16x32bx2_32(tmem + kTmemS + 64 * g + lanes, s);
        tc5::fence_before_sync();
      } else {
#pragma unroll
        for (int j = 0; j < 32; ++j) s[j] = 0.f;
      }
      tc5::mbar_arrive(smem_u32(&sm.s_empty[g]));
      // tile max of the scaled scores over the rows that exist (log2 units),
      // as four independent running maxima, then across the pair
      const uint32_t mh = (uint32_t)(mk >> (32 * hf));
      float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
      if (mh == 0xffffffffu) {
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          s[j] *= sc2;
          m4[j & 3] = fmaxf(m4[j & 3], s[j]);
        }
      } else {
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          s[j] = ((mh >> j) & 1u) ? s[j] * sc2 : -INFINITY;
          m4[j & 3] = fmaxf(m4[j & 3], s[j]);
        }
      }
      float mt = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
      mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 16));
      // lazy rescale: keep the reference unless the tile max exceeds it by 2^8
      float alpha = 1.f;
      bool resc = false;
      if (first) {
        mref = mt;
        lrun = 0.f;
      } else if (mt > mref + kRescale) {
        alpha = mref == -INFINITY ? 0.f : exp2f(mref - mt);
        mref = mt;
        resc = true;
      }
      // P = 2^(s - m_ref) as bf16: this thread's half (64 bytes) of the
      // head's 128-byte row of P^T (K-major B operand, 128-byte swizzle) in
      // the job's rope sub-tile, which QK is done with; the weights are
      // summed as rounded, like the MMA sees them
      float ps[4] = {0.f, 0.f, 0.f, 0.f};
      if (!bad) {
        uint8_t* prow = gen + g * kBuf + 8 * kSub + h * 128;
        const float mo = mref == -INFINITY ? 0.f : mref;  // no row yet: every score is -inf
#pragma unroll
        for (int cl = 0; cl < 4; ++cl) {
          uint32_t w4[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int j = 8 * cl + 2 * e;
            const float p0 = ex2_approx(s[j] - mo);  // 0 for a masked row (-inf)
            const float p1 = ex2_approx(s[j + 1] - mo);
            const __nv_bfloat162 b2 = __floats2bfloat162_rn(p0, p1);
            ps[e] += __low2float(b2) + __high2float(b2);
            w4[e] = *reinterpret_cast<const uint32_t*>(&b2);
          }
          const int c8 = 4 * hf + cl;  // 16-byte chunk: rows 8 c8 .. 8 c8 + 7
          *reinterpret_cast<uint4*>(prow + ((c8 ^ (h & 7)) << 4)) = make_uint4(w4[0], w4[1], w4[2], w4[3]);
        }
        fence_proxy_async();
      }
      float psum = (ps[0] + ps[1]) + (ps[2] + ps[3]);
      psum += __shfl_xor_sync(0xffffffffu, psum, 16);  // the same sum in both threads of the pair
      lrun = lrun * alpha + psum;
      if (hf == 0) {
        sm.alpha[g][h] = alpha;
        if (last) sm.linv[seg & 1][h] = lrun > 0.f ? 1.f / lrun : 0.f;
      }
      const bool any = __any_sync(0xffffffffu, resc);
      const bool anybad = __any_sync(0xffffffffu, bad);
      if (lane == 0) sm.flag[g][warp] = (any ? 1 : 0) | ((anybad || *abort) ? 2 : 0);
      named_barrier_sync(1, 128);
      const int fl = sm.flag[g][0] | sm.flag[g][1] | sm.flag[g][2] | sm.flag[g][3];
      if (fl & 2) break;  // the same decision in every softmax thread
      if (fl & 1) {
        // O^T of the segment so far, times 2^(m_old - m_new) per head (column),
        // once the previous job's PV is complete; thread = TMEM lane = dim
        if (!bad && !tc5::mbar_wait_backoff(smem_u32(&sm.pv_done), (n - 1) & 1, abort, 64, wpolls)) bad = true;
        if (!bad) {
          tc5::fence_after_sync();
#pragma unroll 1
          for (int cc = 0; cc < 4; ++cc) {
#pragma unroll 1
            for (int half = 0; half < 2; ++half) {
              float o[32];
              const uint32_t col = kTmemO + 64 * cc + 32 * half;
              tc5::tmem_ld32(tmem + col + lanes, o);
#pragma unroll
              for (int i4 = 0; i4 < 8; ++i4) {
                const float4 a4 = reinterpret_cast<const float4*>(sm.alpha[g])[8 * half + i4];
                o[4 * i4 + 0] *= a4.x;
                o[4 * i4 + 1] *= a4.y;
                o[4 * i4 + 2] *= a4.z;
                o[4 * i4 + 3] *= a4.w;
              }
              tc5::tmem_st32(tmem + col + lanes, o);
            }
          }
          tc5::tmem_wait_st();
        }
      }
      tc5::fence_before_sync();
      tc5::mbar_arrive(smem_u32(&sm.p_full[g]));

      if (last) {
        // segment epilogue: thread (warp, lane) owns dim 128cc + 32warp + lane
        // of each chunk; writes the normalised output and each head's
        // log-sum-exp (log2 units)
        if (hf == 0) {
          ws.part_lse[(int64_t)slot * kTcH + h] = lrun > 0.f ? mref + log2f(lrun) : -INFINITY;
        }
        if (!bad && !tc5::mbar_wait_backoff(smem_u32(&sm.o_full), seg & 1, abort, 64, wpolls)) bad = true;
        if (!bad) {
          tc5::fence_after_sync();
          // heads x dims, bf16 (the range of fp32: a partial is a convex
          // combination of value rows, which may be any bf16 magnitude; fp16
          // would overflow past 65504): lanes 2i and 2i+1 swap values so that
          // each holds dims 2i, 2i+1 of one head of a pair (j, j+1); a warp
          // store covers 32 consecutive dims of two heads (two 64-byte runs)
          __nv_bfloat16* po = ws.part_o + (int64_t)slot * kTcH * kTcV;
          const bool odd = lane & 1;
#pragma unroll 1
          for (int half = 0; half < 2; ++half) {
            float inv[32];
#pragma unroll
            for (int i4 = 0; i4 < 8; ++i4) {
              const float4 l4 = reinterpret_cast<const float4*>(sm.linv[seg & 1])[8 * half + i4];
              inv[4 * i4 + 0] = l4.x;
              inv[4 * i4 + 1] = l4.y;
              inv[4 * i4 + 2] = l4.z;
              inv[4 * i4 + 3] = l4.w;
            }
#pragma unroll 1
            for (int cc = 0; cc < 4; ++cc) {
              float o[32];
              tc5::tmem_ld32(tmem + kTmemO + 64 * cc + 32 * half + lanes, o);
              const int d0 = cc * 128 + warp * 32 + (lane & ~1);  // the pair's first dim
              __nv_bfloat16* row = po + (int64_t)(32 * half + (odd ? 1 : 0)) * kTcV + d0;
#pragma unroll
              for (int j = 0; j < 32; j += 2) {
                // even lane keeps head j, odd lane head j+1; each sends the other
                const float mine = odd ? o[j + 1] * inv[j + 1] : o[j] * inv[j];
                const float give = odd ? o[j] * inv[j] : o[j + 1] * inv[j + 1];
                const float got = __shfl_xor_sync(0xffffffffu, give, 1);
                *reinterpret_cast<__nv_bfloat162*>(row + (int64_t)j * kTcV) =
                    odd ? __floats2bfloat162_rn(got, mine) : __floats2bfloat162_rn(mine, got);
              }
            }
          }
        }
        tc5::fence_before_sync();
        tc5::mbar_arrive(smem_u32(&sm.o_empty));
        // publish the segment to the merge kernel: the four warps meet (the
        // barrier orders their partial stores before thread 0's release, which
        // is cumulative over what the barrier ordered before it), and one
        // thread stores this launch's epoch into the segment's flag with
        // release semantics
        named_barrier_sync(2, 128);
        if (tid == 0 && !bad) {
          asm volatile("st.release.gpu.global.b32 [%0], %1;\n" ::"l"(ws.seg_ready + slot), "r"(seg_epoch)
                       : "memory");
        }
        ++seg;
      }
    }
  }

  if (tid == 0 && *abort) set_status(ws.status, kStatusTimeout);
  tc5::fence_before_sync();
  __syncthreads();
  tc5::fence_after_sync();
  if (warp == 4) tc5::tmem_dealloc(tmem, 512);
  // with flags nothing above waited for the previous grid: this grid then
  // completes only after it (the Top-K blocks have published by now), so
  // that every later kernel of the stream still follows the Top-K kernel
  if (flags) pdl_wait();
}

// Per (query, 64 output dims): LSE merge of the query's segment partials,
// inverse RoPE on the last R dims, bf16 store.  The segments are the query's
// W jobs cut at the tile CTAs' W ranges, then its C jobs cut at their C
// ranges (see Sched); the block lists them, thread i testing CTA i.  Thread
// t owns head t >> 2 and 16 consecutive dims (t & 3) of the block's 64: it
// loads its head's LSE and a 32-byte piece of the partials, two segments per
// batch, derives the weights itself (running max across batches), and stores
// 32 bytes.  (Four per batch need 80 registers, so three blocks per SM, and
// the last blocks then start only after the tile grid: measured slower.)
constexpr int kMergeUnroll = 2;  // partials whose loads are in flight together

// Appends to seg[] the partial slots of the CTA ranges that intersect the
// jobs [a, b) of one list of n jobs split at start(i), i < g (id offset
// `base`), in CTA order; returns the new count.  Every thread of the block
// calls it: thread t tests CTAs t, t + blockDim.x, ..., and a ballot per warp
// plus the warps' counts place the pieces in order (a serial walk by one
// thread costs microseconds of dependent divisions at the end of the step).
// `wcnt` holds one int per warp.
template <typename Start>
__device__ int list_segments(int a, int b, int n, int g, int base, Start start, int* seg, int k,
                             int* wcnt) {
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5, nwarps = blockDim.x >> 5;
  if (b <= a || n <= 0) return k;
  for (int i0 = 0; i0 < g; i0 += blockDim.x) {
    const int i = i0 + t;
    bool in = false;
    int slot = 0;
    if (i < g) {
      const int lo = start(i), hi = i + 1 < g ? start(i + 1) : n;
      in = hi > lo && hi > a && lo < b;
      slot = base + (lo > a ? lo : a);
    }
    const uint32_t bal = __ballot_sync(0xffffffffu, in);
    if (lane == 0) wcnt[warp] = __popc(bal);
    __syncthreads();
    int before = 0, tot = 0;
    for (int w = 0; w < nwarps; ++w) {
      const int cw = wcnt[w];
      before += w < warp ? cw : 0;
      tot += cw;
    }
    const int pos = k + before + __popc(bal & ((1u << lane) - 1u));
    if (in && pos < kMergeMaxJobs) seg[pos] = slot;
    k += tot;
    __syncthreads();  // wcnt is rewritten by the next chunk
  }
  return k;
}

// flags != 0: launched right after the tile kernel of the same call, which
// publishes each segment through ws.seg_ready with seg_epoch: a block starts
// as soon as its query's segments are written, and waits for the tile grid
// only at its end.
__global__ void __launch_bounds__(256, 4)
    attn_merge_kernel(const __grid_constant__ JobLists jobs, DevCfg c, DevBatch b, Workspace ws,
                      int G, __nv_bfloat16* __restrict__ out, float* __restrict__ lse_out,
                      int flags, int seg_epoch) {
  __shared__ int seg[kMergeMaxJobs + 1];
  __shared__ int nseg_s;
  __shared__ int wcnt[256 / 32];  // per-warp piece counts of list_segments (256 threads)
  __shared__ float2 rope[kRopeTable];  // cos, sin of the block's rotary pairs
  // The segment list and the rotary table need only the job lists and the
  // lengths, which are complete before the tile kernel lets this grid
  // launch (the tile kernel waits for the job-list kernel before it
  // triggers, and for the caller's inputs before it or its predecessor
  // does); only the partials wait for the tile grid.
  // the blocks of the last dims (the rotary ones, whose table takes longest
  // to set up) are dispatched first
  const int q = blockIdx.x, dg = gridDim.y - 1 - blockIdx.y, t = threadIdx.x;
  const int T = b.B * b.S;
  const int rope0 = kTcV - c.R;  // first rotary dim
  if (dg * kMergeDims + kMergeDims > rope0 && t >= 64 && t < 64 + c.R / 2 && t - 64 < kRopeTable) {
    const int bi = q / b.S;
    const QueryPlan p = query_plan(c, b.S, b.ctx_len[bi], q - bi * b.S, 0);
    const int i = t - 64;
    rope[i] = (p.flags & kPlanBad) ? make_float2(1.f, 0.f) : rope_cos_sin((double)p.pos, c.rope_theta[i]);
  }
  {
    Sched sc;
    sc.wp = jobs.host_T >= 0 ? jobs.wprefix : ws.job_prefix;
    sc.cp = jobs.host_T >= 0 ? jobs.cprefix : ws.job_prefix + (T + 1);
    sc.cq = nullptr;
    sc.cspan = nullptr;
    sc.T = T;
    sc.NW = jobs.host_T >= 0 ? jobs.NW : sc.wp[T];
    sc.NC = jobs.host_T >= 0 ? jobs.NC : sc.cp[T];
    sc.G = G;
    sc.E = (jobs.host_T >= 0 && jobs.early > 0 && jobs.early < G) ? jobs.early : G;
    sc.weights(jobs);
    // the query's job ranges, loaded together before the first barrier
    const int wa = sc.wp[q], wb = sc.wp[q + 1], ca = sc.cp[q], cb = sc.cp[q + 1];
    int k = list_segments(wa, wb, sc.NW, sc.E, 0, [&](int i) { return sc.wstart(i); }, seg, 0, wcnt);
    k = list_segments(ca, cb, sc.NC, sc.G, sc.NW, [&](int i) { return sc.cstart(i); }, seg, k, wcnt);
    if (t == 0) nseg_s = k;
  }
  __syncthreads();
  if (flags) {
    // thread k < nseg polls segment k's flag (bounded); a wait that gives up
    // reports a timeout and the query is written as zeros
    pdl_trigger();
    const int ns = min(nseg_s, kMergeMaxJobs);
    if (t < ns) {
      const uint32_t limit = c.wait_polls < 0 ? (1u << 23) : (uint32_t)c.wait_polls;
      const int* f = ws.seg_ready + seg[t];
      uint32_t i = 0, nsl = 32;
      while (ld_acquire(f) != seg_epoch) {
        if (++i >= limit) {
          set_status(ws.status, kStatusTimeout);
          nseg_s = 0;
          break;
        }
        if (i >= 8) {
          __nanosleep(nsl);
          nsl = nsl * 2 > 256 ? 256 : nsl * 2;
        }
      }
    }
    __syncthreads();
  } else {
    pdl_wait();
    pdl_trigger();
  }
  const int nseg = min(nseg_s, kMergeMaxJobs);
  const int h = t >> 2;
  const int v0 = dg * kMergeDims + 16 * (t & 3);
  // partials and LSEs in batches of kMergeUnroll, loaded together; a running
  // max over the batches rescales what is summed so far
  float M = -INFINITY, tot = 0.f;
  float acc[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) acc[i] = 0.f;
  for (int k0 = 0; k0 < nseg; k0 += kMergeUnroll) {
    uint4 u[kMergeUnroll][2];
    float lk[kMergeUnroll];
#pragma unroll
    for (int kk = 0; kk < kMergeUnroll; ++kk) {
      if (k0 + kk < nseg) {
        const int64_t sb = (int64_t)seg[k0 + kk] * kTcH + h;
        // L2-coherent loads: with flags the tile kernel may still be running
        const uint4* src = reinterpret_cast<const uint4*>(ws.part_o + sb * kTcV + v0);
        u[kk][0] = __ldcg(src);
        u[kk][1] = __ldcg(src + 1);
        lk[kk] = __ldcg(ws.part_lse + sb);
      } else {
        u[kk][0] = u[kk][1] = make_uint4(0u, 0u, 0u, 0u);
        lk[kk] = -INFINITY;
      }
    }
    float Mn = M;
#pragma unroll
    for (int kk = 0; kk < kMergeUnroll; ++kk) Mn = fmaxf(Mn, lk[kk]);
    if (Mn > M && M != -INFINITY) {
      const float sc = exp2f(M - Mn);
      tot *= sc;
#pragma unroll
      for (int i = 0; i < 16; ++i) acc[i] *= sc;
    }
    M = Mn;
#pragma unroll
    for (int kk = 0; kk < kMergeUnroll; ++kk) {
      const float w = (M == -INFINITY || lk[kk] == -INFINITY) ? 0.f : exp2f(lk[kk] - M);
      tot += w;
      const __nv_bfloat162* a = reinterpret_cast<const __nv_bfloat162*>(&u[kk][0]);
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        acc[2 * e] = fmaf(w, __low2float(a[e]), acc[2 * e]);
        acc[2 * e + 1] = fmaf(w, __high2float(a[e]), acc[2 * e + 1]);
      }
    }
  }
  const float it = tot > 0.f ? 1.f / tot : 0.f;
  uint32_t pk[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    const int v = v0 + 2 * e;
    const float x0 = acc[2 * e] * it, x1 = acc[2 * e + 1] * it;
    float cs = 1.f, sn = 0.f;
    if (v >= rope0) {
      const float2 r = rope[(v - rope0) >> 1];
      cs = r.x;
      sn = r.y;
    }
    pk[e] = pack_bf16x2(x0 * cs + x1 * sn, -x0 * sn + x1 * cs);
  }
  uint4* dst = reinterpret_cast<uint4*>(out + ((int64_t)q * kTcH + h) * kTcV + v0);
  dst[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
  dst[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
  if (lse_out && dg == 0 && (t & 3) == 0)
    lse_out[(int64_t)q * kTcH + h] = M == -INFINITY ? -INFINITY : (M + log2f(tot)) * 0.6931471805599453f;
  // with flags nothing above waited for the tile grid: this grid completes
  // only after it, so that every later kernel of the stream follows it
  if (flags) pdl_wait();
}

// W and C job counts of a query (see JobLists), from the bound min(vis, K).
__host__ __device__ __forceinline__ void query_jobs(int nwin, int cnt, int vis2, int* nw, int* nc) {
  *nw = (nwin + kTile - 1) / kTile + (vis2 + kTile - 1) / kTile;
  *nc = (cnt + kTile - 1) / kTile;
}

// Builds the job lists into ws.job_prefix when the host has no lengths.
__global__ void __launch_bounds__(1024) job_prep_kernel(DevCfg c, DevBatch b, Workspace ws) {
  __shared__ int scan_tmp[33];
  __shared__ int wcarry, ccarry;
  pdl_wait();
  const int T = b.B * b.S;
  int* wp = ws.job_prefix;
  int* cp = ws.job_prefix + (T + 1);
  if (threadIdx.x == 0) wcarry = ccarry = 0;
  __syncthreads();
  for (int base = 0; base < T; base += blockDim.x) {
    const int q = base + threadIdx.x;
    int nw = 0, nc = 0;
    if (q < T) {  // no split: every tile of the query in the C list
      const int bi = q / b.S;
      const QueryPlan p = query_plan(c, b.S, b.ctx_len[bi], q - bi * b.S, 0);
      query_jobs(p.nwin, p.cnt, p.vis2, &nw, &nc);
      nc += nw;
      nw = 0;
    }
    int wtot, ctot;
    const int wex = block_exclusive_scan(nw, scan_tmp, &wtot);
    const int cex = block_exclusive_scan(nc, scan_tmp, &ctot);
    if (q < T) {
      wp[q] = wcarry + wex;
      cp[q] = ccarry + cex;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      wcarry += wtot;
      ccarry += ctot;
    }
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    wp[T] = wcarry;
    cp[T] = ccarry;
  }
  pdl_trigger();
}

bool make_map(CUtensorMap* m, const void* ptr, uint64_t rows, uint64_t stride, uint32_t box_rows) {
  auto fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(tensor_map_encoder());
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)kTcD, rows};
  cuuint64_t strides[1] = {stride * 2};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

// Builds the job lists on the host when the lengths are known (jobs.host_T =
// number of queries), else leaves host_T = -1 for the device job-list kernel.
// The W jobs go to the tile CTAs that find a free SM when the grid starts:
// the grid's CTAs take SMs in index order, and the Top-K blocks that select
// hold topk_blocks SMs until they finish.
void host_jobs(const DevCfg& c, int B, int S, const int32_t* lens_host, int num_sms, int topk_blocks,
               JobLists* jobs) {
  jobs->host_T = -1;
  jobs->split = 0;
  jobs->early = 0;
  jobs->cw_early = jobs->cw_a = jobs->cw_b = 0;
  if (!lens_host || B * S > kMaxHostReq) return;
  // CSA_EARLY_SPLIT=1: the W / C split (see JobLists); by default one list
  static const bool split = [] {
    const char* e = getenv("CSA_EARLY_SPLIT");
    return e && e[0] == '1';
  }();
  int wacc = 0, cacc = 0;
  for (int bi = 0; bi < B; ++bi)
    for (int s = 0; s < S; ++s) {
      jobs->wprefix[bi * S + s] = wacc;
      jobs->cprefix[bi * S + s] = cacc;
      const int L = lens_host[bi];
      if (L < S || L > c.max_context) continue;
      const int pos = L - S + s;
      const int vis = (pos + 1) / c.ratio;
      const int nwin = c.win < pos + 1 ? c.win : pos + 1;
      const int cnt = vis < c.K ? vis : c.K;
      const int vis2 = c.hca_ratio > 0 ? (pos + 1) / c.hca_ratio : 0;
      int nw, nc;
      query_jobs(nwin, cnt, vis2, &nw, &nc);
      if (!split) {
        nc += nw;
        nw = 0;
      }
      wacc += nw;
      cacc += nc;
    }
  jobs->wprefix[B * S] = wacc;
  jobs->cprefix[B * S] = cacc;
  jobs->host_T = B * S;
  jobs->split = split ? 1 : 0;
  // early CTAs: the SMs the selecting Top-K blocks leave free; too few of
  // them would be swamped with the W jobs, and then all CTAs share them
  const int early = num_sms - (topk_blocks < num_sms ? topk_blocks : num_sms);
  jobs->early = (split && topk_blocks > 0 && early >= num_sms / 4) ? early : 0;
  // Without the split, the CTAs that start while the Top-K blocks still
  // hold their SMs take more of the list: an even split whose left-over jobs
  // go to them first (cw_a = 0).  A late CTA's start (its SM freed, the
  // CTA's set-up, the first rows) costs about a job's time, so it gets no
  // more than the average; measured on a 64-query long-context step against
  // weight ratios from 2:1 to 1:1 (5:4 was 1 us slower, 12:11, which gives
  // the same split there, as fast).  CSA_TILE_WEIGHT=a:b sets weights instead.
  static const int2 wt = [] {
    int2 r = make_int2(0, 0);
    if (const char* e = getenv("CSA_TILE_WEIGHT")) {
      int a = 0, b2 = 0;
      if (sscanf(e, "%d:%d", &a, &b2) == 2 && a > 0 && b2 > 0 && a <= 64 && b2 <= 64) r = make_int2(a, b2);
    }
    return r;
  }();
  if (!split && topk_blocks > 0 && early > 0 && (wt.x == 0 || wt.x != wt.y)) {
    jobs->cw_early = early;
    jobs->cw_a = wt.x;
    jobs->cw_b = wt.y;
  }
}

namespace {
// The query holding each tile CTA's first job of each list, from the same
// split of the lists as Sched (wstart / cstart), for host-built lists.
void host_cta_queries(JobLists& jobs, int grid) {
  const int T = jobs.host_T;
  jobs.NW = jobs.wprefix[T];
  jobs.NC = jobs.cprefix[T];
  jobs.cta_first = grid <= kMaxTileCtas && T <= 65536 ? 1 : 0;
  if (!jobs.cta_first) return;
  const int E = (jobs.early > 0 && jobs.early < grid) ? jobs.early : grid;
  const bool w = jobs.cw_early > 0 && (jobs.cw_a == 0 || (jobs.cw_a > 0 && jobs.cw_b > 0));
  const int CE = w ? jobs.cw_early : grid, wa = w ? jobs.cw_a : 1, wb = w ? jobs.cw_b : 1;
  for (int list = 0; list < 2; ++list) {
    const int* p = list == 0 ? jobs.wprefix : jobs.cprefix;
    const int N = list == 0 ? jobs.NW : jobs.NC;
    int q = 0;
    for (int i = 0; i < grid; ++i) {
      const int lo = list == 0 ? (i >= E ? N : (int)((int64_t)i * N / E))
                               : c_list_start(i, N, grid, CE, wa, wb);
      // the largest q with p[q] <= lo (lo only grows with i)
      while (q + 1 < T && p[q + 1] <= lo) ++q;
      jobs.cta_q[list][i] = (uint16_t)q;
      jobs.cta_span[list][i][0] = p[q];
      jobs.cta_span[list][i][1] = p[q + 1];
    }
  }
}
}  // namespace

// Jobs one query can have at most (sizes the partial-output workspace).
int max_jobs_per_query(const DevCfg& c) {
  const int kmax = c.K < c.max_vis ? c.K : c.max_vis;
  int n = (c.win + kTile - 1) / kTile + (kmax + kTile - 1) / kTile;
  if (c.hca_ratio > 0) n += (c.max_context / c.hca_ratio + kTile - 1) / kTile;
  return n;
}

// Returns launches (>= 1), 0 with nothing to do, -1 on failure, -2 if the
// batch does not fit this path (the caller then uses the warp-MMA kernel).
int launch_attention_tc5(const DevCfg& c, const DevBatch& b, const Workspace& ws,
                         JobLists& jobs, const int* topk_idx, const int* topk_cnt, void* out,
                         float* lse_out, int num_sms, cudaStream_t st, bool pdl, bool early,
                         int epoch, int seg_epoch) {
  const int T = b.B * b.S;
  if (T == 0) return 0;
  if (!ws.part_o || max_jobs_per_query(c) > kMergeMaxJobs || b.raw_rows > 0x7fffffffLL ||
      b.cmp_rows > 0x7fffffffLL || b.hca_rows > 0x7fffffffLL || (int64_t)T * kTcH > 0x7fffffffLL)
    return -2;
  CUtensorMap qmap;
  if (!make_map(&qmap, b.q, (uint64_t)T * kTcH, kTcD, kTcH))
    return launch_fail("cuTensorMapEncodeTiled(q)", cudaSuccess);
  static PerDeviceOnce attr;
  if (const cudaError_t e = attr.run([] {
        cudaError_t r = allow_max_dynamic_smem(attn_tile_kernel<false>);
        if (r == cudaSuccess) r = allow_max_dynamic_smem(attn_tile_kernel<true>);
        return r;
      }))
    return launch_fail("cudaFuncSetAttribute(attn_tile_kernel)", e);
  const bool paged = b.raw_table || b.cmp_table || b.hca_table;
  int n = 0;
  if (jobs.host_T < 0) {
    if (launch_kernel(job_prep_kernel, dim3(1), dim3(1024), 0, st, pdl, c, b, ws) < 0) return -1;
    ++n;
  }
  int grid = num_sms;
  if (jobs.host_T >= 0) {
    const int total = jobs.wprefix[T] + jobs.cprefix[T];
    if (total < grid) grid = total > 0 ? total : 1;
    host_cta_queries(jobs, grid);
  }
  // the Top-K ready flags stand in for the grid dependency only when this
  // kernel follows the step's own Top-K kernel through a programmatic launch
  if (launch_kernel(paged ? attn_tile_kernel<true> : attn_tile_kernel<false>, dim3(grid),
                    dim3(kA5Threads), kA5Dyn, st, pdl, qmap, jobs, c, b, ws, topk_idx, topk_cnt,
                    (pdl && early) ? 1 : 0, epoch, seg_epoch) < 0)
    return -1;
  ++n;
  // the segment flags stand in for the tile grid's completion when the merge
  // follows it through a programmatic launch
  if (launch_kernel(attn_merge_kernel, dim3(T, kTcV / kMergeDims), dim3(256), 0, st, pdl, jobs, c,
                    b, ws, grid, static_cast<__nv_bfloat16*>(out), lse_out, pdl ? 1 : 0, seg_epoch) < 0)
    return -1;
  return n + 1;
}

}  // namespace csa
