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
// CTA takes a contiguous range of the job list, and the jobs of one query
// inside that range form a segment whose output accumulates in TMEM.
//   warps 5-10, two groups of three: group g gathers every other job into
//            job buffer g with coalesced 16-byte cp.async, rows scattered
//            over the pools, into nine 128-byte-swizzled 64-dim sub-tiles
//            (72 KB); each thread fences its copies for the async proxy and
//            arrives on the buffer's barrier.  Two buffers: one job's rows
//            land while the previous job is computed;
//   warp 4   loads the query's 64 heads x 576 (72 KB, TMA) when the query
//            changes and issues the tcgen05 MMAs as their inputs become
//            ready: S[64 heads x 64 rows] = Q . R^T over 576 dims (M = 64,
//            N = 64) into one of two TMEM score buffers; after the softmax,
//            O^T[512 dims x 64 heads] += V^T . P^T (M = 128 per 128-dim
//            chunk, N = 64; V read in place as an MN-major operand, P^T
//            from the rope sub-tile that QK no longer needs) into TMEM;
//   warps 0-3 softmax, one thread per head (lanes 0-15: the M = 64 layout
//            puts head 16w + i in lane 32w + i): scale and mask the job's 64
//            scores, keep a per-head reference max that moves only when a
//            tile max exceeds it by 2^8 (then O^T is rescaled in TMEM by all
//            128 threads), write the head's row of P^T as bf16 and sum the
//            rounded weights.  At a segment's end all four warps read O^T
//            (thread = dim) and write the normalised partial output (bf16,
//            heads x dims) and the heads' log-sum-exp to the workspace.
// attn_merge_kernel: per query and 64 output dims, the log-sum-exp merge of
// the query's segments in job order, inverse RoPE on the last R dims, the
// bf16 store.  Because the merge is exact, segment softmax + merge equals
// one softmax over the union of the streams' rows.
#include <cudaTypedefs.h>
#include <stddef.h>
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

// Job list: jobs of query q are [prefix[q], prefix[q+1]); in each query the
// window tiles, then the compressed tiles, then the heavy tiles.
struct JobCursor {
  const int* prefix;
  int q, first, end;
  __device__ __forceinline__ void init(const int* p, int T, int job) {
    prefix = p;
    int l = 0, r = T - 1;
    while (l < r) {
      const int m = (l + r + 1) >> 1;
      if (p[m] <= job) l = m; else r = m - 1;
    }
    q = l;
    first = p[l];
    end = p[l + 1];
  }
  __device__ __forceinline__ void advance(int job) {
    while (job >= end) {
      ++q;
      first = end;
      end = prefix[q + 1];
    }
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
__device__ __forceinline__ JobCtx job_ctx(const DevCfg& c, const DevBatch& b, int q) {
  JobCtx x;
  x.bi = q / b.S;
  x.p = query_plan(c, b.S, b.ctx_len[x.bi], q - x.bi * b.S, 0);
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
__device__ __forceinline__ void job_topk_cnt(JobCtx& x, int q, const int* __restrict__ topk_cnt) {
  int cnt = 0;
  if (!(x.p.flags & kPlanBad)) {
    cnt = topk_cnt[q];
    cnt = cnt < 0 ? 0 : (cnt > x.p.cnt ? x.p.cnt : cnt);
  }
  x.n[1] = cnt;
}

__device__ __forceinline__ void job_stream(const JobCtx& x, int local, int& sid, int& t) {
  if (local < x.nt[0]) { sid = 0; t = local; }
  else if (local < x.nt[0] + x.nt[1]) { sid = 1; t = local - x.nt[0]; }
  else { sid = 2; t = local - x.nt[0] - x.nt[1]; }
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
    attn_tile_kernel(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ ItemList jobs, DevCfg c, DevBatch b, Workspace ws,
                     const int* __restrict__ topk_idx, const int* __restrict__ topk_cnt,
                     int early) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  __shared__ A5Smem sm;
  const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
  const uint32_t qres = base;                 // 72 KB: the query's 64 heads
  const uint32_t bufs = qres + kQBytes;       // 2 x 72 KB: the jobs' rows
  uint8_t* gen = smem_raw + (bufs - smem_u32(smem_raw));

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int T = b.B * b.S;
  // Launched right after this library's Top-K kernel of the same step
  // (early != 0), every input but the Top-K outputs was complete before the
  // step's first kernel passed its own wait, so only the row loaders wait
  // for the previous grid, when they first read topk_idx / topk_cnt, and
  // setup, Q and window rows overlap its tail.  Otherwise (a caller's kernel
  // before this one, or a job list built on the device) every thread waits
  // first.
  const bool wait_all = !(early && jobs.host_B >= 0);
  if (wait_all) pdl_wait();
  const int* __restrict__ prefix = jobs.host_B >= 0 ? jobs.prefix : ws.job_prefix;
  const int N = prefix[T];
  const int lo = (int)((int64_t)blockIdx.x * N / gridDim.x);
  const int hi = (int)((int64_t)(blockIdx.x + 1) * N / gridDim.x);
  pdl_trigger();
  if (lo >= hi) return;
  volatile int* abort = &sm.abort;
  // polls before a consumer wait gives up (the default: about a second)
  const uint32_t wpolls = c.wait_polls < 0 ? tc5::kBackoffPolls : (uint32_t)c.wait_polls;

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
    JobCursor cur;
    cur.init(prefix, T, lo);
    int m = 0;
    bool waited = wait_all;
    for (int job = lo + g; job < hi; job += 2, ++m) {
      if (__shfl_sync(0xffffffffu, *abort, 0)) break;
      cur.advance(job);
      const int q = cur.q;
      JobCtx x = job_ctx(c, b, q);
      int sid, t;
      job_stream(x, job - cur.first, sid, t);
      const __nv_bfloat16* pool = static_cast<const __nv_bfloat16*>(
          sid == 0 ? b.raw : (sid == 1 ? b.cmp : b.hca));
      const int64_t stride = sid == 0 ? b.raw_stride : (sid == 1 ? b.cmp_stride : b.hca_stride);
      const int* tbl = kPaged ? (sid == 0 ? b.raw_table : (sid == 1 ? b.cmp_table : b.hca_table)) : nullptr;
      const int64_t off = tbl ? -1 : (sid == 0 ? b.raw_off[x.bi] : (sid == 1 ? b.cmp_off[x.bi] : b.hca_off[x.bi]));
      // this lane's rows: their Top-K indices are loaded together with the
      // count they are checked against
      int jr[kQuadsPerWarp];
#pragma unroll
      for (int i = 0; i < kQuadsPerWarp; ++i) jr[i] = -1;
      if (sid == 1) {
        if (!waited) {
          pdl_wait();
          waited = true;
        }
#pragma unroll
        for (int i = 0; i < kQuadsPerWarp; ++i) {
          const int rq = lw + kLoadWarps * i;
          const int ri = t * kTile + 4 * rq + (lane >> 3);
          if (rq < kTile / 4 && ri < c.K) jr[i] = topk_idx[(int64_t)q * c.K + ri];
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
      JobCursor qc, pc;  // cursors of the next QK job and the next PV job
      qc.init(prefix, T, lo);
      pc.init(prefix, T, lo);
      const int J = hi - lo;
      int nk = 0, np = 0;  // CTA-local index of the next job to QK / to PV
      int nq = 0, nqd = 0, seg = 0, cur_q = -1;
      int qstate = 0;      // 0 Q of cur_q resident, 1 waiting for qdone, 2 waiting for qfull
      uint32_t idle = 0;
      while (np < J) {
        bool progressed = false;
        if (np < nk) {
          const int job = lo + np;
          pc.advance(job);
          const bool first = job == lo || job == pc.first;
          const bool last = job + 1 == hi || job + 1 == pc.end;
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
          const int job = lo + nk;
          qc.advance(job);
          if (qc.q != cur_q) {
            // a new query: its heads replace Q once the QK MMAs of the
            // previous query are done (qdone)
            if (qstate == 0) qstate = nk == 0 ? 3 : 1;
            if (qstate == 1 && tc5::mbar_try_wait(smem_u32(&sm.qdone), nqd & 1)) {
              ++nqd;
              qstate = 3;
            }
            if (qstate == 3) {
              tc5::mbar_expect_tx(smem_u32(&sm.qfull), kQBytes);
              for (int k = 0; k < 9; ++k)
                tc5::tma_load_2d(qres + k * kQSub, &qmap, k * 64, qc.q * kTcH, smem_u32(&sm.qfull));
              qstate = 2;
            }
            if (qstate == 2 && tc5::mbar_try_wait(smem_u32(&sm.qfull), nq & 1)) {
              ++nq;
              qstate = 0;
              cur_q = qc.q;
            }
          }
          const int g = nk & 1, m = nk >> 1;
          if (qc.q == cur_q && (m == 0 || tc5::mbar_try_wait(smem_u32(&sm.s_empty[g]), (m - 1) & 1)) &&
              tc5::mbar_try_wait(smem_u32(&sm.full[g]), m & 1)) {
            // S = Q . R^T over 576 dims (M = 64 heads, N = 64 rows)
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
            if (job + 1 < hi && job + 1 == qc.end) tc5::mma_commit(smem_u32(&sm.qdone));
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
    JobCursor cur;
    cur.init(prefix, T, lo);
    int n = 0, seg = 0, slot = lo;
    bool bad = false;  // a wait of this thread gave up
    for (int job = lo; job < hi; ++job, ++n) {
      cur.advance(job);
      const bool first = job == lo || job == cur.first;
      const bool last = job + 1 == hi || job + 1 == cur.end;
      if (first) slot = job;
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
        ++seg;
      }
    }
  }

  if (tid == 0 && *abort) set_status(ws.status, kStatusTimeout);
  tc5::fence_before_sync();
  __syncthreads();
  tc5::fence_after_sync();
  if (warp == 4) tc5::tmem_dealloc(tmem, 512);
}

// Per (query, 64 output dims): LSE merge of the query's segment partials in
// job order, inverse RoPE on the last R dims, bf16 store.  The segments are
// the query's job range cut at the tile kernel's CTA boundaries (CTA i takes
// jobs [iN/G, (i+1)N/G)); with N >= G the starts are strictly increasing, so
// segment k > 0 starts at (i0 + k)N/G directly.  Thread t owns head t >> 2 and
// 16 consecutive dims (t & 3) of the block's 64: it loads its head's LSE and
// a 32-byte piece of the partials, four segments per batch, derives the
// weights itself (running max across batches), and stores 32 bytes.
constexpr int kMergeUnroll = 2;  // partials whose loads are in flight together
__global__ void __launch_bounds__(256, 3)
    attn_merge_kernel(const __grid_constant__ ItemList jobs, DevCfg c, DevBatch b, Workspace ws,
                      int G, __nv_bfloat16* __restrict__ out, float* __restrict__ lse_out) {
  __shared__ int seg[kMergeMaxJobs + 1];
  __shared__ int nseg_s;
  __shared__ float2 rope[kRopeTable];  // cos, sin of the block's rotary pairs
  // The segment list and the rotary table need only the job list and the
  // lengths, which are complete before the tile kernel lets this grid
  // launch (the tile kernel waits for the job-list kernel before it
  // triggers, and for the caller's inputs before it or its predecessor
  // does); only the partials wait for the tile grid.
  const int q = blockIdx.x, dg = blockIdx.y, t = threadIdx.x;
  const int T = b.B * b.S;
  const int* __restrict__ prefix = jobs.host_B >= 0 ? jobs.prefix : ws.job_prefix;
  const int N = prefix[T], j0 = prefix[q], j1 = prefix[q + 1];
  const int rope0 = kTcV - c.R;  // first rotary dim
  if (dg * kMergeDims + kMergeDims > rope0 && t >= 64 && t < 64 + c.R / 2 && t - 64 < kRopeTable) {
    const int bi = q / b.S;
    const QueryPlan p = query_plan(c, b.S, b.ctx_len[bi], q - bi * b.S, 0);
    const int i = t - 64;
    rope[i] = (p.flags & kPlanBad) ? make_float2(1.f, 0.f) : rope_cos_sin((double)p.pos, c.rope_theta[i]);
  }
  // CTA i starts at job (i N) / G; 32-bit arithmetic while i N fits
  const bool small = (uint64_t)N * (uint64_t)G < (1ull << 32);
  auto cta_start = [&](int i) -> int {
    return small ? (int)((uint32_t)i * (uint32_t)N / (uint32_t)G) : (int)((int64_t)i * N / G);
  };
  if (j1 <= j0) {
    if (t == 0) nseg_s = 0;
  } else if (N >= G) {
    // starts strictly increase: with i0 the CTA holding j0, segment t > 0
    // starts at (i0 + t)N/G while that is < j1
    if (t < kMergeMaxJobs) {
      int i0 = small ? (int)((uint32_t)j0 * (uint32_t)G / (uint32_t)N) : (int)((int64_t)j0 * G / N);
      if (i0 + 1 < G && cta_start(i0 + 1) <= j0) ++i0;
      const int i = i0 + t;
      const int l = t == 0 ? j0 : (i < G ? cta_start(i) : j1);
      if (l < j1) seg[t] = l;
      const int lnext = i + 1 < G ? cta_start(i + 1) : j1;
      if (l < j1 && lnext >= j1) nseg_s = t + 1;  // the last segment
    }
  } else if (t == 0) {
    // more CTAs than jobs: runs of equal starts, walked in order
    int k = 0, last = j0;
    seg[k++] = j0;
    for (int i = (int)((int64_t)j0 * G / N) + 1; i < G && k < kMergeMaxJobs; ++i) {
      const int l = cta_start(i);
      if (l >= j1) break;
      if (l > last) {
        seg[k++] = l;
        last = l;
      }
    }
    nseg_s = k;
  }
  __syncthreads();
  pdl_wait();
  pdl_trigger();
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
        const uint4* src = reinterpret_cast<const uint4*>(ws.part_o + sb * kTcV + v0);
        u[kk][0] = src[0];
        u[kk][1] = src[1];
        lk[kk] = ws.part_lse[sb];
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
}

// Counts each query's jobs into ws.job_prefix when the host has no lengths.
__global__ void __launch_bounds__(1024) job_prep_kernel(DevCfg c, DevBatch b, Workspace ws) {
  __shared__ int scan_tmp[33];
  __shared__ int carry;
  pdl_wait();
  const int T = b.B * b.S;
  if (threadIdx.x == 0) carry = 0;
  __syncthreads();
  for (int base = 0; base < T; base += blockDim.x) {
    const int q = base + threadIdx.x;
    int n = 0;
    if (q < T) {
      const int bi = q / b.S;
      const QueryPlan p = query_plan(c, b.S, b.ctx_len[bi], q - bi * b.S, 0);
      n = (p.nwin + kTile - 1) / kTile + (p.cnt + kTile - 1) / kTile + (p.vis2 + kTile - 1) / kTile;
    }
    int total;
    const int ex = block_exclusive_scan(n, scan_tmp, &total);
    if (q < T) ws.job_prefix[q] = carry + ex;
    __syncthreads();
    if (threadIdx.x == 0) carry += total;
    __syncthreads();
  }
  if (threadIdx.x == 0) ws.job_prefix[T] = carry;
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

// Builds the job list on the host when the lengths are known (jobs.host_B =
// number of queries), else leaves host_B = -1 for the device prep kernel.
void host_jobs(const DevCfg& c, int B, int S, const int32_t* lens_host, ItemList* jobs) {
  jobs->host_B = -1;
  if (!lens_host || B * S > kMaxHostReq) return;
  int acc = 0;
  for (int bi = 0; bi < B; ++bi)
    for (int s = 0; s < S; ++s) {
      jobs->prefix[bi * S + s] = acc;
      const int L = lens_host[bi];
      if (L < S || L > c.max_context) continue;
      const int pos = L - S + s;
      const int vis = (pos + 1) / c.ratio;
      const int nwin = c.win < pos + 1 ? c.win : pos + 1;
      const int cnt = vis < c.K ? vis : c.K;
      const int vis2 = c.hca_ratio > 0 ? (pos + 1) / c.hca_ratio : 0;
      acc += (nwin + kTile - 1) / kTile + (cnt + kTile - 1) / kTile + (vis2 + kTile - 1) / kTile;
    }
  jobs->prefix[B * S] = acc;
  jobs->host_B = B * S;
}

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
                         const ItemList& jobs, const int* topk_idx, const int* topk_cnt, void* out,
                         float* lse_out, int num_sms, cudaStream_t st, bool pdl, bool early) {
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
  if (jobs.host_B < 0) {
    if (launch_kernel(job_prep_kernel, dim3(1), dim3(1024), 0, st, pdl, c, b, ws) < 0) return -1;
    ++n;
  }
  int grid = num_sms;
  if (jobs.host_B >= 0 && jobs.prefix[T] < grid) grid = jobs.prefix[T] > 0 ? jobs.prefix[T] : 1;
  if (launch_kernel(paged ? attn_tile_kernel<true> : attn_tile_kernel<false>, dim3(grid),
                    dim3(kA5Threads), kA5Dyn, st, pdl, qmap, jobs, c, b, ws, topk_idx, topk_cnt,
                    (pdl && early) ? 1 : 0) < 0)
    return -1;
  ++n;
  if (launch_kernel(attn_merge_kernel, dim3(T, kTcV / kMergeDims), dim3(256), 0, st, pdl, jobs, c,
                    b, ws, grid, static_cast<__nv_bfloat16*>(out), lse_out) < 0)
    return -1;
  return n + 1;
}

}  // namespace csa
