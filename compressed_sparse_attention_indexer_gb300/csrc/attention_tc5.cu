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
// one 128-row tile of one stream (window, compressed, heavy) of one query.
//   warps 5-8 gather the tile's rows with coalesced 16-byte cp.async into
//            128-byte-swizzled sub-tiles (value dims as four 32 KB pairs of
//            64-dim sub-tiles, rope dims as one 16 KB sub-tile), each thread
//            fencing its copies for the async proxy before it arrives on the
//            stage barrier; the query's 64 heads x 576 (72 KB) are loaded by
//            TMA when the query changes and stay resident;
//   warp 4   issues tcgen05 MMAs: S^T[128 rows x 64 heads] = R . Q^T over
//            576 dims (36 MMAs, M = 128, N = 64, K = 16) into TMEM; after the
//            softmax, O^T[512 dims x 64 heads] = V^T . P^T (four 128-dim
//            chunks x eight K = 16 steps, V read in place as an MN-major
//            operand, P^T from the rope slot that QK no longer needs) into
//            TMEM;
//   warps 0-3 thread r owns TMEM lane r = row r: it reads the row's 64 head
//            scores, masks rows that do not exist, and the block takes the
//            exact per-head max and sum over the tile (shuffle transposes,
//            fixed order); P^T goes to shared memory as bf16.  After PV each
//            thread reads its 128-dim slice of O^T and writes the tile's
//            normalised output (fp16) and its lse per head to the workspace.
// attn_merge_kernel: per query and head, the log-sum-exp merge of its tiles
// in fixed order (window, compressed, heavy; tiles ascending), then inverse
// RoPE on the last R dims and the bf16 store.  Because the LSE merge is
// exact, the per-tile softmax + merge equals one softmax per stream merged
// across streams.
#include <cudaTypedefs.h>
#include <stddef.h>
#include <stdlib.h>

#include "csa_internal.cuh"
#include "tc5.cuh"

namespace csa {

namespace {

constexpr int kA5Threads = 288;  // warps 0-3 softmax, 4 MMA, 5-8 row loaders
constexpr int kTile = 128;
constexpr int kSubBytes = kTile * 128;   // 128 rows x 64 dims bf16: 16 KB
constexpr int kPairBytes = 2 * kSubBytes;
constexpr int kQSub = kTcH * 128;        // 64 heads x 64 dims: 8 KB
constexpr int kNPair = 4;               // one job's value dims, 4 x 32 KB
constexpr int kQBytes = 9 * kQSub;      // the query's heads, resident: 72 KB
// the rope sub-tile slot holds P^T (64 heads x 128 rows bf16) once QK is done
constexpr int kA5Dyn = 1024 + kNPair * kPairBytes + kSubBytes + kQBytes;
constexpr float kLog2e = 1.4426950408889634f;
constexpr int kMergeHeads = 4;     // heads per merge block
constexpr int kMergeMaxJobs = 64;  // tiles per query the merge handles (else the warp-MMA path)

struct __align__(16) A5Smem {
  uint64_t pfull[kNPair], pempty[kNPair], rfull, rempty, qfull, qempty, mfull[2], mempty[2];
  uint64_t s_full, s_empty, p_full, o_full, o_empty, done;
  uint32_t tmem_base;
  int abort;
  uint32_t mask[2][4];  // per job: bit l of word w = row 32w + l exists
  alignas(16) float red[4][kTcH];
  alignas(16) float mtile[kTcH];  // read as float4
  alignas(16) float ltile[kTcH];  // read as float4
};
static_assert(offsetof(A5Smem, mtile) % 16 == 0 && offsetof(A5Smem, ltile) % 16 == 0,
              "per-head tile statistics are read with 16-byte loads");

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

__device__ __forceinline__ void gather4(uint32_t dst, const CUtensorMap* map, int x, int r0, int r1,
                                        int r2, int r3, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%2, %3, %4, %5, %6}], [%7];\n" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(r0), "r"(r1), "r"(r2), "r"(r3), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
}

// Job list: jobs of query q are [prefix[q], prefix[q+1]); in each query the
// window tiles, then the compressed tiles, then the heavy tiles.
struct JobOf {
  int q, sid, t;
};

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

__device__ __forceinline__ JobCtx job_ctx(const DevCfg& c, const DevBatch& b, int q,
                                          const int* __restrict__ topk_cnt) {
  JobCtx x;
  x.bi = q / b.S;
  x.p = query_plan(c, b.S, b.ctx_len[x.bi], q - x.bi * b.S, 0);
  int cnt = 0;
  if (!(x.p.flags & kPlanBad)) {
    cnt = topk_cnt[q];
    cnt = cnt < 0 ? 0 : (cnt > x.p.cnt ? x.p.cnt : cnt);
  }
  x.n[0] = x.p.nwin;
  x.n[1] = cnt;
  x.n[2] = x.p.vis2;
  // tiles per stream from the bound min(vis, K), as the job list counts them
  x.nt[0] = (x.p.nwin + kTile - 1) / kTile;
  x.nt[1] = (x.p.cnt + kTile - 1) / kTile;
  x.nt[2] = (x.p.vis2 + kTile - 1) / kTile;
  return x;
}

__device__ __forceinline__ void job_stream(const JobCtx& x, int local, int& sid, int& t) {
  if (local < x.nt[0]) { sid = 0; t = local; }
  else if (local < x.nt[0] + x.nt[1]) { sid = 1; t = local - x.nt[0]; }
  else { sid = 2; t = local - x.nt[0] - x.nt[1]; }
}

// Pool row of stream row i of the job, or -1 (read as zeros by the gather and
// masked by the softmax) when the row does not exist or is out of range.
__device__ __forceinline__ int job_row(const DevCfg& c, const DevBatch& b, const JobCtx& x, int q,
                                       int sid, int i, const int* __restrict__ topk_idx,
                                       int* status) {
  if (i >= x.n[sid]) return -1;
  int64_t gr;
  int64_t rows;
  if (sid == 0) {
    gr = b.raw_off[x.bi] + (x.p.pos - x.p.nwin + 1 + i);
    rows = b.raw_rows;
  } else if (sid == 1) {
    const int j = topk_idx[(int64_t)q * c.K + i];
    if (j < 0 || j >= x.p.vis) {
      set_status(status, kStatusBadIndex);
      return -1;
    }
    gr = b.cmp_off[x.bi] + j;
    rows = b.cmp_rows;
  } else {
    gr = b.hca_off[x.bi] + i;
    rows = b.hca_rows;
  }
  if (gr < 0 || gr >= rows) {
    set_status(status, kStatusBadIndex);
    return -1;
  }
  return (int)gr;
}

// Max (op 0) or sum (op 1) of each of 64 per-row values over the 32 lanes of
// a warp, by a butterfly that halves the values each step; lane l ends with
// the results for heads 2l and 2l+1 in v[0], v[1].  Fixed order.
template <int OP>
__device__ __forceinline__ void warp_transpose_reduce(float* v, int lane) {
#pragma unroll
  for (int w = 32, o = 16; o >= 1; w >>= 1, o >>= 1) {
    const bool up = (lane & o) != 0;
#pragma unroll
    for (int i = 0; i < w; ++i) {
      const float send = up ? v[i] : v[i + w];
      const float keep = up ? v[i + w] : v[i];
      const float recv = __shfl_xor_sync(0xffffffffu, send, o);
      v[i] = OP == 0 ? fmaxf(keep, recv) : (up ? recv + keep : keep + recv);
    }
  }
}

__global__ void __launch_bounds__(kA5Threads, 1)
    attn_tile_kernel(const __grid_constant__ CUtensorMap rawmap,
                     const __grid_constant__ CUtensorMap cmpmap,
                     const __grid_constant__ CUtensorMap hcamap,
                     const __grid_constant__ CUtensorMap qmap,
                     const __grid_constant__ ItemList jobs, DevCfg c, DevBatch b, Workspace ws,
                     const int* __restrict__ topk_idx, const int* __restrict__ topk_cnt) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  __shared__ A5Smem sm;
  const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
  const uint32_t pairs = base;                            // 4 x 32 KB: value dims
  const uint32_t rp = pairs + kNPair * kPairBytes;       // 16 KB: rope dims, then P^T
  const uint32_t qres = rp + kSubBytes;                  // 72 KB: the query's 64 heads
  uint8_t* rp_gen = smem_raw + (rp - smem_u32(smem_raw));

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int T = b.B * b.S;
  pdl_wait();
  const int* __restrict__ prefix = jobs.host_B >= 0 ? jobs.prefix : ws.job_prefix;
  const int N = prefix[T];
  const int lo = (int)((int64_t)blockIdx.x * N / gridDim.x);
  const int hi = (int)((int64_t)(blockIdx.x + 1) * N / gridDim.x);
  pdl_trigger();
  if (lo >= hi) return;
  volatile int* abort = &sm.abort;

  if (warp == 4) {
    tc5::tmem_alloc(smem_u32(&sm.tmem_base), 512);
    tc5::tmem_relinquish();
  }
  if (tid == 0) {
    for (int i = 0; i < kNPair; ++i) {
      tc5::mbar_init(smem_u32(&sm.pfull[i]), 128);  // every loader thread arrives
      tc5::mbar_init(smem_u32(&sm.pempty[i]), 1);
    }
    tc5::mbar_init(smem_u32(&sm.rfull), 128);
    tc5::mbar_init(smem_u32(&sm.rempty), 1);
    tc5::mbar_init(smem_u32(&sm.qfull), 1);
    tc5::mbar_init(smem_u32(&sm.qempty), 1);
    for (int i = 0; i < 2; ++i) {
      tc5::mbar_init(smem_u32(&sm.mfull[i]), 4);  // one arrival per loader warp
      tc5::mbar_init(smem_u32(&sm.mempty[i]), 128);
    }
    tc5::mbar_init(smem_u32(&sm.s_full), 1);
    tc5::mbar_init(smem_u32(&sm.s_empty), 128);
    tc5::mbar_init(smem_u32(&sm.p_full), 128);
    tc5::mbar_init(smem_u32(&sm.o_full), 1);
    tc5::mbar_init(smem_u32(&sm.o_empty), 128);
    tc5::mbar_init(smem_u32(&sm.done), 1);
    sm.abort = 0;
    tc5::fence_mbar_init();
  }
  tc5::fence_before_sync();
  __syncthreads();
  tc5::fence_after_sync();
  const uint32_t tmem = sm.tmem_base;
  const uint32_t tmem_s = tmem;          // S^T: columns [0, 64)
  const uint32_t tmem_o = tmem + 256;    // O^T: columns [256, 512), 64 per 128-dim chunk

  if (warp >= 5) {
    // ------------------------------------------------------------ row loaders
    // loader warp lw gathers rows 32lw .. 32lw+31 of each job with 16-byte
    // cp.async (two rows x 256 bytes per instruction, coalesced) into the
    // 128-byte-swizzled sub-tiles the MMAs read; each thread waits for its
    // own copies and makes them visible to the tensor core (proxy fence)
    // before arriving on the stage's barrier
    const int lw = warp - 5;
    if (lw == 0 && lane == 0) tc5::prefetch_tmap(&qmap);
    const __nv_bfloat16* null_src = static_cast<const __nv_bfloat16*>(b.q);
    int nq = 0, n = 0, cur_q = -1;
    JobCursor cur;
    cur.init(prefix, T, lo);
    bool ok = true;
    for (int job = lo; job < hi && ok && !*abort; ++job, ++n) {
      cur.advance(job);
      const int q = cur.q;
      const JobCtx x = job_ctx(c, b, q, topk_cnt);
      int sid, t;
      job_stream(x, job - cur.first, sid, t);
      const int row = 32 * lw + lane;  // this lane's row of the tile
      const int gr = job_row(c, b, x, q, sid, t * kTile + row, topk_idx, ws.status);
      const __nv_bfloat16* pool = static_cast<const __nv_bfloat16*>(
          sid == 0 ? b.raw : (sid == 1 ? b.cmp : b.hca));
      const int64_t stride = sid == 0 ? b.raw_stride : (sid == 1 ? b.cmp_stride : b.hca_stride);
      const __nv_bfloat16* my = gr >= 0 ? pool + (int64_t)gr * stride : nullptr;
      // the rows that exist, for the softmax
      const int mb = n & 1;
      if (lane == 0 && n >= 2 && !tc5::mbar_wait(smem_u32(&sm.mempty[mb]), ((n >> 1) - 1) & 1, abort))
        ok = false;
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      const uint32_t bits = __ballot_sync(0xffffffffu, gr >= 0);
      if (lane == 0) {
        sm.mask[mb][lw] = bits;
        tc5::mbar_arrive(smem_u32(&sm.mfull[mb]));
      }
      // the query's heads (TMA, 9 boxes) when the query changes
      if (q != cur_q) {
        if (lw == 0 && lane == 0) {
          if (nq > 0 && !tc5::mbar_wait(smem_u32(&sm.qempty), (nq - 1) & 1, abort)) ok = false;
          if (ok) {
            tc5::mbar_expect_tx(smem_u32(&sm.qfull), kQBytes);
            for (int k = 0; k < 9; ++k)
              tc5::tma_load_2d(qres + k * kQSub, &qmap, k * 64, q * kTcH, smem_u32(&sm.qfull));
          }
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
        ++nq;
        cur_q = q;
      }
      // issue: four pairs of 64-dim sub-tiles, then the rope sub-tile
      for (int cp = 0; cp < kNPair + 1 && ok; ++cp) {
        const bool rope = cp == kNPair;
        const uint32_t wbar = rope ? smem_u32(&sm.rempty) : smem_u32(&sm.pempty[cp]);
        if (lane == 0 && n >= 1 && !tc5::mbar_wait(wbar, (n - 1) & 1, abort)) ok = false;
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
        const uint32_t dst0 = rope ? rp : pairs + cp * kPairBytes;
        const int nch = rope ? 8 : 16;   // 16-byte chunks per row in this stage
        const int rows_per = 32 / nch;   // rows per warp instruction
        for (int j = 0; j < 32; j += rows_per) {
          const int rl = j + lane / nch;                 // row within the warp's 32
          const int ch = lane % nch;
          const __nv_bfloat16* src = reinterpret_cast<const __nv_bfloat16*>(
              __shfl_sync(0xffffffffu, reinterpret_cast<uintptr_t>(my), rl));
          const int rt = 32 * lw + rl;                   // row within the tile
          const uint32_t dst = dst0 + (ch >> 3) * kSubBytes + rt * 128 + (((ch & 7) ^ (rt & 7)) << 4);
          const int col = (rope ? 512 : cp * 128) + ch * 8;
          cp_async16(dst, src ? (const void*)(src + col) : (const void*)null_src, src ? 16 : 0);
        }
        cp_async_commit();
      }
      if (!ok) break;
      // completion, stage by stage: copies landed, visible to the async proxy
      cp_async_wait<4>();
      fence_proxy_async();
      tc5::mbar_arrive(smem_u32(&sm.pfull[0]));
      cp_async_wait<3>();
      fence_proxy_async();
      tc5::mbar_arrive(smem_u32(&sm.pfull[1]));
      cp_async_wait<2>();
      fence_proxy_async();
      tc5::mbar_arrive(smem_u32(&sm.pfull[2]));
      cp_async_wait<1>();
      fence_proxy_async();
      tc5::mbar_arrive(smem_u32(&sm.pfull[3]));
      cp_async_wait<0>();
      fence_proxy_async();
      tc5::mbar_arrive(smem_u32(&sm.rfull));
    }
    cp_async_wait<0>();
    if (lw == 0 && lane == 0 && nq > 0) tc5::mbar_wait_drain(smem_u32(&sm.qfull), (nq - 1) & 1);
  } else if (warp == 4) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idesc_s = tc5::idesc_bf16_f32(128, kTcH);
      const uint32_t idesc_o = tc5::idesc_bf16_f32(128, kTcH) | (1u << 15);  // A (V^T) MN-major
      JobCursor cur;
      cur.init(prefix, T, lo);
      int n = 0, nq = 0, cur_q = -1;
      for (int job = lo; job < hi && !*abort; ++job, ++n) {
        cur.advance(job);
        if (cur.q != cur_q) {
          if (nq > 0) tc5::mma_commit(smem_u32(&sm.qempty));  // previous query's MMAs
          if (!tc5::mbar_wait(smem_u32(&sm.qfull), nq & 1, abort)) break;
          ++nq;
          cur_q = cur.q;
        }
        if (n > 0 && !tc5::mbar_wait(smem_u32(&sm.s_empty), (n - 1) & 1, abort)) break;
        // S^T = R . Q^T over 9 sub-tiles of 64 dims
        bool ok = true;
        for (int k = 0; k < 9 && ok; ++k) {
          uint32_t rsub;
          if (k < 8) {
            if ((k & 1) == 0 && !tc5::mbar_wait(smem_u32(&sm.pfull[k >> 1]), n & 1, abort)) ok = false;
            rsub = pairs + (k >> 1) * kPairBytes + (k & 1) * kSubBytes;
          } else {
            if (!tc5::mbar_wait(smem_u32(&sm.rfull), n & 1, abort)) ok = false;
            rsub = rp;
          }
          if (!ok) break;
          tc5::fence_after_sync();
          const uint32_t qsub = qres + k * kQSub;
#pragma unroll
          for (int i = 0; i < 4; ++i)
            tc5::mma_bf16(tmem_s, tc5::sdesc_k_sw128(rsub + 32 * i),
                          tc5::sdesc_k_sw128(qsub + 32 * i), idesc_s, (k | i) ? 1u : 0u);
        }
        if (!ok) break;
        tc5::mma_commit(smem_u32(&sm.s_full));
        // O^T = V^T . P^T once the softmax has written P^T into the rope slot
        if (!tc5::mbar_wait(smem_u32(&sm.p_full), n & 1, abort)) break;
        if (n > 0 && !tc5::mbar_wait(smem_u32(&sm.o_empty), (n - 1) & 1, abort)) break;
        tc5::fence_after_sync();
        for (int cc = 0; cc < kNPair; ++cc) {
          const uint32_t vb = pairs + cc * kPairBytes;
#pragma unroll
          for (int i = 0; i < 8; ++i)
            tc5::mma_bf16(tmem_o + 64 * cc, sdesc_mn_sw128(vb + i * 2048, kSubBytes),
                          tc5::sdesc_k_sw128(rp + (i >> 2) * (kTcH * 128) + (i & 3) * 32), idesc_o,
                          i > 0 ? 1u : 0u);
          tc5::mma_commit(smem_u32(&sm.pempty[cc]));
        }
        tc5::mma_commit(smem_u32(&sm.rempty));
        tc5::mma_commit(smem_u32(&sm.o_full));
      }
      tc5::mma_commit(smem_u32(&sm.done));
      tc5::mbar_wait_drain(smem_u32(&sm.done), 0);
    }
  } else {
    // ------------------------------------------------------------ softmax + epilogue
    const int r = tid;  // row of the tile = TMEM lane
    const float sc2 = c.scale * kLog2e;
    __half* part = ws.part_o;
    float* part_lse = ws.part_lse;
    int n = 0;
    for (int job = lo; job < hi && !*abort; ++job, ++n) {
      const int mb = n & 1;
      if (!tc5::mbar_wait(smem_u32(&sm.mfull[mb]), (n >> 1) & 1, abort)) break;
      const bool valid = (sm.mask[mb][r >> 5] >> (r & 31)) & 1u;
      tc5::mbar_arrive(smem_u32(&sm.mempty[mb]));

      if (!tc5::mbar_wait(smem_u32(&sm.s_full), n & 1, abort)) break;
      tc5::fence_after_sync();
      float s[64];
      tc5::tmem_ld32x2(tmem_s + ((uint32_t)(warp * 32) << 16), s, s + 32);
      tc5::fence_before_sync();
      tc5::mbar_arrive(smem_u32(&sm.s_empty));
#pragma unroll
      for (int h = 0; h < 64; ++h) s[h] = valid ? s[h] * sc2 : -INFINITY;

      // per-head max over the 128 rows
      float v[64];
#pragma unroll
      for (int h = 0; h < 64; ++h) v[h] = s[h];
      warp_transpose_reduce<0>(v, lane);
      sm.red[warp][2 * lane] = v[0];
      sm.red[warp][2 * lane + 1] = v[1];
      named_barrier_sync(1, 128);
      if (warp == 0) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int h = 2 * lane + e;
          sm.mtile[h] = fmaxf(fmaxf(sm.red[0][h], sm.red[1][h]), fmaxf(sm.red[2][h], sm.red[3][h]));
        }
      }
      named_barrier_sync(1, 128);
      float p[64];
#pragma unroll
      for (int h4 = 0; h4 < 16; ++h4) {
        const float4 m4 = reinterpret_cast<const float4*>(sm.mtile)[h4];
        const float mm[4] = {m4.x, m4.y, m4.z, m4.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int h = h4 * 4 + e;
          p[h] = mm[e] == -INFINITY ? 0.f : exp2f(s[h] - mm[e]);
        }
      }
      // per-head sum over the rows (fixed order: butterfly, then warps 0..3)
#pragma unroll
      for (int h = 0; h < 64; ++h) v[h] = p[h];
      warp_transpose_reduce<1>(v, lane);
      sm.red[warp][2 * lane] = v[0];
      sm.red[warp][2 * lane + 1] = v[1];
      // P^T (bf16) into the rope slot, whose QK reads are complete (s_full):
      // the K-major B operand [64-row sub-tile][head][64 rows]
      {
        uint8_t* pt = rp_gen + (r >> 6) * (kTcH * 128);
        const int rr = r & 63;
#pragma unroll
        for (int h = 0; h < 64; ++h)
          *reinterpret_cast<__nv_bfloat16*>(pt + h * 128 + ((((rr >> 3) ^ (h & 7)) << 4)) +
                                            (rr & 7) * 2) = __float2bfloat16_rn(p[h]);
      }
      fence_proxy_async();
      named_barrier_sync(1, 128);
      if (warp == 0) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int h = 2 * lane + e;
          sm.ltile[h] = ((sm.red[0][h] + sm.red[1][h]) + sm.red[2][h]) + sm.red[3][h];
        }
      }
      tc5::mbar_arrive(smem_u32(&sm.p_full));
      named_barrier_sync(1, 128);

      // epilogue: normalised tile output (fp16) and lse (log2 units) per head
      if (!tc5::mbar_wait(smem_u32(&sm.o_full), n & 1, abort)) break;
      tc5::fence_after_sync();
      float inv[64];
#pragma unroll
      for (int h4 = 0; h4 < 16; ++h4) {
        const float4 l4 = reinterpret_cast<const float4*>(sm.ltile)[h4];
        inv[h4 * 4 + 0] = l4.x > 0.f ? 1.f / l4.x : 0.f;
        inv[h4 * 4 + 1] = l4.y > 0.f ? 1.f / l4.y : 0.f;
        inv[h4 * 4 + 2] = l4.z > 0.f ? 1.f / l4.z : 0.f;
        inv[h4 * 4 + 3] = l4.w > 0.f ? 1.f / l4.w : 0.f;
      }
      __half* pj = part + (int64_t)job * kTcH * kTcV;
      for (int cc = 0; cc < 4; ++cc) {
        float o[64];
        tc5::tmem_ld32x2(tmem_o + 64 * cc + ((uint32_t)(warp * 32) << 16), o, o + 32);
        const int vcol = cc * 128 + r;
#pragma unroll
        for (int h = 0; h < 64; ++h) pj[h * kTcV + vcol] = __float2half_rn(o[h] * inv[h]);
      }
      tc5::fence_before_sync();
      tc5::mbar_arrive(smem_u32(&sm.o_empty));
      if (warp == 0) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int h = 2 * lane + e;
          const float l = sm.ltile[h];
          part_lse[(int64_t)job * kTcH + h] = l > 0.f ? sm.mtile[h] + log2f(l) : -INFINITY;
        }
      }
    }
  }

  if (tid == 0 && *abort) set_status(ws.status, kStatusTimeout);
  tc5::fence_before_sync();
  __syncthreads();
  tc5::fence_after_sync();
  if (warp == 4) tc5::tmem_dealloc(tmem, 512);
}

// Per (query, 16 heads): LSE merge of the query's tiles in job order, inverse
// RoPE, bf16 store.  The tiles' lse values are staged in shared memory and
// turned into merge weights once; thread t then owns output dims 2t, 2t+1 and
// reads the partials of all tiles for a head at once.
__global__ void __launch_bounds__(256)
    attn_merge_kernel(const __grid_constant__ ItemList jobs, DevCfg c, DevBatch b, Workspace ws,
                      __nv_bfloat16* __restrict__ out, float* __restrict__ lse_out) {
  __shared__ float wgt[kMergeMaxJobs][kMergeHeads];
  __shared__ float Mh[kMergeHeads], tot[kMergeHeads];
  pdl_wait();
  pdl_trigger();
  const int q = blockIdx.x, hg = blockIdx.y, t = threadIdx.x;
  const int* __restrict__ prefix = jobs.host_B >= 0 ? jobs.prefix : ws.job_prefix;
  const int j0 = prefix[q];
  const int nj = min(prefix[q + 1] - j0, kMergeMaxJobs);
  for (int e = t; e < nj * kMergeHeads; e += blockDim.x) {
    const int j = e / kMergeHeads, hh = e - j * kMergeHeads;
    wgt[j][hh] = ws.part_lse[(int64_t)(j0 + j) * kTcH + hg * kMergeHeads + hh];
  }
  __syncthreads();
  if (t < kMergeHeads) {
    float M = -INFINITY;
    for (int j = 0; j < nj; ++j) M = fmaxf(M, wgt[j][t]);
    float sum = 0.f;
    for (int j = 0; j < nj; ++j) {
      const float wj = M == -INFINITY ? 0.f : exp2f(wgt[j][t] - M);
      wgt[j][t] = wj;
      sum += wj;
    }
    Mh[t] = M;
    tot[t] = sum;
  }
  __syncthreads();
  const int bi = q / b.S;
  const QueryPlan p = query_plan(c, b.S, b.ctx_len[bi], q - bi * b.S, 0);
  const int v = 2 * t;
  float acc0[kMergeHeads], acc1[kMergeHeads];
#pragma unroll
  for (int hh = 0; hh < kMergeHeads; ++hh) acc0[hh] = acc1[hh] = 0.f;
  float cs = 1.f, sn = 0.f;
  if (v >= kTcV - c.R && !(p.flags & kPlanBad)) {
    const float2 r = rope_cos_sin((double)p.pos, c.rope_theta[(v - (kTcV - c.R)) >> 1]);
    cs = r.x;
    sn = r.y;
  }
  const __half* pbase = ws.part_o + ((int64_t)j0 * kTcH + hg * kMergeHeads) * kTcV + v;
  // all tiles' partials of the block's heads are loaded before any is used
  constexpr int kJ = 8;
  for (int jb = 0; jb < nj; jb += kJ) {
    __half2 o2[kMergeHeads][kJ];
#pragma unroll
    for (int hh = 0; hh < kMergeHeads; ++hh)
#pragma unroll
      for (int k = 0; k < kJ; ++k)
        o2[hh][k] = jb + k < nj ? *reinterpret_cast<const __half2*>(
                                      pbase + ((int64_t)(jb + k) * kTcH + hh) * kTcV)
                                : __floats2half2_rn(0.f, 0.f);
#pragma unroll
    for (int hh = 0; hh < kMergeHeads; ++hh) {
#pragma unroll
      for (int k = 0; k < kJ; ++k) {
        if (jb + k < nj) {
          acc0[hh] = fmaf(wgt[jb + k][hh], __low2float(o2[hh][k]), acc0[hh]);
          acc1[hh] = fmaf(wgt[jb + k][hh], __high2float(o2[hh][k]), acc1[hh]);
        }
      }
    }
  }
#pragma unroll
  for (int hh = 0; hh < kMergeHeads; ++hh) {
    const float it = tot[hh] > 0.f ? 1.f / tot[hh] : 0.f;
    const float x0 = acc0[hh] * it, x1 = acc1[hh] * it;
    const int h = hg * kMergeHeads + hh;
    const float y0 = x0 * cs + x1 * sn, y1 = -x0 * sn + x1 * cs;
    *reinterpret_cast<uint32_t*>(out + ((int64_t)q * kTcH + h) * kTcV + v) = pack_bf16x2(y0, y1);
    if (lse_out && t == 0)
      lse_out[(int64_t)q * kTcH + h] =
          Mh[hh] == -INFINITY ? -INFINITY : (Mh[hh] + log2f(tot[hh])) * 0.6931471805599453f;
  }
}

// Counts each query's tiles into ws.job_prefix when the host has no lengths.
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

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult r;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &r) ==
            cudaSuccess &&
        r == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

bool make_map(CUtensorMap* m, const void* ptr, uint64_t rows, uint64_t stride, uint32_t box_rows) {
  auto fn = encode_fn();
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
                         float* lse_out, int num_sms, cudaStream_t st, bool pdl) {
  const int T = b.B * b.S;
  if (T == 0) return 0;
  if (!ws.part_o || max_jobs_per_query(c) > kMergeMaxJobs || b.raw_rows > 0x7fffffffLL || b.cmp_rows > 0x7fffffffLL ||
      b.hca_rows > 0x7fffffffLL || (int64_t)T * kTcH > 0x7fffffffLL)
    return -2;
  CUtensorMap rawmap, cmpmap, hcamap, qmap;
  if (!make_map(&rawmap, b.raw, (uint64_t)(b.raw_rows > 0 ? b.raw_rows : 1), b.raw_stride, 1)) return -1;
  if (!make_map(&cmpmap, b.cmp, (uint64_t)(b.cmp_rows > 0 ? b.cmp_rows : 1), b.cmp_stride, 1)) return -1;
  if (c.hca_ratio > 0) {
    if (!make_map(&hcamap, b.hca, (uint64_t)(b.hca_rows > 0 ? b.hca_rows : 1), b.hca_stride, 1)) return -1;
  } else {
    hcamap = cmpmap;
  }
  if (!make_map(&qmap, b.q, (uint64_t)T * kTcH, kTcD, kTcH)) return -1;
  static bool attr = false;
  if (!attr) {
    cudaFuncSetAttribute(attn_tile_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kA5Dyn);
    attr = true;
  }
  int n = 0;
  if (jobs.host_B < 0) {
    if (launch_kernel(job_prep_kernel, dim3(1), dim3(1024), 0, st, pdl, c, b, ws) < 0) return -1;
    ++n;
  }
  int grid = num_sms;
  if (jobs.host_B >= 0 && jobs.prefix[T] < grid) grid = jobs.prefix[T] > 0 ? jobs.prefix[T] : 1;
  if (launch_kernel(attn_tile_kernel, dim3(grid), dim3(kA5Threads), kA5Dyn, st, pdl, rawmap, cmpmap,
                    hcamap, qmap, jobs, c, b, ws, topk_idx, topk_cnt) < 0)
    return -1;
  ++n;
  if (launch_kernel(attn_merge_kernel, dim3(T, kTcH / kMergeHeads), dim3(256), 0, st, pdl, jobs, c, b, ws,
                    static_cast<__nv_bfloat16*>(out), lse_out) < 0)
    return -1;
  return n + 1;
}

}  // namespace csa
