// Step (b): exact Top-K of each query's indexer scores, ties to the lower
// index, output in ascending index order and -1 padded; the bypass takes
// every visible row when vis <= K.  hw-native-sys/pypto-lib "Perf: skip
// redundant CSA scoring and fuse gather unpack" (bounded Top-K indices,
// bypass) and "Fix: port the DeepSeek-V4 MoE, hc_pre and prefill fixes to
// DSpark" (a staged sort that stops at 256 picks wrong keys past 256: the
// selection here is exact at any width).
//
// One 1024-thread block per query, in one of two kernels: topk_reg_kernel
// (below) keeps a row of up to 16384 keys in registers and resolves the last
// candidates by ranking them; topk_kernel, for longer rows, works as follows.
// Scores become order-preserving 32-bit
// keys in shared memory (-0.0 folded onto +0.0, NaN below every number).  The
// bits above the highest bit on which the keys differ are skipped; then
// radix-select passes of up to 11 bits each build a histogram of the next
// digit among keys that still match the prefix (shared-memory integer
// atomics: counts, so the result is order independent) and pick the
// digit holding the K-th largest key.  The passes stop as soon as the digit's
// keys are exactly the ones still needed.  A final pass over contiguous index
// ranges keeps every key above the prefix and the lowest-index keys equal to
// it, and writes them in ascending index order through two block scans.
#include "csa_internal.cuh"
#include "ptx.cuh"

namespace csa {

namespace {

constexpr int kTopkThreads = 1024;
constexpr int kBins = 2048;
// dynamic shared memory of topk_kernel at the longest row a config may have
// (max_context / ratio <= 40960 keys, one pad word per 16)
constexpr int kMaxRowKeys = 40960;
constexpr int kTopkSmemMax = (kMaxRowKeys + kMaxRowKeys / 16 + 1) * 4;

__device__ __forceinline__ uint32_t score_key(float f) {
  uint32_t u = __float_as_uint(f);
  if ((u & 0x7fffffffu) > 0x7f800000u) return 0u;  // NaN: lowest
  if (u == 0x80000000u) u = 0u;                   // -0.0 == +0.0
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}


// Publishes a query's Top-K output to the attention kernel of the same step,
// which may already be running (it waits for the flag with bounded polls):
// the block meets (the barrier orders every thread's output stores before
// thread 0's release, which is cumulative over what the barrier ordered
// before it), and one thread stores the step's epoch with release semantics.
// A no-op without a flag array.
__device__ __forceinline__ void signal_ready(int* ready, int q, int epoch) {
  if (!ready) return;
  __syncthreads();
  if (threadIdx.x == 0) {
    asm volatile("st.release.gpu.global.b32 [%0], %1;\n" ::"l"(ready + q), "r"(epoch) : "memory");
  }
}

// Waits until the indexer of the same call has published `target` scored
// items of request bi in done[bi] (thread 0 polls with acquire loads,
// bounded: a wait that gives up records CSA_ERR_TIMEOUT and the block goes
// on), then the block meets, so that every thread's score loads follow it.
__device__ __forceinline__ void wait_request_scored(const int* done, int bi, int target, int* status,
                                                    int polls) {
  if (threadIdx.x == 0) {
    const uint32_t limit = polls < 0 ? (1u << 23) : (uint32_t)polls;
    uint32_t i = 0, ns = 32;
    while (true) {
      int v;
      asm volatile("ld.acquire.gpu.global.b32 %0, [%1];\n" : "=r"(v) : "l"(done + bi) : "memory");
      if (v >= target) break;
      if (++i >= limit) {
        set_status(status, kStatusTimeout);
        break;
      }
      if (i >= 8) {
        __nanosleep(ns);
        ns = ns * 2 > 256 ? 256 : ns * 2;
      }
    }
  }
  __syncthreads();
}

// Block-wide exclusive scan of one int per thread with a single barrier: each
// warp scans the per-warp sums itself.  `warp_tmp` (>= 32 ints) is written
// before the barrier and read after it, so consecutive calls alternate two
// buffers (a call's barrier then separates the reads of one use of a buffer
// from the writes of its next use).  *total receives the block sum.
__device__ __forceinline__ int block_exclusive_scan1(int v, int* warp_tmp, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nwarps = blockDim.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_tmp[warp] = x;
  __syncthreads();
  int t = lane < nwarps ? warp_tmp[lane] : 0;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, t, o);
    if (lane >= o) t += y;
  }
  const int base = __shfl_sync(0xffffffffu, t, (warp + 31) & 31);  // inclusive sum of warps < warp
  *total = __shfl_sync(0xffffffffu, t, 31);
  return (warp > 0 ? base : 0) + x - v;
}

// Key i lives at keys[kpad(i)]: one pad word per 16 keys, so the final pass
// (thread t reads keys 16t .. 16t+15) hits 32 different banks.
__device__ __forceinline__ int kpad(int i) { return i + (i >> 4); }

__global__ void __launch_bounds__(kTopkThreads, 1)
    topk_kernel(DevCfg c, DevBatch b, const float* __restrict__ scores, int64_t ld,
                const int* __restrict__ n_override, int* __restrict__ idx_out,
                int* __restrict__ cnt_out, int* __restrict__ status, int max_vis, int* ready,
                int epoch) {
  extern __shared__ __align__(16) uint32_t keys[];
  __shared__ int hist[kBins];
  __shared__ int scan_tmp[33];
  __shared__ uint32_t s_or;
  __shared__ int s_bin, s_above;

  const int K = c.K;
  const int q = blockIdx.x, tid = threadIdx.x, lane = tid & 31;
  pdl_wait();
  pdl_trigger();
  int n;
  bool do_select;
  if (n_override) {
    n = n_override[q];
    if (n < 0 || n > max_vis || (int64_t)n > ld) {  // never read past the caller's row
      if (tid == 0) set_status(status, kStatusBadIndex);
      n = 0;
    }
    do_select = n > K;
  } else {
    const int bi = q / b.S;
    const QueryPlan p = query_plan(c, b.S, b.ctx_len[bi], q - bi * b.S, 0);
    if ((p.flags & kPlanBad) && tid == 0) set_status(status, kStatusBadIndex);
    n = p.vis;
    do_select = n > K;  // vis > K: scored; otherwise the bypass
  }
  int* out = idx_out + (int64_t)q * K;
  if (!do_select) {  // bypass: every visible row
    for (int i = tid; i < K; i += kTopkThreads) out[i] = i < n ? i : -1;
    if (tid == 0) cnt_out[q] = n < K ? n : K;
    signal_ready(ready, q, epoch);
    return;
  }
  const float* sc = scores + (int64_t)q * ld;
  if (tid == 0) s_or = 0u;
  __syncthreads();
  // keys, and the OR of (key ^ key0): its top set bit is the highest bit on
  // which the keys differ
  const uint32_t k0 = score_key(sc[0]);
  uint32_t acc_or = 0u;
  for (int base = 0; base < n; base += 8 * kTopkThreads) {
    float v[8];  // eight loads in flight per thread
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int i = base + j * kTopkThreads + tid;
      v[j] = i < n ? __ldg(sc + i) : 0.f;
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int i = base + j * kTopkThreads + tid;
      if (i < n) {
        const uint32_t k = score_key(v[j]);
        keys[kpad(i)] = k;
        acc_or |= k ^ k0;
      }
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc_or |= __shfl_xor_sync(0xffffffffu, acc_or, o);
  if (lane == 0 && acc_or) atomicOr(&s_or, acc_or);
  __syncthreads();
  const uint32_t diff = s_or;

  int start = diff ? 32 - __clz(diff) : 0;  // bits [start, 32) are common to all keys
  uint32_t prefix = start < 32 ? (k0 >> start) : 0u;
  int need = K;
  const int rounds = (n + kTopkThreads - 1) / kTopkThreads;
  while (start > 0) {
    const int wbits = start < 11 ? start : 11;
    const int sh = start - wbits;
    const uint32_t mask = (1u << wbits) - 1u;
    for (int i = tid; i < kBins; i += kTopkThreads) hist[i] = 0;
    __syncthreads();
    for (int r = 0; r < rounds; ++r) {
      const int i = r * kTopkThreads + tid;
      if (i < n) {
        const uint32_t k = keys[kpad(i)];
        if ((start >= 32) || ((k >> start) == prefix)) atomicAdd(&hist[(k >> sh) & mask], 1);
      }
    }
    __syncthreads();
    // the digit holding the need-th largest key: suffix sums over bins
    {
      const int b0 = 2 * tid, b1 = 2 * tid + 1;
      const int h0 = hist[b0], h1 = hist[b1];
      // exclusive scan over threads in reverse order = count of keys in higher bins
      const int rv = h0 + h1;
      int tot;
      // reverse: thread tid gets the sum over threads > tid
      const int ex_rev = block_exclusive_scan(rv, scan_tmp, &tot);  // sum over threads < tid
      const int above_t = tot - ex_rev - rv;                          // sum over threads > tid
      if (above_t < need && above_t + rv >= need) {
        if (above_t + h1 >= need) {
          s_bin = b1;
          s_above = above_t;
        } else {
          s_bin = b0;
          s_above = above_t + h1;
        }
      }
    }
    __syncthreads();
    const int bin = s_bin;
    need -= s_above;
    prefix = (start >= 32 ? 0u : (prefix << wbits)) | (uint32_t)bin;
    start = sh;
    const int in_bin = hist[bin];
    __syncthreads();
    if (in_bin == need) break;  // all keys of this digit are kept
  }

  // final selection over contiguous ranges, ascending index order
  const int per = (n + kTopkThreads - 1) / kTopkThreads;
  const int i0 = tid * per, i1 = min(n, i0 + per);
  int gt = 0, eq = 0;
  for (int i = i0; i < i1; ++i) {
    const uint32_t hk = start >= 32 ? 0u : (keys[kpad(i)] >> start);
    gt += hk > prefix;
    eq += hk == prefix;
  }
  int tot;
  const int eq_before = block_exclusive_scan(eq, scan_tmp, &tot);
  int eq_take = need - eq_before;
  eq_take = eq_take < 0 ? 0 : (eq_take > eq ? eq : eq_take);
  const int pos0 = block_exclusive_scan(gt + eq_take, scan_tmp, &tot);
  int pos = pos0, taken_eq = 0;
  for (int i = i0; i < i1; ++i) {
    const uint32_t hk = start >= 32 ? 0u : (keys[kpad(i)] >> start);
    bool sel = hk > prefix;
    if (hk == prefix && taken_eq < eq_take) {
      sel = true;
      ++taken_eq;
    }
    if (sel) out[pos++] = i;
  }
  if (tid == 0) cnt_out[q] = K;
  signal_ready(ready, q, epoch);
}

// Register-resident variant for rows of at most kJ * 1024 keys (the common
// case: max_context / ratio <= 16384).  Thread t holds the kJ consecutive
// keys kJ t .. kJ t + kJ - 1 in registers for the whole selection (kJ = 16,
// or kJ = 2 for rows of at most 2048 keys: short contexts, prefill chunks,
// whose smaller register footprint fits two blocks per SM), so the block's
// threads and each thread's keys are both in index order.  The result is
// defined by a threshold pair (tkey, tidx): the K-th entry in the order (key
// descending, index ascending); a key is selected iff it precedes or is that
// entry.
//   1. radix passes as above (histogram of the next digit among keys that
//      match the prefix), until the digit's keys are exactly the ones needed
//      (threshold = the digit's lowest key, any index) or few enough to rank
//      directly;
//   2. ranking: the <= 1024 candidates left are compacted into shared memory
//      and each candidate's rank among them is counted by one thread; rank
//      need - 1 is the threshold;
//   3. keys all equal and more than 1024 of them straddle the threshold: the
//      threshold index is the need-th of them in index order (a block scan of
//      the per-thread counts);
//   4. output: a block scan of the per-thread counts of selected keys gives
//      each thread its first output position; it writes its selected indices
//      there in order, so the output is in ascending index order.
constexpr int kRegKeys = 16;  // keys per thread of the long-row instantiation
constexpr int kRegMax = kRegKeys * kTopkThreads;
constexpr int kShortKeys = 2;  // keys per thread of the short-row one
constexpr int kCand = kTopkThreads;  // candidates ranked directly

// A global load issued exactly where it is written (asm volatile): the value
// then lives in a register (or is spilled) for the rest of the kernel,
// instead of a read-only load that the compiler may issue again at a later
// use when registers are scarce.
__device__ __forceinline__ float ld_once(const float* p) {
  float v;
  asm volatile("ld.global.cg.f32 %0, [%1];\n" : "=f"(v) : "l"(p) : "memory");
  return v;
}
// The same for two and four consecutive floats.
__device__ __forceinline__ float4 ld_once4(const float* p) {
  float4 v;
  asm volatile("ld.global.cg.v4.f32 {%0, %1, %2, %3}, [%4];\n"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "l"(p)
               : "memory");
  return v;
}
__device__ __forceinline__ float2 ld_once2(const float* p) {
  float2 v;
  asm volatile("ld.global.cg.v2.f32 {%0, %1}, [%2];\n" : "=f"(v.x), "=f"(v.y) : "l"(p) : "memory");
  return v;
}

template <int kJ>
__global__ void __launch_bounds__(kTopkThreads, kJ <= kShortKeys ? 2 : 1)
    topk_reg_kernel(DevCfg c, DevBatch b, const float* __restrict__ scores, int64_t ld,
                    const int* __restrict__ n_override, int* __restrict__ idx_out,
                    int* __restrict__ cnt_out, int* __restrict__ status, int max_vis,
                    int early, int* ready, int epoch, const int* __restrict__ done, int qsplit,
                    int keys) {
  static_assert(kJ == 2 || kJ % 4 == 0, "keys are loaded as float2 or float4 vectors");
  constexpr uint32_t kFull = (1u << kJ) - 1u;  // every key of the thread exists
  __shared__ int hist[kBins];
  __shared__ uint32_t cand_key[kCand];
  __shared__ int cand_idx[kCand];
  __shared__ int scan_tmp[2][32];  // alternating buffers of block_exclusive_scan1
  __shared__ uint32_t warp_or[32], warp_and[32];
  __shared__ uint32_t s_tkey;
  __shared__ int s_ncand, s_tidx;

  const int K = c.K;
  const int q = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // The row length from the plan.  Launched right after this library's own
  // kernel of the same call (early != 0), which waits for its predecessor
  // before it lets this grid launch, the lengths (the caller's inputs) are
  // complete already, so only the scores wait.
  int n = 0, len = 0;
  bool bad = false;
  auto plan_len = [&] {
    const int bi = q / b.S;
    len = b.ctx_len[bi];
    const QueryPlan p = query_plan(c, b.S, len, q - bi * b.S, 0);
    bad = p.flags & kPlanBad;
    n = p.vis;
  };
  // With the indexer's per-request counters (done), a block waits for its
  // request's scores only, and for the indexer grid at its end (so that this
  // grid still completes after it)
  const bool by_request = done && early && !n_override;
  if (!n_override && early) plan_len();
  if (!by_request) pdl_wait();
  pdl_trigger();
  bool do_select;
  if (n_override) {
    n = n_override[q];
    if (n < 0 || n > max_vis || (int64_t)n > ld) {  // never read past the caller's row
      if (tid == 0) set_status(status, kStatusBadIndex);
      n = 0;
    }
  } else {
    if (!early) plan_len();
    if (bad && tid == 0) set_status(status, kStatusBadIndex);
  }
  if (n > kJ * kTopkThreads) {  // the launcher picks this kernel only for rows that fit
    if (tid == 0) set_status(status, kStatusBadIndex);
    n = 0;
  }
  do_select = n > K;  // vis > K: scored; otherwise the bypass
  int* out = idx_out + (int64_t)q * K;
  if (!do_select) {  // bypass: every visible row
    for (int i = tid; i < K; i += kTopkThreads) out[i] = i < n ? i : -1;
    if (tid == 0) cnt_out[q] = n < K ? n : K;
    signal_ready(ready, q, epoch);
    if (by_request) pdl_wait();
    return;
  }
  if (by_request) wait_request_scored(done, q / b.S, request_items(c, b.S, len, 0, qsplit), status, c.wait_polls);
  const float* sc = scores + (int64_t)q * ld;
  if (tid == 0) s_ncand = 0;
  // this thread's keys (all loads in flight at once), and the OR / AND over
  // the row: bits where they differ are the ones still to decide
  const int i0 = tid * kJ;
  uint32_t k[kJ];
  uint32_t vmask = 0u, aor = 0u, aand = ~0u;
  {
    float v[kJ];
    const bool vec = ((reinterpret_cast<uintptr_t>(sc) & (kJ == 2 ? 7u : 15u)) == 0) && i0 + kJ <= n;
    if (vec) {  // every key of this thread exists: no per-key checks
      if (kJ == 2) {
        const float2 x = ld_once2(sc + i0);
        v[0] = x.x;
        v[1] = x.y;
      } else {
#pragma unroll
        for (int j = 0; j < kJ; j += 4) {
          const float4 x = ld_once4(sc + i0 + j);
          v[j] = x.x;
          v[j + 1] = x.y;
          v[j + 2] = x.z;
          v[j + 3] = x.w;
        }
      }
#pragma unroll
      for (int j = 0; j < kJ; ++j) {
        k[j] = keys ? __float_as_uint(v[j]) : score_order_key(v[j]);
        aor |= k[j];
        aand &= k[j];
      }
      vmask = kFull;
    } else {
#pragma unroll
      for (int j = 0; j < kJ; ++j) v[j] = i0 + j < n ? ld_once(sc + i0 + j) : 0.f;
#pragma unroll
      for (int j = 0; j < kJ; ++j) {
        k[j] = keys ? __float_as_uint(v[j]) : score_order_key(v[j]);
        if (i0 + j < n) {
          vmask |= 1u << j;
          aor |= k[j];
          aand &= k[j];
        }
      }
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    aor |= __shfl_xor_sync(0xffffffffu, aor, o);
    aand &= __shfl_xor_sync(0xffffffffu, aand, o);
  }
  if (lane == 0) {
    warp_or[warp] = aor;
    warp_and[warp] = aand;
  }
  // the first radix pass's histogram is cleared under the same barrier
  hist[tid] = 0;
  hist[tid + kTopkThreads] = 0;
  __syncthreads();
  aor = warp_or[lane];
  aand = warp_and[lane];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    aor |= __shfl_xor_sync(0xffffffffu, aor, o);
    aand &= __shfl_xor_sync(0xffffffffu, aand, o);
  }
  const uint32_t diff = aor & ~aand;

  int start = diff ? 32 - __clz(diff) : 0;  // bits [start, 32) are common to all keys
  uint32_t prefix = start < 32 ? (aor >> start) : 0u;
  int need = K, in_bin = n;
  uint32_t tkey = 0u;
  int tidx = 0;
  int mode = 0;  // 1: threshold known, 2: rank the candidates, 0: equal keys
  int sb = 0;    // scan buffer of the last block_exclusive_scan1
  for (bool first_pass = true; start > 0; first_pass = false) {
    const int wbits = start < 11 ? start : 11;
    const int sh = start - wbits;
    const uint32_t mask = (1u << wbits) - 1u;
    if (!first_pass) {
      hist[tid] = 0;
      hist[tid + kTopkThreads] = 0;
      __syncthreads();
    }
    if (first_pass) {  // every key shares the common prefix
      if (vmask == kFull) {
#pragma unroll
        for (int j = 0; j < kJ; ++j) atomicAdd(&hist[(k[j] >> sh) & mask], 1);
      } else if (vmask) {
#pragma unroll
        for (int j = 0; j < kJ; ++j)
          if ((vmask >> j) & 1u) atomicAdd(&hist[(k[j] >> sh) & mask], 1);
      }
    } else {  // start < 32 after a pass
#pragma unroll
      for (int j = 0; j < kJ; ++j)
        if (((vmask >> j) & 1u) && (k[j] >> start) == prefix) atomicAdd(&hist[(k[j] >> sh) & mask], 1);
    }
    __syncthreads();
    // the digit holding the need-th largest key, found by every warp alike
    // after one barrier: warp w's lanes hold bins 64 w .. 64 w + 63 (two
    // each); the warps' totals go through shared memory, then each warp
    // finds the warp w* whose bins hold the key (keys in higher warps' bins
    // fewer than need, with w*'s at least need), and within w* the lane and
    // the bin, from suffix sums
    int bin, above;
    {
      int wt = hist[2 * tid] + hist[2 * tid + 1];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) wt += __shfl_xor_sync(0xffffffffu, wt, o);
      int* wsum = scan_tmp[sb ^= 1];
      if (lane == 0) wsum[warp] = wt;
      __syncthreads();
      static_assert(kTopkThreads == 32 * 32, "one warp total per lane: 32 warps of 64 bins");
      const int ws = wsum[lane];
      int suf = ws;               // keys in the bins of warps >= lane
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_down_sync(0xffffffffu, suf, o);
        if (lane + o < 32) suf += y;
      }
      const int wabove = suf - ws;
      const uint32_t wb = __ballot_sync(0xffffffffu, wabove < need && suf >= need);
      const int wstar = wb ? __ffs(wb) - 1 : 0;  // (never 0: need <= the keys left)
      const int above_w = __shfl_sync(0xffffffffu, wabove, wstar);
      const int g0 = hist[64 * wstar + 2 * lane], g1 = hist[64 * wstar + 2 * lane + 1];
      const int r = g0 + g1;
      int sr = r;  // keys in the pairs of lanes >= lane of warp w*
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_down_sync(0xffffffffu, sr, o);
        if (lane + o < 32) sr += y;
      }
      const int above_l = above_w + sr - r;
      const uint32_t lb = __ballot_sync(0xffffffffu, above_l < need && above_l + r >= need);
      const int ls = lb ? __ffs(lb) - 1 : 0;
      const int al = __shfl_sync(0xffffffffu, above_l, ls);
      const int h1s = __shfl_sync(0xffffffffu, g1, ls);
      if (al + h1s >= need) {
        bin = 64 * wstar + 2 * ls + 1;
        above = al;
      } else {
        bin = 64 * wstar + 2 * ls;
        above = al + h1s;
      }
    }
    need -= above;
    prefix = (start >= 32 ? 0u : (prefix << wbits)) | (uint32_t)bin;
    start = sh;
    in_bin = hist[bin];
    if (in_bin == need) {  // every key of the digit is kept
      tkey = prefix << start;
      tidx = 0x7fffffff;
      mode = 1;
      break;
    }
    if (in_bin <= kCand) {
      mode = 2;
      break;
    }
    __syncthreads();  // hist is cleared and rewritten by the next pass
  }
  if (mode == 0 && in_bin <= kCand) mode = 2;

  if (mode == 2) {
    // compact the keys that match the prefix (this thread's, contiguous
    // slots), then rank each among them
    uint32_t m = 0u;
#pragma unroll
    for (int j = 0; j < kJ; ++j) m |= (uint32_t)((k[j] >> start) == prefix) << j;  // start < 32 here
    m &= vmask;
    if (m) {
      int slot = atomicAdd(&s_ncand, __popc(m));
      // the set bits only (a thread has few candidates); k[] stays in
      // registers: the key is picked by a fixed-index select
      for (uint32_t mm = m; mm; mm &= mm - 1u, ++slot) {
        const int j = __ffs(mm) - 1;
        uint32_t kj = 0u;
#pragma unroll
        for (int jj = 0; jj < kJ; ++jj) kj = jj == j ? k[jj] : kj;
        if (slot < kCand) {
          cand_key[slot] = kj;
          cand_idx[slot] = i0 + j;
        }
      }
    }
    __syncthreads();
    if (tid < in_bin) {
      const uint32_t kk = cand_key[tid];
      const int ii = cand_idx[tid];
      int rank = 0;
      for (int x = 0; x < in_bin; ++x) {
        const uint32_t kx = cand_key[x];
        rank += (kx > kk) || (kx == kk && cand_idx[x] < ii);
      }
      if (rank == need - 1) {
        s_tkey = kk;
        s_tidx = ii;
      }
    }
    __syncthreads();
    tkey = s_tkey;
    tidx = s_tidx;
  } else if (mode == 0) {
    // start == 0: more than kCand keys equal `prefix` and `need` of them are
    // kept, the lowest indices first: the thread holding the need-th of them
    // in index order finds it among its keys
    int eq = 0;
#pragma unroll
    for (int j = 0; j < kJ; ++j) eq += (((vmask >> j) & 1u) && k[j] == prefix) ? 1 : 0;
    int tot;
    const int ex = block_exclusive_scan1(eq, scan_tmp[sb ^= 1], &tot);
    if (ex < need && ex + eq >= need) {
      int r = ex;
#pragma unroll
      for (int j = 0; j < kJ; ++j)
        if (((vmask >> j) & 1u) && k[j] == prefix && ++r == need) s_tidx = i0 + j;
    }
    __syncthreads();
    tkey = prefix;
    tidx = s_tidx;
  }

  // selection: keys before the threshold in (key desc, index asc) order;
  // a block scan of the per-thread counts gives each thread its output slot
  uint32_t smask = 0u;
#pragma unroll
  for (int j = 0; j < kJ; ++j) {
    const bool sel = k[j] > tkey || (k[j] == tkey && i0 + j <= tidx);
    smask |= (uint32_t)sel << j;
  }
  smask &= vmask;  // keys past the row are never kept
  int tot;
  int pos = block_exclusive_scan1(__popc(smask), scan_tmp[sb ^= 1], &tot);
  for (uint32_t mm = smask; mm; mm &= mm - 1u, ++pos)  // the set bits only
    if (pos < K) out[pos] = i0 + __ffs(mm) - 1;
  if (tid == 0) cnt_out[q] = K;
  signal_ready(ready, q, epoch);
  if (by_request) pdl_wait();
}

}  // namespace

// The register kernel when every row fits it (CSA_TOPK=radix keeps the
// shared-memory kernel, its measured baseline).
bool topk_use_reg(int max_vis) {
  static const bool forced = [] {
    const char* e = getenv("CSA_TOPK");
    return e && e[0] == 'r';
  }();
  return !forced && max_vis <= kRegMax;
}

int launch_topk(const DevCfg& c, const DevBatch* b, int nq, const float* scores, int64_t ld,
                const int* n_override, int* idx_out, int* cnt_out, int* status, int max_vis,
                cudaStream_t st, bool pdl, bool early, int* ready, int epoch, const int* done,
                int qsplit, bool keys) {
  if (nq == 0) return 0;
  DevBatch none = {};
  none.S = 1;
  if (topk_use_reg(max_vis))
    return launch_kernel(max_vis <= kShortKeys * kTopkThreads ? topk_reg_kernel<kShortKeys>
                                                              : topk_reg_kernel<kRegKeys>,
                         dim3(nq), dim3(kTopkThreads), 0, st, pdl, c, b ? *b : none, scores, ld,
                         n_override, idx_out, cnt_out, status, max_vis, (pdl && early) ? 1 : 0,
                         ready, epoch, (pdl && early && b) ? done : nullptr, qsplit, keys ? 1 : 0);
  if (keys) return launch_fail("Top-K: score keys need the register kernel", cudaSuccess);
  const int smem = (max_vis + max_vis / 16 + 1) * 4;
  if (smem > kTopkSmemMax)  // rows are bounded at create time
    return launch_fail("Top-K: rows longer than the kernel holds", cudaSuccess);
  // the opt-in for the longest rows a config may have, once per device
  static PerDeviceOnce attr;
  if (smem > 48 * 1024) {
    if (const cudaError_t e = attr.run([] {
          return allow_max_dynamic_smem(topk_kernel);
        }))
      return launch_fail("cudaFuncSetAttribute(topk_kernel)", e);
  }
  return launch_kernel(topk_kernel, dim3(nq), dim3(kTopkThreads), smem, st, pdl, c, b ? *b : none,
                       scores, ld, n_override, idx_out, cnt_out, status, max_vis, ready, epoch);
}

}  // namespace csa
