// Step (b): exact Top-K of each query's indexer scores, ties to the lower
// index, output in ascending index order and -1 padded; the bypass takes
// every visible row when vis <= K.  hw-native-sys/pypto-lib "Perf: skip
// redundant CSA scoring and fuse gather unpack" (bounded Top-K indices,
// bypass) and "Fix: port the DeepSeek-V4 MoE, hc_pre and prefill fixes to
// DSpark" (a staged sort that stops at 256 picks wrong keys past 256: the
// selection here is exact at any width).
//
// One 1024-thread block per query.  Scores become order-preserving 32-bit
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

__device__ __forceinline__ uint32_t score_key(float f) {
  uint32_t u = __float_as_uint(f);
  if ((u & 0x7fffffffu) > 0x7f800000u) return 0u;  // NaN: lowest
  if (u == 0x80000000u) u = 0u;                   // -0.0 == +0.0
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Key i lives at keys[kpad(i)]: one pad word per 16 keys, so the final pass
// (thread t reads keys 16t .. 16t+15) hits 32 different banks.
__device__ __forceinline__ int kpad(int i) { return i + (i >> 4); }

__global__ void __launch_bounds__(kTopkThreads, 1)
    topk_kernel(DevCfg c, DevBatch b, const float* __restrict__ scores, int64_t ld,
                const int* __restrict__ n_override, int* __restrict__ idx_out,
                int* __restrict__ cnt_out, int* __restrict__ status, int max_vis) {
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
}

}  // namespace

int launch_topk(const DevCfg& c, const DevBatch* b, int nq, const float* scores, int64_t ld,
                const int* n_override, int* idx_out, int* cnt_out, int* status, int max_vis,
                cudaStream_t st, bool pdl) {
  if (nq == 0) return 0;
  const int smem = (max_vis + max_vis / 16 + 1) * 4;
  static int attr_smem = 0;
  if (smem > 48 * 1024 && smem > attr_smem) {
    cudaFuncSetAttribute(topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    attr_smem = smem;
  }
  DevBatch none = {};
  none.S = 1;
  return launch_kernel(topk_kernel, dim3(nq), dim3(kTopkThreads), smem, st, pdl, c, b ? *b : none,
                       scores, ld, n_override, idx_out, cnt_out, status, max_vis);
}

}  // namespace csa
