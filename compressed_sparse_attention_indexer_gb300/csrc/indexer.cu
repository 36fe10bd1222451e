// Step (a): the lightning-indexer score of every visible compressed row,
//   score_j = sum_h w_h * ReLU(q_idx[h] . k_idx[j]),
// written to an fp32 score buffer.  hw-native-sys/pypto-lib "Perf: skip
// redundant CSA scoring and fuse gather unpack" (the indexer and the query
// scoring it skips) and "Fix: port the DeepSeek-V4 MoE, hc_pre and prefill
// fixes to DSpark" (partials reduced in a fixed ascending order, no atomics).
//
// This file holds the launcher and two kernels:
//  - a warp-MMA (mma.sync) kernel for the tensor-core shape, kept as the
//    measured baseline of the tcgen05 kernel (indexer_tc5.cu), selected with
//    CSA_INDEXER=mma: a persistent grid walks the work list of 128-row
//    chunks; each chunk of k_idx rows is streamed once into shared memory
//    through a multi-stage cp.async ring and reused by every scored query of
//    its request; rows are the M side of the MMA, heads the N side; lanes of
//    a row sum w_h * ReLU(.) over h = 0..31 and 32..63 in order and the two
//    halves are added in that order;
//  - a SIMT kernel for any other shape / dtype: one warp per row, fp32 FMA.
#include <stdlib.h>
#include <string.h>

#include "csa_internal.cuh"
#include "ptx.cuh"

namespace csa {

namespace {

constexpr int kIdxThreads = 256;                    // 8 warps x 16 rows = kIdxChunk
constexpr int kQBytes = kTcHi * kTcDi * 2;          // one query's q_idx: 16 KB
constexpr int kKStageBytes = kIdxChunk * kTcDi * 2; // one chunk of keys: 32 KB
constexpr int kStashLd = 65;                        // 64 heads + 1 pad (bank spread)
constexpr int kStashBytes = (kIdxThreads / 32) * 16 * kStashLd * 4;

__device__ __forceinline__ void wait_stages(int nst) {
  // keep at most nst-2 groups pending
  if (nst >= 4) cp_async_wait<2>();
  else if (nst == 3) cp_async_wait<1>();
  else cp_async_wait<0>();
}

__device__ __forceinline__ int request_of(const int* prefix, int B, int item) {
  int l = 0, r = B - 1;
  while (l < r) {
    const int m = (l + r + 1) >> 1;
    if (prefix[m] <= item) l = m; else r = m - 1;
  }
  return l;
}

__global__ void __launch_bounds__(kIdxThreads, 1)
    indexer_mma_kernel(const __grid_constant__ ItemList items, DevCfg c, DevBatch b, Workspace ws,
                       int score_all, float* __restrict__ scores, int64_t ld, int SG, int NST,
                       int qsplit) {
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t* Qs = smem;
  uint8_t* Ks = Qs + SG * kQBytes;
  float* stash = reinterpret_cast<float*>(Ks + NST * kKStageBytes);
  float* w_s = stash + (kIdxThreads / 32) * 16 * kStashLd;

  pdl_wait();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int* __restrict__ prefix = items.host_B >= 0 ? items.prefix : ws.item_prefix;
  const int N = prefix[b.B];
  const int G = gridDim.x;
  const int lo = (int)((int64_t)blockIdx.x * N / G);
  const int hi = (int)((int64_t)(blockIdx.x + 1) * N / G);
  pdl_trigger();
  if (lo >= hi) return;

  const int b0 = request_of(prefix, b.B, lo);
  const __nv_bfloat16* __restrict__ kbase = static_cast<const __nv_bfloat16*>(b.idx);

  // issue cursor, with the request's values cached
  int ib = b0, ib_end = prefix[b0 + 1], ib_first = prefix[b0];
  int ib_rows = request_rows(c, b.S, b.ctx_len[b0], score_all);
  // with qsplit, a request's items are (query group, key chunk) pairs, group
  // major: item i of the request is chunk i % chunks of group i / chunks
  auto issue = [&](int item) {
    while (item >= ib_end) {
      ++ib;
      ib_first = ib_end;
      ib_end = prefix[ib + 1];
      ib_rows = request_rows(c, b.S, b.ctx_len[ib], score_all);
    }
    const int ib_chunks = (ib_rows + kIdxChunk - 1) / kIdxChunk;
    const int li = item - ib_first;
    const int c0 = (qsplit ? li % ib_chunks : li) * kIdxChunk;
    uint8_t* dst0 = Ks + (item % NST) * kKStageBytes;
#pragma unroll
    for (int i = 0; i < (kIdxChunk * 16) / kIdxThreads; ++i) {
      const int id = tid + i * kIdxThreads;
      const int row = id >> 4, ch = id & 15;
      const int r = c0 + row;
      const int64_t gr = r < ib_rows ? idx_row(b, ib, r) : -1;
      const bool inb = gr >= 0 && gr < b.idx_rows;
      const bool want = r < ib_rows;
      if (want && !inb && ch == 0) set_status(ws.status, kStatusBadIndex);
      const bool ok = want && inb;
      const void* src = ok ? (const void*)(kbase + gr * b.idx_stride + ch * 8) : (const void*)kbase;
      cp_async16(smem_u32(dst0 + row * 256 + ((ch ^ (row & 7)) << 4)), src, ok ? 16 : 0);
    }
  };

  for (int k = 0; k < NST - 1; ++k) {
    if (lo + k < hi) issue(lo + k);
    cp_async_commit();
  }

  int cb = b0, cb_end = prefix[b0 + 1], cb_first = prefix[b0], cb_L = b.ctx_len[b0];
  int q_b = -1, q_g = -1;
  for (int it = lo; it < hi; ++it) {
    wait_stages(NST);
    __syncthreads();
    {
      const int nxt = it + NST - 1;
      if (nxt < hi) issue(nxt);
      cp_async_commit();
    }
    while (it >= cb_end) {
      ++cb;
      cb_first = cb_end;
      cb_end = prefix[cb + 1];
      cb_L = b.ctx_len[cb];
    }
    const int cb_chunks = (request_rows(c, b.S, cb_L, score_all) + kIdxChunk - 1) / kIdxChunk;
    const int li = it - cb_first;
    const int c0 = (qsplit ? li % cb_chunks : li) * kIdxChunk;
    const int gfirst = qsplit ? (li / cb_chunks) * qsplit : 0;      // this item's query group
    const int gend = qsplit ? min(b.S, gfirst + qsplit) : b.S;
    const uint8_t* Kst = Ks + (it % NST) * kKStageBytes;

    // A fragments: this warp's 16 key rows x 128 dims, kept across queries
    uint32_t a[8][4];
    {
      const int row = warp * 16 + (lane & 15);
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        const int ch = 2 * kk + (lane >> 4);
        ldsm_x4(smem_u32(Kst + row * 256 + ((ch ^ (row & 7)) << 4)), a[kk][0], a[kk][1],
                a[kk][2], a[kk][3]);
      }
    }

    for (int g0 = gfirst; g0 < gend; g0 += SG) {
      const int ng = min(SG, gend - g0);
      if (cb != q_b || g0 != q_g) {
        __syncthreads();  // every warp is done with the previous q_idx group
        const uint4* src = reinterpret_cast<const uint4*>(
            static_cast<const __nv_bfloat16*>(b.q_idx) + ((int64_t)cb * b.S + g0) * kTcHi * kTcDi);
        for (int v = tid; v < ng * kTcHi * 16; v += kIdxThreads) {
          const int row = v >> 4, ch = v & 15;  // row = s_local*64 + h
          const uint4 x = __ldg(src + v);
          *reinterpret_cast<uint4*>(Qs + row * 256 + ((ch ^ (row & 7)) << 4)) = x;
        }
        for (int v = tid; v < ng * kTcHi; v += kIdxThreads)
          w_s[v] = __ldg(b.w + ((int64_t)cb * b.S + g0) * kTcHi + v);
        __syncthreads();
        q_b = cb;
        q_g = g0;
      }
      for (int sl = 0; sl < ng; ++sl) {
        const int qid = cb * b.S + g0 + sl;
        const QueryPlan p = query_plan(c, b.S, cb_L, g0 + sl, score_all);
        if (!(p.flags & kPlanScore) || p.vis <= c0) continue;  // warp-uniform
        float acc[8][4];
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.f;
        const uint8_t* Qq = Qs + sl * kQBytes;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
#pragma unroll
          for (int pp = 0; pp < 4; ++pp) {
            const int head = 16 * pp + ((lane >> 4) << 3) + (lane & 7);
            const int ch = 2 * kk + ((lane >> 3) & 1);
            uint32_t r0, r1, r2, r3;
            ldsm_x4(smem_u32(Qq + head * 256 + ((ch ^ (head & 7)) << 4)), r0, r1, r2, r3);
            mma_bf16_16816(acc[2 * pp], a[kk], r0, r1);
            mma_bf16_16816(acc[2 * pp + 1], a[kk], r2, r3);
          }
        }
        // epilogue: ReLU, then w-weighted sum over heads in ascending order
        float* st = stash + warp * 16 * kStashLd;
        const int g = lane >> 2, t = lane & 3;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          st[g * kStashLd + 8 * j + 2 * t] = fmaxf(acc[j][0], 0.f);
          st[g * kStashLd + 8 * j + 2 * t + 1] = fmaxf(acc[j][1], 0.f);
          st[(g + 8) * kStashLd + 8 * j + 2 * t] = fmaxf(acc[j][2], 0.f);
          st[(g + 8) * kStashLd + 8 * j + 2 * t + 1] = fmaxf(acc[j][3], 0.f);
        }
        __syncwarp();
        const int row = lane & 15, half = lane >> 4;
        const float* wq = w_s + sl * kTcHi + half * 32;
        const float* sr = st + row * kStashLd + half * 32;
        float sum = 0.f;
#pragma unroll 8
        for (int h = 0; h < 32; ++h) sum = fmaf(wq[h], sr[h], sum);
        const float upper = __shfl_down_sync(0xffffffffu, sum, 16);
        const int j = c0 + warp * 16 + row;
        if (half == 0 && j < p.vis) scores[(int64_t)qid * ld + j] = sum + upper;
        __syncwarp();
      }
    }
  }
  cp_async_wait<0>();
}

// ---------------------------------------------------------------------------
template <typename T>
__device__ __forceinline__ float ldf(const T* p, int64_t i);
template <>
__device__ __forceinline__ float ldf<float>(const float* p, int64_t i) { return p[i]; }
template <>
__device__ __forceinline__ float ldf<__nv_bfloat16>(const __nv_bfloat16* p, int64_t i) {
  return __bfloat162float(p[i]);
}

template <typename T>
__global__ void __launch_bounds__(256) indexer_simt_kernel(DevCfg c, DevBatch b, Workspace ws,
                                                           int score_all,
                                                           float* __restrict__ scores,
                                                           int64_t ld) {
  pdl_wait();
  pdl_trigger();
  const int q = blockIdx.x;
  const int bi = q / b.S;
  const QueryPlan p = query_plan(c, b.S, b.ctx_len[bi], q - bi * b.S, score_all);
  if (!(p.flags & kPlanScore)) return;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const T* qi = static_cast<const T*>(b.q_idx) + (int64_t)q * c.Hi * c.Di;
  const float* wq = b.w + (int64_t)q * c.Hi;
  const T* kp = static_cast<const T*>(b.idx);
  for (int j = blockIdx.y * 8 + warp; j < p.vis; j += gridDim.y * 8) {
    const int64_t gr = idx_row(b, bi, j);
    float acc;
    if (gr < 0 || gr >= b.idx_rows) {
      if (lane == 0) set_status(ws.status, kStatusBadIndex);
      acc = -INFINITY;
    } else {
      acc = 0.f;
      const T* kr = kp + gr * b.idx_stride;
      for (int h = 0; h < c.Hi; ++h) {
        float dot = 0.f;
        for (int d = lane; d < c.Di; d += 32) dot = fmaf(ldf(qi, (int64_t)h * c.Di + d), ldf(kr, d), dot);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, o);
        acc = fmaf(wq[h], fmaxf(dot, 0.f), acc);
      }
    }
    if (lane == 0) scores[(int64_t)q * ld + j] = acc;
  }
}

}  // namespace

// Indexer kernel for the tensor-core shape: the tcgen05 kernel by default;
// CSA_INDEXER=mma in the environment selects the warp-MMA kernel (kept as the
// measured baseline of the tcgen05 one).
int indexer_impl() {
  static const int impl = [] {
    const char* e = getenv("CSA_INDEXER");
    return (e && strcmp(e, "mma") == 0) ? kIndexerMma : kIndexerTc5;
  }();
  return impl;
}

bool tensor_core_shape(const DevCfg& c) {
  return c.dtype == CSA_DTYPE_BF16 && c.H == kTcH && c.D == kTcD && c.V == kTcV &&
         c.Hi == kTcHi && c.Di == kTcDi;
}

// Queries per work item: 0 keeps one item per key chunk with all of the
// request's queries.  A request whose queries do not fit the kernel at once (a
// prefill chunk) has its work split by query group, items being (group, key
// chunk) pairs that spread over the SMs: groups of kT5Group queries for the
// tcgen05 kernel (the FP8 keys' only kernel), of kMmaGroup for the warp-MMA
// one.  The work list and the kernel take the same value.
int indexer_qsplit(const DevCfg& c, int S) {
  if (c.dtype != CSA_DTYPE_BF16 || c.Hi != kTcHi || c.Di != kTcDi) return 0;
  if (c.idx_fp8 || (tensor_core_shape(c) && indexer_impl() == kIndexerTc5)) {
    if (indexer_tc5_fits(c, S)) return 0;
    if (S > kT5Group && indexer_tc5_fits(c, kT5Group)) return kT5Group;
    if (c.idx_fp8) return 0;  // unreachable: kT5Group queries always fit
  }
  return S > kMmaGroup ? kMmaGroup : 0;
}

int launch_indexer(const DevCfg& c, const DevBatch& b, const Workspace& ws, const ItemList& items,
                   int score_all, float* scores, int64_t ld, int num_sms, cudaStream_t st,
                   bool pdl, int* done, int* done_clear, bool* published, bool keys, bool* keyed) {
  if (published) *published = false;
  if (keyed) *keyed = false;
  const int known = items.host_B >= 0 ? items.prefix[items.host_B] : -1;  // items, if known
  if (known == 0) return 0;
  const int qsplit = indexer_qsplit(c, b.S);
  if (c.idx_fp8) {  // FP8 keys: the tcgen05 kernel only (its shape is checked at create)
    const int r = launch_indexer_tc5(c, b, ws, items, score_all, scores, ld, num_sms, qsplit, st,
                                     pdl, done, done_clear, keys);
    if (r > 0 && published) *published = done != nullptr;
    if (r > 0 && keyed) *keyed = keys;
    return r == -2 ? -1 : r;
  }
  if (tensor_core_shape(c) && indexer_impl() == kIndexerTc5) {
    const int r = launch_indexer_tc5(c, b, ws, items, score_all, scores, ld, num_sms, qsplit, st,
                                     pdl, done, done_clear, keys);
    if (r > 0 && published) *published = done != nullptr;
    if (r > 0 && keyed) *keyed = keys;
    if (r != -2) return r;  // -2: shape outside the tcgen05 kernel, use warp MMA
  }
  if (tensor_core_shape(c)) {
    const int SG = b.S < kMmaGroup ? b.S : kMmaGroup;
    const int fixed = SG * kQBytes + kStashBytes + SG * kTcHi * 4;
    int NST = (227 * 1024 - fixed) / kKStageBytes;
    NST = NST > 4 ? 4 : NST;
    if (NST < 2) return launch_fail("warp-MMA indexer: no room for two key stages", cudaSuccess);
    const int smem = fixed + NST * kKStageBytes;
    static PerDeviceOnce attr;
    if (const cudaError_t e = attr.run([] {
          return allow_max_dynamic_smem(indexer_mma_kernel);
        }))
      return launch_fail("cudaFuncSetAttribute(indexer_mma_kernel)", e);
    int grid = num_sms;
    if (known > 0 && known < grid) grid = known;
    return launch_kernel(indexer_mma_kernel, dim3(grid), dim3(kIdxThreads), smem, st, pdl, items,
                         c, b, ws, score_all, scores, ld, SG, NST, qsplit);
  }
  int y = (c.max_vis + 7) / 8;
  if (y > 64) y = 64;
  if (y < 1) y = 1;
  const dim3 grid(b.B * b.S, y);
  if (c.dtype == CSA_DTYPE_BF16)
    return launch_kernel(indexer_simt_kernel<__nv_bfloat16>, grid, dim3(256), 0, st, pdl, c, b, ws,
                         score_all, scores, ld);
  return launch_kernel(indexer_simt_kernel<float>, grid, dim3(256), 0, st, pdl, c, b, ws,
                       score_all, scores, ld);
}

}  // namespace csa
