// Step (a0): per-query visibility, window, bypass decision and the indexer's
// work list.  One block; integer work only.
//
// hw-native-sys/pypto-lib "Perf: skip redundant CSA scoring and fuse gather
// unpack", PR description: a query whose visible ratio-4 rows fit Top-K
// (vis <= K) skips scoring and sorting and takes every visible row, with
// causal visibility retained.  "Fix: port the DeepSeek-V4 MoE, hc_pre and
// prefill fixes to DSpark", PR description: the rows a query reads are
// bounded by WIN + min(max_visible_cmp, IDX_TOPK).
#include "csa_internal.cuh"
#include "ptx.cuh"

namespace csa {

__global__ void __launch_bounds__(1024) plan_kernel(DevCfg c, DevBatch b, Workspace ws,
                                                    int score_all, const int* cnt_in) {
  __shared__ int scan_tmp[33];
  __shared__ int carry;
  const int T = b.B * b.S;
  for (int q = threadIdx.x; q < T; q += blockDim.x) {
    const int bi = q / b.S, s = q - bi * b.S;
    const int L = b.ctx_len[bi];
    QueryPlan p;
    p.pos = p.vis = p.nwin = p.cnt = p.vis2 = 0;
    p.flags = 0;
    if (L < b.S || L > c.max_context) {
      p.flags = kPlanBad;
      set_status(ws.status, kStatusBadIndex);
    } else {
      p.pos = L - b.S + s;
      p.vis = (p.pos + 1) / c.ratio;
      p.nwin = min(c.win, p.pos + 1);
      p.vis2 = c.hca_ratio > 0 ? (p.pos + 1) / c.hca_ratio : 0;
      p.cnt = min(p.vis, c.K);
      const bool score = p.vis > c.K || (score_all && p.vis > 0);
      p.flags = score ? kPlanScore : 0;
      if (cnt_in) {  // caller-supplied Top-K counts
        int ci = cnt_in[q];
        if (ci < 0 || ci > p.cnt) {
          set_status(ws.status, kStatusBadIndex);
          ci = ci < 0 ? 0 : p.cnt;
        }
        p.cnt = ci;
      }
    }
    ws.plan[q] = p;
  }
  // rows to score per request = the largest vis among its scored queries;
  // work items are chunks of kIdxChunk rows
  if (threadIdx.x == 0) carry = 0;
  __syncthreads();
  for (int base = 0; base < b.B; base += blockDim.x) {
    const int bi = base + threadIdx.x;
    int items = 0;
    if (bi < b.B) {
      const int L = b.ctx_len[bi];
      int rows = 0;
      if (L >= b.S && L <= c.max_context) {
        for (int s = 0; s < b.S; ++s) {
          const int pos = L - b.S + s;
          const int vis = (pos + 1) / c.ratio;
          if (vis > c.K || (score_all && vis > 0)) rows = max(rows, vis);
        }
      }
      ws.req_rows[bi] = rows;
      items = (rows + kIdxChunk - 1) / kIdxChunk;
    }
    int total;
    const int ex = block_exclusive_scan(items, scan_tmp, &total);
    if (bi < b.B) ws.item_prefix[bi] = carry + ex;
    __syncthreads();
    if (threadIdx.x == 0) carry += total;
    __syncthreads();
  }
  if (threadIdx.x == 0) ws.item_prefix[b.B] = carry;
}

int launch_plan(const DevCfg& c, const DevBatch& b, const Workspace& ws, int score_all,
                const int* topk_cnt_in, cudaStream_t st) {
  plan_kernel<<<1, 1024, 0, st>>>(c, b, ws, score_all, topk_cnt_in);
  return cudaGetLastError() == cudaSuccess ? 1 : -1;
}

}  // namespace csa
