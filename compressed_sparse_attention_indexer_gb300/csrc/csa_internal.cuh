// Internal definitions shared by the kernels of libcsa (not part of the ABI).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

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

struct DevCfg {
  int H, D, V, R, Hi, Di, ratio, K, win, hca_ratio, dtype;
  float scale, rope_base;
  int max_context, max_vis;
};

struct DevBatch {
  int B, S;
  const int* ctx_len;
  const void* q;
  const void* q_idx;
  const float* w;
  const void* raw; const int64_t* raw_off; int64_t raw_stride, raw_rows;
  const void* cmp; const int64_t* cmp_off; int64_t cmp_stride, cmp_rows;
  const void* idx; const int64_t* idx_off; int64_t idx_stride, idx_rows;
  const void* hca; const int64_t* hca_off; int64_t hca_stride, hca_rows;
};

struct QueryPlan {
  int pos, vis, nwin, cnt, vis2, flags;
};

// Device workspace owned by a handle.
struct Workspace {
  int* status;        // [1]
  QueryPlan* plan;    // [max_T]
  int* item_prefix;   // [max_batch + 1] indexer work items (row chunks) per request, prefix
  int* req_rows;      // [max_batch] rows the indexer scores for request b
  float* scores;      // [max_T, max_vis]
  int* topk_idx;      // [max_T, K]
  int* topk_cnt;      // [max_T]
  int max_T, max_batch;
  int64_t scores_ld;
};

// Rows of one indexer work item (tensor-core and SIMT paths).
constexpr int kIdxChunk = 128;

__device__ __forceinline__ void set_status(int* status, int bit) {
  atomicOr(status, bit);
}

// ---- launch wrappers (defined in the kernel files) -------------------------
// Each returns the number of kernels launched (>= 0) or -1 on a launch error.
int launch_plan(const DevCfg& c, const DevBatch& b, const Workspace& ws, int score_all,
                const int* topk_cnt_in, cudaStream_t st);
int launch_indexer(const DevCfg& c, const DevBatch& b, const Workspace& ws, float* scores,
                   int64_t ld, int total_items_hint, int num_sms, cudaStream_t st);
int launch_topk(const DevCfg& c, int nq, const QueryPlan* plan, const float* scores, int64_t ld,
                const int* n_override, int* idx_out, int* cnt_out, int* status, int max_vis,
                cudaStream_t st);
int launch_attention(const DevCfg& c, const DevBatch& b, const Workspace& ws, const int* topk_idx,
                     const int* topk_cnt, void* out, float* lse_out, int num_sms,
                     cudaStream_t st);

bool tensor_core_shape(const DevCfg& c);

}  // namespace csa
