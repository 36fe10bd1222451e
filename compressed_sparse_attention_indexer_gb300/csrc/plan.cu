// The indexer's work list when the host does not pass the lengths: one
// block turns ctx_len into prefix[b] = first 128-row chunk of request b
// (prefix[B] = number of chunks).  Integer work only.
//
// hw-native-sys/pypto-lib "Perf: skip redundant CSA scoring and fuse gather
// unpack", PR description: a query whose visible ratio-4 rows fit Top-K
// (vis <= K) skips scoring, so its rows are not in the list.
#include "csa_internal.cuh"
#include "ptx.cuh"

namespace csa {

__global__ void __launch_bounds__(1024) prep_kernel(DevCfg c, DevBatch b, Workspace ws,
                                                    int score_all, int qsplit) {
  __shared__ int scan_tmp[33];
  __shared__ int carry;
  pdl_wait();
  if (threadIdx.x == 0) carry = 0;
  __syncthreads();
  for (int base = 0; base < b.B; base += blockDim.x) {
    const int bi = base + threadIdx.x;
    int items = 0;
    if (bi < b.B) {
      const int L = b.ctx_len[bi];
      items = request_items(c, b.S, L, score_all, qsplit);  // (query group, key chunk) items
    }
    int total;
    const int ex = block_exclusive_scan(items, scan_tmp, &total);
    if (bi < b.B) ws.item_prefix[bi] = carry + ex;
    __syncthreads();
    if (threadIdx.x == 0) carry += total;
    __syncthreads();
  }
  if (threadIdx.x == 0) ws.item_prefix[b.B] = carry;
  pdl_trigger();
}

void* tensor_map_encoder() {
  static void* const fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult r;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &r) !=
            cudaSuccess ||
        r != cudaDriverEntryPointSuccess)
      p = nullptr;
    return p;
  }();
  return fn;
}

int launch_prep(const DevCfg& c, const DevBatch& b, const Workspace& ws, int score_all, int qsplit,
                cudaStream_t st, bool pdl) {
  return launch_kernel(prep_kernel, dim3(1), dim3(1024), 0, st, pdl, c, b, ws, score_all, qsplit);
}

}  // namespace csa
