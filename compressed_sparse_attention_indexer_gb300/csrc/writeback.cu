// The cache update that precedes a decode step: every new token's row is
// written into a cache pool at the row its slot mapping names.
// hw-native-sys/pypto-lib "Perf: parallelize the DSpark TP-4 SWA decode hot
// tasks", PR description: the SWA KV scatter runs by slot mapping over token
// tiles whose count is a ceiling division with the last tile clamped to the
// remaining rows, so every slot-mapping entry is committed.
//
// Here one grid-stride loop covers every (row, copy unit) pair of the n rows,
// so there is no tile count to round and no entry can be left out.  A row is
// row_bytes bytes; the copy unit is 16, 4 or 1 bytes, the largest that
// divides the row size, both strides and both base addresses.  A negative
// slot is a padding token (skipped); a slot at or past pool_rows is skipped
// and recorded in the status word.  Slots are expected to be collision-free
// (each pool row written by at most one token), as an allocator hands them
// out; with a repeated slot the row holds one of the rows written to it.
#include "csa_internal.cuh"

namespace csa {

namespace {

template <typename U>
__global__ void __launch_bounds__(256)
    writeback_kernel(const uint8_t* __restrict__ src, int64_t src_stride,
                     const int64_t* __restrict__ slot, int n, uint8_t* __restrict__ pool,
                     int64_t pool_stride, int64_t pool_rows, int64_t units, int* __restrict__ status) {
  pdl_wait();
  pdl_trigger();
  const int64_t total = (int64_t)n * units;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t t = i / units, u = i - t * units;
    const int64_t s = slot[t];
    if (s < 0) continue;  // a padding token
    if (s >= pool_rows) {
      if (u == 0 && status) set_status(status, kStatusBadIndex);
      continue;
    }
    const U v = *reinterpret_cast<const U*>(src + t * src_stride + u * (int64_t)sizeof(U));
    *reinterpret_cast<U*>(pool + s * pool_stride + u * (int64_t)sizeof(U)) = v;
  }
}

template <typename U>
int launch_unit(const void* src, int64_t src_stride, const int64_t* slot, int n, void* pool,
                int64_t pool_stride, int64_t pool_rows, int64_t row_bytes, int* status,
                cudaStream_t st, bool pdl) {
  const int64_t units = row_bytes / (int64_t)sizeof(U);
  const int64_t total = (int64_t)n * units;
  int64_t blocks = (total + 255) / 256;
  if (blocks > 4096) blocks = 4096;  // grid-stride beyond
  return launch_kernel(writeback_kernel<U>, dim3((unsigned)blocks), dim3(256), 0, st, pdl,
                       static_cast<const uint8_t*>(src), src_stride, slot, n,
                       static_cast<uint8_t*>(pool), pool_stride, pool_rows, units, status);
}

}  // namespace

int launch_writeback(const void* src, int64_t src_stride, const int64_t* slot, int n, void* pool,
                     int64_t pool_stride, int64_t pool_rows, int64_t row_bytes, int* status,
                     cudaStream_t st, bool pdl) {
  if (n == 0 || row_bytes == 0) return 0;
  const uint64_t all = (uint64_t)row_bytes | (uint64_t)src_stride | (uint64_t)pool_stride |
                       reinterpret_cast<uintptr_t>(src) | reinterpret_cast<uintptr_t>(pool);
  if ((all & 15u) == 0)
    return launch_unit<uint4>(src, src_stride, slot, n, pool, pool_stride, pool_rows, row_bytes,
                              status, st, pdl);
  if ((all & 3u) == 0)
    return launch_unit<uint32_t>(src, src_stride, slot, n, pool, pool_stride, pool_rows,
                                 row_bytes, status, st, pdl);
  return launch_unit<uint8_t>(src, src_stride, slot, n, pool, pool_stride, pool_rows, row_bytes,
                              status, st, pdl);
}

}  // namespace csa
