// Step (a) on the fifth-generation tensor cores: the lightning-indexer score
//   score_j = sum_h w_h * ReLU(q_idx[h] . k_idx[j])
// with TMA-fed shared memory, tcgen05 MMA and TMEM accumulators.
// hw-native-sys/pypto-lib "Perf: skip redundant CSA scoring and fuse gather
// unpack" (the indexer) and "Fix: port the DeepSeek-V4 MoE, hc_pre and
// prefill fixes to DSpark" (fixed, ascending reduction order; no atomics).
//
// Persistent kernel, two CTAs per SM (one when a work unit's q_idx leaves no
// room), warp-specialised:
//   warp 4  TMA producer: per work item (128 key rows of one request) two
//           128x64 bf16 boxes, 128-byte swizzled, into a ring of stages;
//           the work unit's q_idx (its queries x 64 heads x 128) when the
//           unit changes.  A unit is a request's S queries, or, for a
//           request whose queries do not fit (a prefill chunk), a group of
//           four of them: the request's items are then (group, key chunk)
//           pairs, group major;
//   warp 5  allocates TMEM; one thread issues the MMAs:
//           D[128 rows x 64*G heads] = K_tile[128 x 128] . Q^T, M = 128,
//           N = 64*G (G <= 4 queries per MMA), eight K = 16 steps, into one
//           of NB TMEM accumulators (8 of 64 columns when S = 1, so the MMAs
//           run up to 8 items ahead of the epilogue), then commits to
//           mbarriers;
//   warps 6-9 (FP8 keys) converters: one thread per key row turns the
//           item's E4M3 codes into the bf16 tile the MMA reads;
//   warps 0-3 epilogue: thread t owns TMEM lane t = key row t of the item;
//           it reads that row's 64 head dot products of a query and sums
//           w_h * ReLU(.) as four 16-head partials (h ascending within each),
//           added in ascending order, then writes the score.  w of the
//           unit is cached in shared memory.
// HBM reads per item are the 32 KB of keys (q_idx comes from L2), so the
// kernel runs at the HBM roofline when enough stages are in flight.
// Every mbarrier wait is bounded; a wait that gives up records
// CSA_ERR_TIMEOUT in the status word and the whole block winds down.
#include <cudaTypedefs.h>
#include <stdlib.h>

#include "csa_internal.cuh"
#include "tc5.cuh"

namespace csa {

namespace {

constexpr int kT5Threads = 192;
constexpr int kConvWarps = 4;                   // FP8: converter warps, one thread per key row
constexpr int kConvThreads = 32 * kConvWarps;
constexpr int kFp8CtasPerSm = 2;                // FP8: CTAs per SM (register budget of the launch)
constexpr int kT5ThreadsFp8 = kT5Threads + kConvThreads;
constexpr int kSubBytes = kIdxChunk * 64 * 2;   // 128 rows x 64 dims bf16 = 16 KB
constexpr int kStageBytes = 2 * kSubBytes;      // 32 KB: one item of keys
constexpr int kStage8Bytes = kIdxChunk * kTcDi; // 16 KB: one item of FP8 keys
constexpr int kConvBufs = 2;                    // FP8: converted (bf16) items in flight
constexpr int kQSubBytes = kTcHi * 64 * 2;      // 64 heads x 64 dims = 8 KB
constexpr int kMaxG = 4;                        // queries per MMA group

struct T5Smem {
  uint64_t full[8], empty[8], qfull[2], qempty[2], tfull[8], tempty[8], done;
  uint64_t cfull[kConvBufs], cempty[kConvBufs];  // FP8 keys: converted items
  uint64_t ebar;                                 // the epilogue warps' bounded barrier
  uint32_t tmem_base;
  int abort;
};

// Sixteen FP8 E4M3 keys (one 16-byte chunk) to sixteen bf16, exactly: every
// E4M3 value (subnormals included, NaN stays NaN) is an f16 value, every f16
// value an f32 value, and every such value a bf16 value.  Byte 2i of the
// chunk is dim 2i; each pair is E4M3x2 -> f16x2 -> two f32 -> one bf16x2.
__device__ __forceinline__ void e4m3x16_to_bf16(const uint4 in, uint32_t out[8]) {
  const uint32_t w[4] = {in.x, in.y, in.z, in.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      const uint16_t pair = (uint16_t)(w[i] >> (16 * half));
      uint32_t o;
      asm("{\n .reg .b32 h2;\n .reg .b16 a, b;\n .reg .f32 fa, fb;\n"
          " cvt.rn.f16x2.e4m3x2 h2, %1;\n mov.b32 {a, b}, h2;\n"
          " cvt.f32.f16 fa, a;\n cvt.f32.f16 fb, b;\n cvt.rn.bf16x2.f32 %0, fb, fa;\n}\n"
          : "=r"(o) : "h"(pair));
      out[2 * i + half] = o;
    }
  }
}

// Adds v to *p with release semantics at GPU scope (a reader that acquires
// the sum sees every store that happened before the add).
__device__ __forceinline__ void red_release_add(int* p, int v) {
  asm volatile("red.release.gpu.global.add.s32 [%0], %1;\n" ::"l"(p), "r"(v) : "memory");
}

// Walks the work list in item order: the request owning the current item and
// its item range, re-read only when the request changes (the single-thread
// roles would otherwise pay a dependent global load per item).
struct ReqCursor {
  const int* prefix;
  int bi, first, end;
  __device__ __forceinline__ void init(const int* p, int B, int item) {
    prefix = p;
    int l = 0, r = B - 1;
    while (l < r) {
      const int m = (l + r + 1) >> 1;
      if (p[m] <= item) l = m; else r = m - 1;
    }
    bi = l;
    first = p[l];
    end = p[l + 1];
  }
  // advances to the request owning `item`; true if it changed
  __device__ __forceinline__ bool advance(int item) {
    bool moved = false;
    while (item >= end) {
      ++bi;
      first = end;
      end = prefix[bi + 1];
      moved = true;
    }
    return moved;
  }
};

// The work unit of the current item within its request: the unit's first
// query g0, its su queries (all S, or a group of qsplit of them) in ngroups
// MMA groups of G, and the item's key chunk.  Placed with one division when a
// request starts, then advanced item by item.
struct UnitCursor {
  int S, SU, G, qsplit;
  int chunk, chunks, g0, su, ngroups;
  __device__ __forceinline__ void set_unit() {
    su = min(SU, S - g0);
    ngroups = (su + G - 1) / G;
  }
  // item li of a request of `nchunks` key chunks (1 without qsplit)
  __device__ __forceinline__ void start(int li, int nchunks) {
    chunks = nchunks;
    const int gq = qsplit ? li / chunks : 0;
    chunk = li - gq * chunks;
    g0 = gq * SU;
    set_unit();
  }
  // to the request's next item; true if that item starts a new unit
  __device__ __forceinline__ bool step() {
    if (++chunk < chunks || !qsplit) return false;
    chunk = 0;
    g0 += SU;
    set_unit();
    return true;
  }
};

// kFp8: the key pool holds FP8 E4M3 rows with a per-row fp32 scale
// (b.idx_scale).  Warps 6-13 then convert each item's FP8 tile (one TMA box)
// into the bf16 tile layout the MMA reads, and the epilogue multiplies each
// row's dot products by its scale before the ReLU.
// kSplit: the work list splits requests by query group (qsplit queries per
// unit); without it the unit bookkeeping folds away.
template <bool kFp8, bool kSplit>
__global__ void __launch_bounds__(kFp8 ? kT5ThreadsFp8 : kT5Threads, kFp8 ? kFp8CtasPerSm : 1)
    indexer_tc5_kernel(const __grid_constant__ CUtensorMap kmap,
                       const __grid_constant__ CUtensorMap qmap,
                       const __grid_constant__ ItemList items, DevCfg c, DevBatch b, Workspace ws,
                       int score_all, float* __restrict__ scores, int64_t ld, int NST, int NQB,
                       int acc_cols, int NB, int NCB, int qsplit_arg, int* __restrict__ done,
                       int* __restrict__ done_clear, int a_tmem, int keys) {
  const int qsplit = kSplit ? qsplit_arg : 0;
  // NB TMEM accumulators of acc_cols columns (>= 64 * queries per group): the
  // MMAs run up to NB jobs ahead of the epilogue
  // FP8 keys with a_tmem: the NCB converted items (128 rows x 64 columns of
  // bf16 pairs each) sit in TMEM after the accumulators, as the MMAs' A
  // operand, instead of in shared memory
  const bool a_in_tmem = kFp8 && a_tmem;
  const uint32_t tmem_cols = (uint32_t)(NB * acc_cols + (a_in_tmem ? NCB * 64 : 0));
  const uint32_t acol = (uint32_t)(NB * acc_cols);  // the first converted item's column
  extern __shared__ __align__(16) uint8_t smem_raw[];  // aligned to 1024 below
  __shared__ T5Smem sm;
  const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
  const uint32_t kbuf = base;                                  // NST x 32 KB (FP8: 16 KB)
  const uint32_t stage_bytes = kFp8 ? kStage8Bytes : kStageBytes;
  const uint32_t cbuf = kbuf + (uint32_t)NST * stage_bytes;    // FP8: converted items
  // Work unit: a request's queries, or with qsplit a group of qsplit of them
  // (a prefill chunk); a request's items are then (group, key chunk) pairs,
  // group major, and a unit's q_idx / w are loaded when the unit changes.
  const int S = b.S;
  const int SU = qsplit ? qsplit : S;                          // queries per unit
  const uint32_t qbytes = (uint32_t)SU * 2u * kQSubBytes;      // one unit's q_idx
  const uint32_t qbuf = cbuf + ((kFp8 && !a_tmem) ? (uint32_t)NCB * kStageBytes : 0u);  // NQB x qbytes
  float* w_sm = reinterpret_cast<float*>(smem_raw + (qbuf + (uint32_t)NQB * qbytes - smem_u32(smem_raw)));

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // barrier setup and the tensor-map prefetch need nothing from the previous
  // grid, so they overlap its tail
  if (tid == 0) {
    for (int i = 0; i < NST; ++i) {
      tc5::mbar_init(smem_u32(&sm.full[i]), 1);
      tc5::mbar_init(smem_u32(&sm.empty[i]), kFp8 ? kConvThreads : 1);  // FP8: the converters free a stage
    }
    for (int i = 0; i < NCB; ++i) {
      tc5::mbar_init(smem_u32(&sm.cfull[i]), kConvThreads);
      tc5::mbar_init(smem_u32(&sm.cempty[i]), 1);
    }
    for (int i = 0; i < 2; ++i) {
      tc5::mbar_init(smem_u32(&sm.qfull[i]), 1);
      tc5::mbar_init(smem_u32(&sm.qempty[i]), 1);
    }
    for (int i = 0; i < NB; ++i) {
      tc5::mbar_init(smem_u32(&sm.tfull[i]), 1);
      tc5::mbar_init(smem_u32(&sm.tempty[i]), 128);
    }
    tc5::mbar_init(smem_u32(&sm.done), 1);
    tc5::mbar_init(smem_u32(&sm.ebar), 128);
    sm.abort = 0;
    tc5::fence_mbar_init();
  }
  if (warp == 4 && lane == 0) {
    tc5::prefetch_tmap(&kmap);
    tc5::prefetch_tmap(&qmap);
  }
  pdl_wait();
  // the set of completion counters the next publishing launch uses starts at
  // zero: all of it (the next batch may be larger than this one, and an entry
  // past this batch may hold an earlier launch's count), cleared by CTA 0
  // whether or not it has items (a small batch leaves it none)
  if (done_clear && blockIdx.x == 0)
    for (int i = threadIdx.x; i < ws.max_batch; i += blockDim.x) done_clear[i] = 0;
  const int* __restrict__ prefix = items.host_B >= 0 ? items.prefix : ws.item_prefix;
  const int N = prefix[b.B];
  const int lo = (int)((int64_t)blockIdx.x * N / gridDim.x);
  const int hi = (int)((int64_t)(blockIdx.x + 1) * N / gridDim.x);
  pdl_trigger();
  if (lo >= hi) return;

  const int G = SU < kMaxG ? SU : kMaxG;
  // the request's key chunks, needed only to walk (group, key chunk) items
  auto chunks_of = [&](int bi) {
    return qsplit ? (request_rows(c, S, b.ctx_len[bi], score_all) + kIdxChunk - 1) / kIdxChunk : 1;
  };
  UnitCursor u;
  u.S = S;
  u.SU = SU;
  u.G = G;
  u.qsplit = qsplit;
  volatile int* abort = &sm.abort;

  if (warp == 5) {
    tc5::tmem_alloc(smem_u32(&sm.tmem_base), tmem_cols);
    tc5::tmem_relinquish();
  }
  tc5::fence_before_sync();
  __syncthreads();
  tc5::fence_after_sync();
  const uint32_t tmem = sm.tmem_base;

  if (warp == 4) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const uint64_t kpol = tc5::policy_evict_first();
      int kc = 0, qc = 0;
      ReqCursor cur;
      cur.init(prefix, b.B, lo);
      int64_t off = 0;
      for (int it = lo; it < hi && !*abort; ++it) {
        bool new_unit = cur.advance(it) || it == lo;
        if (new_unit) {
          off = b.idx_table ? 0 : b.idx_off[cur.bi];
          u.start(it - cur.first, chunks_of(cur.bi));
        } else {
          new_unit = u.step();
        }
        if (new_unit) {
          const int qb = qc % NQB;
          if (qc >= NQB && !tc5::mbar_wait(smem_u32(&sm.qempty[qb]), ((qc / NQB) - 1) & 1, abort))
            break;
          tc5::mbar_expect_tx(smem_u32(&sm.qfull[qb]), (uint32_t)u.su * 2u * kQSubBytes);
          for (int s = 0; s < u.su; ++s)
            for (int kt = 0; kt < 2; ++kt)
              tc5::tma_load_2d(qbuf + qb * qbytes + kt * (SU * kQSubBytes) + s * kQSubBytes, &qmap,
                               kt * 64, (cur.bi * S + u.g0 + s) * kTcHi, smem_u32(&sm.qfull[qb]));
          ++qc;
        }
        const int st = kc % NST;
        if (kc >= NST && !tc5::mbar_wait(smem_u32(&sm.empty[st]), ((kc / NST) - 1) & 1, abort))
          break;
        // the item's first pool row; a paged pool's blocks hold whole items
        // (block a multiple of 128 rows), an unmapped block reads as zeros
        // past the pool (its rows are reported by the epilogue)
        const int64_t c0 = (int64_t)u.chunk * kIdxChunk;
        int64_t y0 = b.idx_table ? idx_row(b, cur.bi, c0) : off + c0;
        if (y0 < 0) y0 = b.idx_rows;
        const int y = (int)y0;
        tc5::mbar_expect_tx(smem_u32(&sm.full[st]), stage_bytes);
        // keys are read once per step: evict them first from L2
        if (kFp8) {  // one box: 128 rows x 128 FP8 keys
          tc5::tma_load_2d_hint(kbuf + st * stage_bytes, &kmap, 0, y, smem_u32(&sm.full[st]), kpol);
        } else {
          tc5::tma_load_2d_hint(kbuf + st * kStageBytes, &kmap, 0, y, smem_u32(&sm.full[st]), kpol);
          tc5::tma_load_2d_hint(kbuf + st * kStageBytes + kSubBytes, &kmap, 64, y, smem_u32(&sm.full[st]),
                                kpol);
        }
        ++kc;
      }
      // let every copy this thread started land before the block exits
      for (int k = (kc > NST ? kc - NST : 0); k < kc; ++k)
        tc5::mbar_wait_drain(smem_u32(&sm.full[k % NST]), (k / NST) & 1);
      if (qc > 0) tc5::mbar_wait_drain(smem_u32(&sm.qfull[(qc - 1) % NQB]), ((qc - 1) / NQB) & 1);
    }
  } else if (warp == 5) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      int kc = 0, qc = 0, job = 0;
      // ring positions and phase parities as wrapping counters: this single
      // thread's loop bounds the item rate, and a division per ring per item
      // (runtime ring sizes) measurably slowed it (~1 us per step)
      int st_i = 0, cb_i = 0, tb_i = 0, q_i = 0;
      uint32_t st_ph = 0, cb_ph = 0, tb_ph = 0;
      ReqCursor cur;
      cur.init(prefix, b.B, lo);
      for (int it = lo; it < hi && !*abort; ++it) {
        bool new_unit = cur.advance(it) || it == lo;
        if (new_unit)
          u.start(it - cur.first, chunks_of(cur.bi));
        else
          new_unit = u.step();
        if (new_unit) {
          if (qc > 0) tc5::mma_commit(smem_u32(&sm.qempty[(qc - 1) % NQB]));
          const int qb = qc % NQB;
          if (!tc5::mbar_wait(smem_u32(&sm.qfull[qb]), (qc / NQB) & 1, abort)) break;
          q_i = qb;
          ++qc;
        }
        const int st = st_i, cb = cb_i;
        if (kFp8) {
          if (!tc5::mbar_wait(smem_u32(&sm.cfull[cb]), cb_ph, abort)) break;
        } else {
          if (!tc5::mbar_wait(smem_u32(&sm.full[st]), st_ph, abort)) break;
        }
        tc5::fence_after_sync();
        const uint32_t ka = kFp8 ? cbuf + cb * kStageBytes : kbuf + st * kStageBytes;
        const uint32_t qa = qbuf + q_i * qbytes;
        bool ok = true;
        for (int g = 0; g < u.ngroups; ++g) {
          const int gn = min(G, u.su - g * G);
          const int tb = tb_i;
          if (job >= NB && !tc5::mbar_wait(smem_u32(&sm.tempty[tb]), tb_ph ^ 1u, abort)) {
            ok = false;
            break;
          }
          tc5::fence_after_sync();
          const uint32_t idesc = tc5::idesc_bf16_f32(128, 64 * gn);
          if (a_in_tmem) {
#pragma unroll
            for (int k = 0; k < 8; ++k) {  // K = 16: eight columns of bf16 pairs per step
              const uint32_t off = (uint32_t)(k & 3) * 32u;
              const uint64_t bd =
                  tc5::sdesc_k_sw128(qa + (k >> 2) * (SU * kQSubBytes) + g * G * kQSubBytes + off);
              tc5::mma_bf16_ta(tmem + tb * acc_cols, tmem + acol + cb * 64 + 8 * k, bd, idesc,
                               k > 0 ? 1u : 0u);
            }
          } else {
#pragma unroll
            for (int k = 0; k < 8; ++k) {
              const uint32_t off = (uint32_t)(k & 3) * 32u;
              const uint64_t ad = tc5::sdesc_k_sw128(ka + (k >> 2) * kSubBytes + off);
              const uint64_t bd =
                  tc5::sdesc_k_sw128(qa + (k >> 2) * (SU * kQSubBytes) + g * G * kQSubBytes + off);
              tc5::mma_bf16(tmem + tb * acc_cols, ad, bd, idesc, k > 0 ? 1u : 0u);
            }
          }
          tc5::mma_commit(smem_u32(&sm.tfull[tb]));
          ++job;
          if (++tb_i == NB) { tb_i = 0; tb_ph ^= 1u; }
        }
        if (!ok) break;
        tc5::mma_commit(smem_u32(kFp8 ? &sm.cempty[cb] : &sm.empty[st]));
        ++kc;
        if (++st_i == NST) { st_i = 0; st_ph ^= 1u; }
        if (kFp8 && ++cb_i == NCB) { cb_i = 0; cb_ph ^= 1u; }
      }
      // every MMA issued above has finished before TMEM is freed
      tc5::mma_commit(smem_u32(&sm.done));
      tc5::mbar_wait_drain(smem_u32(&sm.done), 0);
    }
  } else if (kFp8 && warp >= 6) {
    // ------------------------------------------------------------ converters (FP8 keys)
    // one thread per key row r of each item: the row's eight 16-byte FP8
    // chunks of the TMA tile (128-byte swizzle: chunk c at (c ^ (r & 7)))
    // into the two bf16 sub-tiles of a converted buffer (the same swizzle);
    // then each thread frees the stage and publishes the buffer to the MMA
    // issuer
    // (a_tmem: into the row's TMEM lane, which this warp's lane quarter holds,
    // column 8c + i holding dims 16c + 2i and 16c + 2i + 1)
    const int r = 32 * (warp & 3) + lane;
    int kc = 0;
    for (int it = lo; it < hi && !*abort; ++it, ++kc) {
      const int st = kc % NST, cb = kc % NCB;
      if (!tc5::mbar_wait(smem_u32(&sm.full[st]), (kc / NST) & 1, abort)) break;
      if (kc >= NCB && !tc5::mbar_wait(smem_u32(&sm.cempty[cb]), ((kc / NCB) - 1) & 1, abort))
        break;
      const uint8_t* src = smem_raw + (kbuf + st * kStage8Bytes - smem_u32(smem_raw)) + r * 128;
      if (a_in_tmem) {
        tc5::fence_after_sync();
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          uint32_t o[32];
#pragma unroll
          for (int c4 = 0; c4 < 4; ++c4) {
            const int c = 4 * h + c4;
            const uint4 v = *reinterpret_cast<const uint4*>(src + ((c ^ (r & 7)) << 4));
            e4m3x16_to_bf16(v, o + 8 * c4);
          }
          tc5::tmem_st32(tmem + ((uint32_t)(32 * (warp & 3)) << 16) + acol + cb * 64 + 32 * h,
                         reinterpret_cast<const float*>(o));
        }
        tc5::tmem_wait_st();
        tc5::fence_before_sync();
        tc5::mbar_arrive(smem_u32(&sm.empty[st]));
        tc5::mbar_arrive(smem_u32(&sm.cfull[cb]));
        continue;
      }
      uint8_t* dst = smem_raw + (cbuf + cb * kStageBytes - smem_u32(smem_raw)) + r * 128;
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        const uint4 v = *reinterpret_cast<const uint4*>(src + ((c ^ (r & 7)) << 4));
        uint32_t o[8];
        e4m3x16_to_bf16(v, o);
        // dims 16c .. 16c+15: sub-tile c / 4, bf16 chunks 2(c % 4) and 2(c % 4) + 1
        uint8_t* sub = dst + (c >> 2) * kSubBytes;
        const int c0 = 2 * (c & 3);
        *reinterpret_cast<uint4*>(sub + ((c0 ^ (r & 7)) << 4)) = make_uint4(o[0], o[1], o[2], o[3]);
        *reinterpret_cast<uint4*>(sub + (((c0 + 1) ^ (r & 7)) << 4)) = make_uint4(o[4], o[5], o[6], o[7]);
      }
      tc5::fence_proxy_async_smem();  // the MMA reads the tile through the async proxy
      tc5::mbar_arrive(smem_u32(&sm.empty[st]));
      tc5::mbar_arrive(smem_u32(&sm.cfull[cb]));
    }
  } else if (warp < 4) {
    // ------------------------------------------------------------ epilogue
    const int row = warp * 32 + lane;  // TMEM lane = key row within the item
    int job = 0;
    ReqCursor cur;
    cur.init(prefix, b.B, lo);
    int L = 0;
    int64_t off = 0;
    uint32_t ephase = 0;
    // this CTA's items of request pub_bi scored so far: published (a release
    // add to done[pub_bi]) once every epilogue thread has stored them
    int pub_bi = -1, pub_n = 0;
    for (int it = lo; it < hi && !*abort; ++it) {
      const bool new_req = cur.advance(it) || it == lo;
      bool new_unit = new_req;
      if (new_req) {
        L = b.ctx_len[cur.bi];
        off = b.idx_table ? 0 : b.idx_off[cur.bi];
        u.start(it - cur.first, chunks_of(cur.bi));
      } else {
        new_unit = u.step();
      }
      if (new_unit) {
        // the unit's w (su x 64) into shared memory, shared by its items
        // (bounded barriers: a warp that gave up a wait must not strand the
        // others).  The first barrier also orders every thread's score
        // stores of the previous request before its publication.
        if (!tc5::bar_bounded(smem_u32(&sm.ebar), ephase, abort)) break;
        if (new_req) {
          if (done && row == 0 && pub_n > 0) red_release_add(done + pub_bi, pub_n);
          pub_bi = cur.bi;
          pub_n = 0;
        }
        const float* wsrc = b.w + ((int64_t)cur.bi * S + u.g0) * kTcHi;
        for (int v = row; v < u.su * kTcHi; v += 128) w_sm[v] = __ldg(wsrc + v);
        if (!tc5::bar_bounded(smem_u32(&sm.ebar), ephase, abort)) break;
      }
      const int bi = cur.bi;
      const int c0 = u.chunk * kIdxChunk;
      const int64_t gr = b.idx_table ? idx_row(b, bi, c0 + row) : off + c0 + row;
      const bool in_pool = gr >= 0 && gr < b.idx_rows;
      // FP8: the row's scale (loaded ahead of the accumulator wait); only rows
      // the query may read are used
      float ks = 1.f;
      if (kFp8 && in_pool && c0 + row < L / c.ratio) ks = __ldg(b.idx_scale + gr);
      bool ok = true;
      for (int g = 0; g < u.ngroups; ++g) {
        const int gn = min(G, u.su - g * G);
        const int tb = job % NB;
        if (!tc5::mbar_wait(smem_u32(&sm.tfull[tb]), (job / NB) & 1, abort)) {
          ok = false;
          break;
        }
        tc5::fence_after_sync();
        for (int sl = 0; sl < gn; ++sl) {
          const int s = u.g0 + g * G + sl;  // query within the request
          const int qid = bi * S + s;
          const QueryPlan p = query_plan(c, S, L, s, score_all);
          if (!(p.flags & kPlanScore) || p.vis <= c0) continue;  // warp-uniform
          const uint32_t ta = tmem + ((uint32_t)(warp * 32) << 16) + tb * acc_cols + sl * kTcHi;
          // four disjoint 16-head partials, each summed in ascending h, then
          // added in ascending order; the heads come out of TMEM 32 at a time
          // (FP8 keys: two CTAs per SM leave fewer registers per thread)
          // FP8 keys: with a positive row scale, ReLU(ks x) = ks ReLU(x), so
          // the scale multiplies the row's sum once (any other scale: each
          // dot product, as defined)
          const float4* w4 = reinterpret_cast<const float4*>(w_sm + (g * G + sl) * kTcHi);
          float part[4];
          float v[64];
          const bool per_head = kFp8 && !(ks > 0.f);
          if (!kFp8) tc5::tmem_ld32x2(ta, v, v + 32);
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            if (kFp8 && (k & 1) == 0) tc5::tmem_ld32(ta + 16 * k, v + 16 * k);
            float acc = 0.f;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const float4 wv = w4[k * 4 + i];
              const int h = k * 16 + i * 4;
              if (per_head) {
                acc = fmaf(wv.x, fmaxf(v[h] * ks, 0.f), acc);
                acc = fmaf(wv.y, fmaxf(v[h + 1] * ks, 0.f), acc);
                acc = fmaf(wv.z, fmaxf(v[h + 2] * ks, 0.f), acc);
                acc = fmaf(wv.w, fmaxf(v[h + 3] * ks, 0.f), acc);
              } else {
                acc = fmaf(wv.x, fmaxf(v[h], 0.f), acc);
                acc = fmaf(wv.y, fmaxf(v[h + 1], 0.f), acc);
                acc = fmaf(wv.z, fmaxf(v[h + 2], 0.f), acc);
                acc = fmaf(wv.w, fmaxf(v[h + 3], 0.f), acc);
              }
            }
            part[k] = acc;
          }
          float sum = ((part[0] + part[1]) + part[2]) + part[3];
          if (kFp8 && !per_head) sum *= ks;
          const int j = c0 + row;
          if (j < p.vis) {
            if (!in_pool) set_status(ws.status, kStatusBadIndex);
            if (keys)
              reinterpret_cast<uint32_t*>(scores)[(int64_t)qid * ld + j] = score_order_key(sum);
            else
              scores[(int64_t)qid * ld + j] = sum;
          }
        }
        tc5::fence_before_sync();
        tc5::mbar_arrive(smem_u32(&sm.tempty[tb]));
        ++job;
      }
      if (!ok) break;
      ++pub_n;
    }
    // the last request's items, once every epilogue thread has stored them
    if (done && !*abort && tc5::bar_bounded(smem_u32(&sm.ebar), ephase, abort) && row == 0 && pub_n > 0)
      red_release_add(done + pub_bi, pub_n);
  }

  if (tid == 0 && *abort) set_status(ws.status, kStatusTimeout);
  tc5::fence_before_sync();
  __syncthreads();
  tc5::fence_after_sync();
  if (warp == 5) tc5::tmem_dealloc(tmem, tmem_cols);
}

// 2D tensor [rows, cols] with a row stride in elements; boxes of
// [box_rows, 128 bytes] (one 128-byte swizzle row): 64 bf16 or 128 FP8.
bool make_map(CUtensorMap* m, const void* ptr, uint64_t rows, uint64_t cols, uint64_t stride,
              uint32_t box_rows, bool fp8 = false) {
  auto fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(tensor_map_encoder());
  if (!fn) return false;
  const uint64_t es = fp8 ? 1 : 2;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {stride * es};
  cuuint32_t box[2] = {(cuuint32_t)(128 / es), box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
            const_cast<void*>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

// Launch shape of the tcgen05 indexer for S queries per request; false when
// a request's queries leave no room for two key stages (the caller then uses
// the warp-MMA kernel).  Tuning knobs, read once: CSA_T5_STAGES caps the ring
// depth, CSA_T5_CTAS forces the CTAs per SM (1..4).
struct T5Plan {
  int ctas_per_sm, acc_cols, NB, NCB, NST, NQB, stage_bytes, conv_bytes, qbytes, a_tmem;
};
// The plan for a given number of CTAs per SM (FP8 keys: converted items in
// TMEM or in shared memory); false if two key stages or two accumulators do
// not fit.
static bool plan_t5_with(const DevCfg& c, int S, int ctas, bool a_tmem, int max_stages, T5Plan* p) {
  const bool fp8 = c.idx_fp8 != 0;
  p->ctas_per_sm = ctas;
  p->a_tmem = fp8 && a_tmem ? 1 : 0;
  const int G = S < 4 ? S : 4;
  p->acc_cols = 32;
  while (p->acc_cols < 64 * G) p->acc_cols <<= 1;  // power of two >= 32
  // accumulators that fit in TMEM beside the converted items (two of 64
  // columns with a_tmem); an allocation is a power of two columns
  const int areserve = p->a_tmem ? 2 * 64 : 0;
  p->NB = (512 / p->ctas_per_sm - areserve) / p->acc_cols;
  if (p->NB > 8) p->NB = 8;
  while (p->NB >= 2 && ((p->NB * p->acc_cols + areserve) & (p->NB * p->acc_cols + areserve - 1))) --p->NB;
  if (p->NB < 2) return false;
  p->qbytes = S * 2 * kQSubBytes;
  const int per_cta = 228 * 1024 / p->ctas_per_sm - 1024;  // per-SM shared memory / CTAs
  p->stage_bytes = fp8 ? kStage8Bytes : kStageBytes;
  const int fixed = per_cta - 1024 - (int)sizeof(T5Smem) - 64 - S * kTcHi * 4;
  // FP8 converted items: two in TMEM, or in shared memory two when two key
  // stages still fit beside them, else one (measured: a third adds nothing)
  p->NCB = fp8 ? kConvBufs : 0;
  if (fp8 && !p->a_tmem && fixed - p->NCB * kStageBytes - p->qbytes < 2 * p->stage_bytes) p->NCB = 1;
  p->conv_bytes = (fp8 && !p->a_tmem) ? p->NCB * kStageBytes : 0;
  // key stages first: a CTA spans few requests, so a second q_idx buffer
  // (prefetching the next request's queries) is kept only when it costs no
  // key stage
  const int budget = fixed - p->conv_bytes;
  auto stages = [&](int nqb) {
    const int n = (budget - nqb * p->qbytes) / p->stage_bytes;
    return n > max_stages ? max_stages : n;
  };
  p->NQB = stages(2) >= stages(1) ? 2 : 1;
  p->NST = stages(p->NQB);
  return p->NST >= 2;
}

static bool plan_t5(const DevCfg& c, int S, T5Plan* p) {
  static const int max_stages = [] {
    const char* e = getenv("CSA_T5_STAGES");
    const int v = e ? atoi(e) : 8;
    return (v < 2 || v > 8) ? 8 : v;
  }();
  static const int forced_ctas = [] {
    const char* f = getenv("CSA_T5_CTAS");
    const int v = f ? atoi(f) : 0;
    return (v < 0 || v > 4) ? 0 : v;
  }();
  // FP8 converted items in TMEM unless CSA_T5_ATMEM=0
  static const bool atmem = [] {
    const char* e = getenv("CSA_T5_ATMEM");
    return !(e && e[0] == '0');
  }();
  // CTAs per SM: two independent pipelines per SM stream measurably faster
  // than one deeper ring (the ring depth beyond three stages does not
  // matter), so two whenever a request's q_idx leaves room for two stages
  // each; FP8 keys likewise (the FP8 kernel is compiled for two CTAs'
  // registers), with the converted items in TMEM when they fit beside the
  // accumulators, else in shared memory.
  const bool fp8 = c.idx_fp8 != 0;
  const int first = forced_ctas ? forced_ctas : (fp8 ? kFp8CtasPerSm : (S <= 2 ? 2 : 1));
  const int last = forced_ctas ? forced_ctas : 1;
  for (int ctas = first; ctas >= last; --ctas) {
    if (fp8 && atmem && plan_t5_with(c, S, ctas, true, max_stages, p)) return true;
    if (plan_t5_with(c, S, ctas, false, max_stages, p)) return true;
  }
  return false;
}

bool indexer_tc5_fits(const DevCfg& c, int S) {
  T5Plan p;
  return plan_t5(c, S, &p);
}

// Launches the tcgen05 indexer; returns 1 on launch, 0 with nothing to do,
// -1 if the launch (or the tensor-map encoding) failed, -2 if the shape does
// not fit this kernel (the caller then uses the warp-MMA kernel).  qsplit:
// the work list's queries per item (0: all of a request's).
int launch_indexer_tc5(const DevCfg& c, const DevBatch& b, const Workspace& ws,
                       const ItemList& items, int score_all, float* scores, int64_t ld,
                       int num_sms, int qsplit, cudaStream_t st, bool pdl, int* done,
                       int* done_clear, bool keys) {
  const int known = items.host_B >= 0 ? items.prefix[items.host_B] : -1;
  if (known == 0) return 0;
  if (b.idx_rows <= 0 || b.idx_rows > 0x7fffffffLL) return -2;
  const int S = b.S;
  const bool fp8 = c.idx_fp8 != 0;
  const int SU = qsplit ? qsplit : S;  // queries per work unit
  T5Plan p;
  if (!plan_t5(c, SU, &p)) return -2;
  if (fp8 && !b.idx_scale) return launch_fail("FP8 keys without idx_scale", cudaSuccess);
  CUtensorMap kmap, qmap;
  if (!make_map(&kmap, b.idx, (uint64_t)b.idx_rows, kTcDi, (uint64_t)b.idx_stride, kIdxChunk, fp8))
    return launch_fail("cuTensorMapEncodeTiled(idx_k)", cudaSuccess);
  if (!make_map(&qmap, b.q_idx, (uint64_t)b.B * S * kTcHi, kTcDi, kTcDi, kTcHi))
    return launch_fail("cuTensorMapEncodeTiled(q_idx)", cudaSuccess);
  const int smem = 1024 + p.NST * p.stage_bytes + p.conv_bytes + p.NQB * p.qbytes + SU * kTcHi * 4;
  static PerDeviceOnce attr;
  if (const cudaError_t e = attr.run([] {
        cudaError_t r = allow_max_dynamic_smem(indexer_tc5_kernel<false, false>);
        if (r == cudaSuccess) r = allow_max_dynamic_smem(indexer_tc5_kernel<false, true>);
        if (r == cudaSuccess) r = allow_max_dynamic_smem(indexer_tc5_kernel<true, false>);
        if (r == cudaSuccess) r = allow_max_dynamic_smem(indexer_tc5_kernel<true, true>);
        return r;
      }))
    return launch_fail("cudaFuncSetAttribute(indexer_tc5_kernel)", e);
  int grid = num_sms * p.ctas_per_sm;
  if (known > 0 && known < grid) grid = known;
  const dim3 block(fp8 ? kT5ThreadsFp8 : kT5Threads);
  auto go = [&](auto kernel) {
    return launch_kernel(kernel, dim3(grid), block, smem, st, pdl, kmap, qmap, items, c, b, ws,
                         score_all, scores, ld, p.NST, p.NQB, p.acc_cols, p.NB, p.NCB, qsplit, done,
                         done_clear, p.a_tmem, keys ? 1 : 0);
  };
  if (fp8) return qsplit ? go(indexer_tc5_kernel<true, true>) : go(indexer_tc5_kernel<true, false>);
  return qsplit ? go(indexer_tc5_kernel<false, true>) : go(indexer_tc5_kernel<false, false>);
}

}  // namespace csa
